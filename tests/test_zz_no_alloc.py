"""gemm_relu_f16_splitk_noalloc: split-K for callers that may not allocate.

Some callers cannot call cudaMalloc at all -- a framework whose own pool owns
all device memory, a serving loop that forbids allocation after warm-up, a
plugin handed only its input and output pointers.  For them the library keeps
a fixed 8 MiB device scratch array and this entry point uses it in place of a
caller workspace.

The tests call it through the C ABI, twice in a row on the same problem, with
a call on other, larger inputs in between so that the shared array holds
someone else's partials when the second call starts.  Each result must match
the CPU oracle within the parity tolerance the other tests use and be
bit-identical to gemm_relu_f16_splitk with an ordinary workspace (both run the
same kernels, adding the same partials in the same order).  The file sits on
its own and is collected last; it does not depend on any earlier test having
run (the entry point's first call on the device does its own set-up).
"""
import numpy as np
import pytest

import tiled_tensor_core_03_gb300 as gr
from tiled_tensor_core_03_gb300 import inputs

from gpu_common import abs_dot, assert_parity

pytestmark = pytest.mark.gpu

LIMIT = gr.NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.fixture
def split_form(request):
    """The split-K form under test: the two-stage form is the one that needs
    scratch; splits of 2, 4 and 8 otherwise reduce inside a cluster and need
    none."""
    gr.gemm_relu_debug_force_split(request.param)
    yield request.param
    gr.gemm_relu_debug_force_split(gr.SPLIT_AUTO)


def _stream(torch):
    return torch.cuda.current_stream().cuda_stream


def _noalloc(torch, a, b, M, N, K, S):
    out = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    rc = gr.lib().gemm_relu_f16_splitk_noalloc(a.data_ptr(), b.data_ptr(), out.data_ptr(),
                                               M, N, K, S, _stream(torch))
    assert rc == gr.OK, gr.strerror(rc)
    assert gr.status() == gr.OK
    return out


def _with_workspace(torch, a, b, M, N, K, S):
    need = gr.gemm_relu_f16_splitk_workspace_bytes(M, N, K, S)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    rc = gr.lib().gemm_relu_f16_splitk(a.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, K, S,
                                       ws.data_ptr(), need, _stream(torch))
    assert rc == gr.OK, gr.strerror(rc)
    assert gr.status() == gr.OK
    return out


def _dirty_the_scratch(torch, restore):
    """A two-stage call on other inputs whose partials fill the whole array;
    then the split-form hook goes back to `restore`."""
    M, N, K, S = 64, 4096, 2048, 8                     # 8 * 64 * 4096 * 4 B = 8 MiB
    A, B = inputs.make(M, N, K, dist="uniform", seed=99)
    gr.gemm_relu_debug_force_split(gr.SPLIT_TWO_STAGE)
    try:
        assert gr.gemm_relu_f16_splitk_workspace_bytes(M, N, K, S) == LIMIT
        _noalloc(torch, torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), M, N, K, S)
    finally:
        gr.gemm_relu_debug_force_split(restore)


@pytest.mark.parametrize("split_form", [gr.SPLIT_TWO_STAGE, gr.SPLIT_AUTO], indirect=True,
                         ids=["two_stage", "auto"])
@pytest.mark.parametrize("M,N,K,S", [(16, 8192, 8192, 8), (33, 1000, 1000, 3), (1, 128, 1024, 2),
                                     (64, 4096, 2048, 8)])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(torch, orc, split_form, M, N, K, S):
    A, B = inputs.make(M, N, K, dist="normal", scale_by_sqrt_k=True, seed=M + N + K)
    a = torch.from_numpy(A).cuda()
    b = torch.from_numpy(B).cuda()
    need = gr.gemm_relu_f16_splitk_workspace_bytes(M, N, K, S)
    assert need <= LIMIT
    if split_form == gr.SPLIT_TWO_STAGE or S == 3:
        assert need > 0
    if (M, N, K, S) == (64, 4096, 2048, 8) and split_form == gr.SPLIT_TWO_STAGE:
        assert need == LIMIT                         # exactly the whole array

    want = _with_workspace(torch, a, b, M, N, K, S)
    oracle = orc.gemm_relu_f16(A, B)
    absab = abs_dot(A, B)
    for call in range(2):
        got = _noalloc(torch, a, b, M, N, K, S)
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), call
        assert_parity(got.cpu().numpy(), oracle, absab, K, ("noalloc", call, M, N, K, S))
        if call == 0:
            # leave other partials in the shared array before the second call
            _dirty_the_scratch(torch, split_form)


@pytest.mark.parametrize("split_form,M,S", [(gr.SPLIT_TWO_STAGE, 64, 8), (gr.SPLIT_AUTO, 128, 3)],
                         indirect=["split_form"], ids=["two_stage", "auto"])
def test_noalloc_rejects_problems_beyond_its_scratch(torch, split_form, M, S):
    lib = gr.lib()
    N, K = 8192, 8192                        # S * M * 32 KiB of partials > 8 MiB
    assert gr.gemm_relu_f16_splitk_workspace_bytes(M, N, K, S) > LIMIT
    a = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    b = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    c = torch.full((M, N), 3.0, dtype=torch.float16, device="cuda")
    rc = lib.gemm_relu_f16_splitk_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, S,
                                          _stream(torch))
    assert rc == gr.ERR_SCRATCH_LIMIT
    assert "scratch" in gr.strerror(rc)
    torch.cuda.synchronize()
    assert (c.float() == 3.0).all()          # nothing was launched


def test_noalloc_fallback_needs_no_scratch(torch, orc):
    """Operands that cannot use TMA (N odd) make the split-K call fall back to
    the unsplit kernel, which uses no scratch: the call runs even though the
    two-stage form of the same sizes would need more than the array."""
    M, N, K, S = 128, 8191, 8192, 8
    assert gr.gemm_relu_f16_splitk_workspace_bytes(M, N, K, S) > LIMIT
    A, B = inputs.make(M, N, K, dist="normal", scale_by_sqrt_k=True, seed=5)
    a = torch.from_numpy(A).cuda()
    b = torch.from_numpy(B).cuda()
    got = _noalloc(torch, a, b, M, N, K, S)
    assert torch.equal(got.view(torch.int16), gr.gemm_relu(a, b).view(torch.int16))
    rows = [0, 63, 127]
    want = np.concatenate([orc.gemm_relu_f16_rows(A, B, r, 1) for r in rows])
    assert_parity(got.cpu().numpy()[rows], want, abs_dot(A[rows], B), K, "noalloc fallback")

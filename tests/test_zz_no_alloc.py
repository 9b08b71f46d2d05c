"""gemm_relu_f16_splitk_noalloc: split-K for callers that may not allocate.

Some callers cannot call cudaMalloc at all -- a framework whose own pool owns
all device memory, a serving loop that forbids allocation after warm-up, a
plugin handed only its input and output pointers.  For them the library keeps
a fixed 8 MiB device scratch array and this entry point uses it in place of a
caller workspace.  The test calls it through the C ABI twice in a row and
checks each result against gemm_relu_f16_splitk with an ordinary workspace,
within the parity tolerance the other tests use.  It sits in a file of its
own, collected last, and does not depend on any earlier test having run
(the entry point's first call on the device does its own set-up).
"""
import ctypes

import numpy as np
import pytest

import tiled_tensor_core_03_gb300 as gr
from tiled_tensor_core_03_gb300 import inputs

from gpu_common import abs_dot, compare

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("split_form", [gr.SPLIT_TWO_STAGE, gr.SPLIT_AUTO], indirect=True,
                         ids=["two_stage", "auto"])
@pytest.mark.parametrize("M,N,K,S", [(16, 8192, 8192, 8), (33, 1000, 1000, 3), (1, 128, 1024, 2)])
def test_noalloc_matches_workspace_entry_point_twice(torch, split_form, M, N, K, S):
    lib = gr.lib()
    A, B = inputs.make(M, N, K, dist="normal", scale_by_sqrt_k=True, seed=M + N + K)
    a = torch.from_numpy(A).cuda()
    b = torch.from_numpy(B).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    need = gr.gemm_relu_f16_splitk_workspace_bytes(M, N, K, S)
    assert need <= gr.NOALLOC_SCRATCH_BYTES
    if split_form == gr.SPLIT_TWO_STAGE or S == 3:
        assert need > 0

    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    ref = torch.empty((M, N), dtype=torch.float16, device="cuda")
    rc = lib.gemm_relu_f16_splitk(a.data_ptr(), b.data_ptr(), ref.data_ptr(), M, N, K, S,
                                  ws.data_ptr(), need, stream)
    assert rc == gr.OK
    want = ref.cpu().numpy()
    absab = abs_dot(A, B)

    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        rc = lib.gemm_relu_f16_splitk_noalloc(a.data_ptr(), b.data_ptr(), out.data_ptr(),
                                              M, N, K, S, stream)
        assert rc == gr.OK, gr.strerror(rc)
        assert gr.status() == gr.OK
        got = out.cpu().numpy()
        r = compare(got, want, absab, K)
        assert r["finite"] and r["contract_ok"] and r["strict_ok"], (call, r)


@pytest.mark.parametrize("split_form,M,S", [(gr.SPLIT_TWO_STAGE, 64, 8), (gr.SPLIT_AUTO, 128, 3)],
                         indirect=["split_form"], ids=["two_stage", "auto"])
def test_noalloc_rejects_problems_beyond_its_scratch(torch, split_form, M, S):
    lib = gr.lib()
    N, K = 8192, 8192                        # S * M * 32 KiB of partials > 8 MiB
    assert gr.gemm_relu_f16_splitk_workspace_bytes(M, N, K, S) > gr.NOALLOC_SCRATCH_BYTES
    a = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    b = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    c = torch.full((M, N), 3.0, dtype=torch.float16, device="cuda")
    rc = lib.gemm_relu_f16_splitk_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, S,
                                          torch.cuda.current_stream().cuda_stream)
    assert rc == gr.ERR_SCRATCH_LIMIT
    assert "scratch" in gr.strerror(rc)
    torch.cuda.synchronize()
    assert (c.float() == 3.0).all()          # nothing was launched

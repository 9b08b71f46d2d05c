"""GPU parity on seeded random shapes: every entry point (plain, stream-K,
split-K in both forms) against the oracle, with the contract and the
scale-aware bound of gpu_common.compare.

Shapes are drawn from a fixed generator so that the run is reproducible:
row counts from 1 to ~3000, columns and depths from 1 to ~2500, with odd
pitches (the predicated-load path), multiples of 8 (the TMA paths), skinny
and decode rows, and contractions shorter than one k block.  The full output
is compared where the oracle finishes quickly, else the first and last rows
of every 128-row block plus 2048 random elements.
"""
import numpy as np
import pytest

import tiled_tensor_core_03_gb300 as gr
from tiled_tensor_core_03_gb300 import inputs

from gpu_common import abs_dot, assert_parity, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gr.gemm_relu_debug_set(0, 0)
    yield
    assert gr.status() == gr.OK


def _shapes(seed, n):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        kind = i % 4
        if kind == 0:      # anything, odd pitches likely
            M, N, K = (int(x) for x in rng.integers(1, 2600, 3))
        elif kind == 1:    # TMA-capable pitches
            M = int(rng.integers(1, 3000))
            N, K = (8 * int(x) for x in rng.integers(1, 320, 2))
        elif kind == 2:    # skinny / decode rows
            M = int(rng.integers(1, 65))
            N, K = (8 * int(x) for x in rng.integers(16, 1024, 2))
        else:              # short contractions
            M, N = (int(x) for x in rng.integers(1, 1500, 2))
            K = int(rng.integers(1, 70))
        out.append((M, N, K))
    return out


def _reference(orc, A, B):
    """A checker of outputs for (A, B): the oracle's full output where it
    finishes quickly, else its first and last rows of every 128-row block and
    2048 random elements (computed once, used for every entry point)."""
    M, K = A.shape
    N = B.shape[1]
    if M * N * K <= 6e8:
        want, absab = orc.gemm_relu_f16(A, B), abs_dot(A, B)

        def check(got, what):
            assert_parity(got, want, absab, K, what)
        return check
    rows = sorted({r for mb in range((M + 127) // 128) for r in (mb * 128, min(M - 1, mb * 128 + 127))})
    want_rows = np.concatenate([orc.gemm_relu_f16_rows(A, B, r, 1) for r in rows])
    abs_rows = abs_dot(A[rows], B)
    rng = np.random.default_rng(M + K)
    I = rng.integers(0, M, 2048)
    J = rng.integers(0, N, 2048)
    want_at, abs_at = orc.gemm_relu_f16_at(A, B, I, J), abs_dot(A, B, I, J)

    def check(got, what):
        assert_parity(got[rows], want_rows, abs_rows, K, (what, "rows"))
        assert_parity(got[I, J], want_at, abs_at, K, (what, "samples"))
    return check


@pytest.mark.parametrize("chunk", range(8))
def test_random_shapes_every_entry_point(orc, chunk):
    import torch
    for j, (M, N, K) in enumerate(_shapes(1234 + chunk, 16)):
        A, B = inputs.make(M, N, K, "normal", True, seed=7 * M + 3 * N + K)
        a, b = dev(A), dev(B)
        what = (M, N, K)
        check = _reference(orc, A, B)
        check(host(gr.gemm_relu(a, b)), (what, "gemm_relu_f16"))
        ws = gr.streamk_workspace(M, N, K)
        ws.random_(0, 256)
        check(host(gr.gemm_relu_streamk(a, b, workspace=ws)), (what, "streamk"))
        S = (2, 3, 4, 8)[j % 4]
        check(host(gr.gemm_relu_splitk(a, b, S)), (what, "splitk", S))
        c = torch.empty((M, N), dtype=torch.float16, device="cuda")
        rc = gr.gemm_relu_f16_splitk_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, S,
                                             torch.cuda.current_stream().cuda_stream)
        if rc == gr.OK:
            check(host(c), (what, "splitk_noalloc", S))
        else:
            assert rc == gr.ERR_SCRATCH_LIMIT, (what, rc)
        assert gr.status() == gr.OK, what

"""Largest sizes: outputs past 2^31 elements and very long K.

Every kernel forms output and operand offsets in 64-bit arithmetic; these
tests pin that by writing C matrices of more than 2^31 elements (4.3 GB of
fp16) through the TMA path and the unaligned (LSU) path, and by a
contraction over 2^20 terms.  The outputs are checked on sampled rows and
elements against the oracle: integer-valued operands make every element
exact, so the comparison is bit for bit; the long-K case is held to the
scale-aware bound of the other parity tests.
"""
import numpy as np
import pytest

import tiled_tensor_core_03_gb300 as gr

from gpu_common import abs_dot, compare, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    free, _ = torch.cuda.mem_get_info()
    if free < 12 << 30:
        pytest.skip("needs 12 GB of free device memory")
    return torch


def _ints(rng, shape):
    return rng.integers(-3, 4, size=shape).astype(np.float16)


@pytest.mark.parametrize("N,path", [(65544, gr.PATH_TMA), (65545, gr.PATH_LSU)],
                         ids=["tma", "lsu"])
def test_output_past_2_31_elements(torch, orc, N, path):
    M, K = 32769, 16                     # M * N > 2^31
    assert M * N > 2 ** 31
    rng = np.random.default_rng(N)
    A, B = _ints(rng, (M, K)), _ints(rng, (K, N))
    a, b = dev(A), dev(B)
    c = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    assert gr.gemm_relu_f16_path(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K) == path
    gr.gemm_relu(a, b, out=c)
    assert gr.status() == gr.OK
    # rows on both sides of the 2^31-element mark, the first and the last
    edge = (2 ** 31) // N
    rows = sorted({0, 1, edge - 1, edge, edge + 1, M // 2, M - 2, M - 1})
    got = c[rows].cpu().numpy()
    want = np.concatenate([orc.gemm_relu_f16_rows(A, B, r, 1) for r in rows])
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
    # and elements scattered over the whole output
    I = rng.integers(0, M, 4096)
    J = rng.integers(0, N, 4096)
    I_t = torch.from_numpy(I).cuda()
    J_t = torch.from_numpy(J).cuda()
    got = c[I_t, J_t].cpu().numpy()
    want = orc.gemm_relu_f16_at(A, B, I, J)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))


def test_contraction_over_2_20_terms(torch, orc):
    M, N, K = 256, 256, 1 << 20
    rng = np.random.default_rng(20)
    # outputs of order 1: A ~ N(0, 1), B ~ N(0, 1) / sqrt(K)
    A = rng.standard_normal((M, K), dtype=np.float32).astype(np.float16)
    B = (rng.standard_normal((K, N), dtype=np.float32) / np.float32(np.sqrt(K))).astype(np.float16)
    c = gr.gemm_relu(dev(A), dev(B))
    assert gr.status() == gr.OK
    got = c.cpu().numpy()
    assert np.isfinite(got.astype(np.float32)).all() and (got.astype(np.float32) >= 0).all()
    I = rng.integers(0, M, 48)
    J = rng.integers(0, N, 48)
    want = orc.gemm_relu_f16_at(A, B, I, J)
    r = compare(got[I, J], want, abs_dot(A, B, I, J), K)
    assert r["contract_ok"] and r["strict_ok"], r

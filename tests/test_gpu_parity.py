"""GPU parity: the CUDA path against the CPU oracle, element by element.

Every workload is compared in full, the 4096^3 one with the oracle's rows
spread over the host's threads (computed once per module); the stream-K
shapes other than 4096^3 are compared on sampled rows and elements.  The
tolerance is atol = rtol = 1e-2 per element, and every case must also meet
the scale-aware bound of gpu_common.compare.
"""
import numpy as np
import pytest

import tiled_tensor_core_03_gb300 as gr
from tiled_tensor_core_03_gb300 import inputs

from gpu_common import abs_dot, assert_parity, dev, host, oracle_threaded, run_fused, run_split

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gr.gemm_relu_debug_set(0, 0)
    yield
    assert gr.status() == gr.OK


# ----------------------------------------------------------------- workloads


@pytest.mark.parametrize("name", ["square256", "square1024", "ragged", "decode1"])
def test_workload_full(orc, name):
    w = inputs.WORKLOADS[name]
    A, B = inputs.make_workload(w)
    want = orc.gemm_relu_f16(A, B)
    got = run_fused(A, B)
    assert_parity(got, want, abs_dot(A, B), w.K, name)
    assert gr.status() == gr.OK


def test_ragged_takes_lsu_path_and_aligned_takes_tma():
    import torch
    w = inputs.WORKLOADS["ragged"]
    a = torch.empty((w.M, w.K), dtype=torch.float16, device="cuda")
    b = torch.empty((w.K, w.N), dtype=torch.float16, device="cuda")
    c = torch.empty((w.M, w.N), dtype=torch.float16, device="cuda")
    assert gr.gemm_relu_f16_path(a.data_ptr(), b.data_ptr(), c.data_ptr(), w.M, w.N, w.K) == gr.PATH_LSU
    a = torch.empty((1024, 1024), dtype=torch.float16, device="cuda")
    assert gr.gemm_relu_f16_path(a.data_ptr(), a.data_ptr(), a.data_ptr(), 1024, 1024, 1024) == gr.PATH_TMA


def test_kernel_choice_per_shape():
    """gemm_relu_f16_kernel reports the routing: decode rows to the GEMV
    kernel, skinny rows to the split-K pair form, outputs that one wave of
    128 x 128 tiles covers to the single-CTA kernel, larger ones to CTA
    pairs, unaligned rows to the predicated-load kernel; the force hooks
    override it."""
    import torch
    buf = torch.empty(64 << 20, dtype=torch.float16, device="cuda")
    p = buf.data_ptr()
    cases = [((1, 8192, 8192), gr.KERNEL_GEMV), ((16, 8192, 8192), gr.KERNEL_SPLITK_PAIR),
             ((256, 256, 256), gr.KERNEL_ONE_CTA_128), ((1024, 1024, 1024), gr.KERNEL_ONE_CTA_128),
             ((1920, 1280, 1024), gr.KERNEL_ONE_CTA_128), ((2048, 2048, 2048), gr.KERNEL_PAIR),
             ((4096, 4096, 4096), gr.KERNEL_PAIR), ((128, 4096, 4096), gr.KERNEL_ONE_CTA_128),
             ((1537, 1023, 777), gr.KERNEL_PREDICATED)]
    for (M, N, K), want in cases:
        assert gr.gemm_relu_f16_kernel(p, p, p, M, N, K) == want, (M, N, K)
    assert gr.gemm_relu_f16_kernel(p, p, p, 64, 64, 0) == 0
    assert gr.gemm_relu_f16_kernel(p, p, p, -1, 64, 64) == -1
    try:
        for force, want in ((1, gr.KERNEL_ONE_CTA_256), (2, gr.KERNEL_ONE_CTA_128), (3, gr.KERNEL_PAIR)):
            gr.gemm_relu_debug_force_kernel(force)
            assert gr.gemm_relu_f16_kernel(p, p, p, 1024, 1024, 1024) == want, force
    finally:
        gr.gemm_relu_debug_force_kernel(0)


@pytest.fixture(scope="module")
def square4096(orc):
    """The 4096^3 workload, its full oracle output (rows over the host's
    threads) and sum_k |a||b| for the scale-aware bound."""
    w = inputs.WORKLOADS["square4096"]
    A, B = inputs.make_workload(w)
    return w, A, B, oracle_threaded(orc, A, B), abs_dot(A, B)


def test_square4096_full(square4096):
    """Every element of the 4096^3 output against the oracle."""
    import torch
    w, A, B, want, absab = square4096
    a, b = dev(A), dev(B)
    c = gr.gemm_relu(a, b)
    got = host(c)
    assert_parity(got, want, absab, w.K, "square4096")
    # the stream-K call (the benchmark's path) on the same operands
    ws = gr.streamk_workspace(w.M, w.N, w.K)
    ws.random_(0, 256)
    got_sk = host(gr.gemm_relu_streamk(a, b, workspace=ws))
    assert gr.status() == gr.OK
    assert_parity(got_sk, want, absab, w.K, "square4096 stream-K")


def test_skinny_splitk_full(orc):
    w = inputs.WORKLOADS["skinny"]
    A, B = inputs.make_workload(w)
    want = orc.gemm_relu_f16(A, B)
    absab = abs_dot(A, B)
    got = run_split(A, B, w.split_k)
    assert_parity(got, want, absab, w.K, "skinny split-K")
    fused = run_fused(A, B)
    assert_parity(fused, want, absab, w.K, "skinny fused")


# ----------------------------------------------------------------- sweeps

TMA_SHAPES = [(m, n, k) for m in (1, 7, 128, 129, 257) for n in (8, 136, 256, 264, 520)
              for k in (8, 64, 72, 136)]
LSU_SHAPES = [(m, n, k) for m in (1, 15, 129) for n in (1, 7, 63, 257, 300)
              for k in (1, 15, 65, 127)]


def _sweep(orc, shapes, expect_path):
    import torch
    rng = np.random.default_rng(5)
    bad = []
    for (M, N, K) in shapes:
        A = rng.standard_normal((M, K)).astype(np.float16)
        B = rng.standard_normal((K, N)).astype(np.float16)
        a, b = dev(A), dev(B)
        c = torch.empty((M, N), dtype=torch.float16, device="cuda")
        assert gr.gemm_relu_f16_path(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K) == expect_path
        gr.gemm_relu(a, b, out=c)
        try:
            assert_parity(host(c), orc.gemm_relu_f16(A, B), abs_dot(A, B), K, (M, N, K))
        except AssertionError as e:
            bad.append(str(e)[:300])
    assert not bad, bad[:5]
    assert gr.status() == gr.OK


def test_sweep_tma_path(orc):
    _sweep(orc, TMA_SHAPES, gr.PATH_TMA)


def test_sweep_lsu_path(orc):
    _sweep(orc, LSU_SHAPES, gr.PATH_LSU)


SPLIT_CASES = [(1, 128, 64, 2), (16, 120, 1000, 3), (17, 1000, 1000, 3), (33, 256, 4096, 8),
               (64, 512, 2048, 5), (100, 384, 640, 16), (200, 136, 512, 4), (16, 8, 8192, 8),
               (130, 264, 256, 2)]


@pytest.mark.parametrize("M,N,K,S", SPLIT_CASES)
def test_splitk_sweep(orc, M, N, K, S):
    rng = np.random.default_rng(M * 7 + N + K + S)
    A = rng.standard_normal((M, K)).astype(np.float16)
    B = rng.standard_normal((K, N)).astype(np.float16)
    got = run_split(A, B, S)
    assert_parity(got, orc.gemm_relu_f16(A, B), abs_dot(A, B), K, (M, N, K, S))
    assert gr.status() == gr.OK


@pytest.fixture
def two_stage_split():
    gr.gemm_relu_debug_force_split(gr.SPLIT_TWO_STAGE)
    yield
    gr.gemm_relu_debug_force_split(gr.SPLIT_AUTO)


# (M, N, K, S): M <= 64 and even splits with S * R <= 512 (R = 16, 32, 64 by
# M) take the CTA-pair form in automatic mode; every R, ragged M, N and K,
# S up to 32
CLUSTER_CASES = [(16, 8192, 8192, 8), (1, 128, 1024, 2), (9, 1032, 3000, 4), (32, 640, 2048, 8),
                 (40, 264, 1152, 2), (64, 1024, 4096, 8), (61, 520, 960, 4), (16, 256, 8192, 32),
                 (3, 200, 4096, 6), (30, 1000, 4096, 16), (17, 2056, 1536, 2)]


@pytest.mark.parametrize("M,N,K,S", CLUSTER_CASES)
def test_splitk_cluster_form_matches_two_stage_bits(orc, M, N, K, S):
    """Both forms add the same S partials in the same order: identical bits."""
    import torch
    A, B = inputs.make(M, N, K, dist="normal", scale_by_sqrt_k=True, seed=M + 3 * N + K + S)
    a, b = dev(A), dev(B)
    assert gr.gemm_relu_f16_splitk_workspace_bytes(M, N, K, S) == 0
    c_cluster = gr.gemm_relu_splitk(a, b, S).clone()
    assert gr.status() == gr.OK
    gr.gemm_relu_debug_force_split(gr.SPLIT_TWO_STAGE)
    try:
        assert gr.gemm_relu_f16_splitk_workspace_bytes(M, N, K, S) == S * M * N * 4
        c_two = gr.gemm_relu_splitk(a, b, S).clone()
    finally:
        gr.gemm_relu_debug_force_split(gr.SPLIT_AUTO)
    assert gr.status() == gr.OK
    assert torch.equal(c_cluster.view(torch.int16), c_two.view(torch.int16))
    rows = sorted({0, M // 2, M - 1})
    want = np.concatenate([orc.gemm_relu_f16_rows(A, B, r, 1) for r in rows])
    assert_parity(host(c_cluster)[rows], want, abs_dot(A[rows], B), K, (M, N, K, S))


def test_splitk_cluster_form_unaligned_output():
    """C at a 2-byte offset: the owners fall back to 2-byte stores."""
    import torch
    M, N, K, S = 20, 264, 2048, 4
    A, B = inputs.make(M, N, K, seed=21)
    a, b = dev(A), dev(B)
    want = gr.gemm_relu_splitk(a, b, S)
    buf = torch.full((M * N + 2,), float("nan"), dtype=torch.float16, device="cuda")
    c = buf[1:1 + M * N].view(M, N)
    gr.gemm_relu_splitk(a, b, S, out=c)
    assert gr.status() == gr.OK
    assert torch.equal(c.view(torch.int16), want.view(torch.int16))
    assert torch.isnan(buf[0]) and torch.isnan(buf[-1])


def test_splitk_deterministic_and_workspace_contents_irrelevant(two_stage_split):
    import torch
    w = inputs.WORKLOADS["skinny"]
    A, B = inputs.make_workload(w)
    a, b = dev(A), dev(B)
    ws = gr.splitk_workspace(w.M, w.N, w.K, w.split_k)
    c1 = gr.gemm_relu_splitk(a, b, w.split_k, workspace=ws).clone()
    ws.random_(0, 256)                          # garbage, including the counters
    c2 = gr.gemm_relu_splitk(a, b, w.split_k, workspace=ws).clone()
    c3 = gr.gemm_relu_splitk(a, b, w.split_k, workspace=ws).clone()
    torch.cuda.synchronize()
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))
    assert torch.equal(c1.view(torch.int16), c3.view(torch.int16))


# ----------------------------------------------------------------- exact cases


@pytest.mark.parametrize("M,N,K", [(1537, 1023, 63), (300, 520, 64), (129, 257, 17), (256, 256, 64)])
def test_integer_inputs_bit_exact(orc, M, N, K):
    rng = np.random.default_rng(M + N + K)
    A = rng.integers(-4, 5, (M, K)).astype(np.float16)
    B = rng.integers(-4, 5, (K, N)).astype(np.float16)
    got = run_fused(A, B).astype(np.float64)
    want = orc.gemm_relu_f16(A, B).astype(np.float64)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("n", [200, 256])
def test_identity_gives_relu_of_A(n):
    rng = np.random.default_rng(n)
    A = (rng.standard_normal((n, n)) * 3).astype(np.float16)
    eye = np.eye(n, dtype=np.float16)
    assert np.array_equal(run_fused(A, eye).astype(np.float64), np.maximum(A, 0).astype(np.float64))
    assert np.array_equal(run_fused(eye, A).astype(np.float64), np.maximum(A, 0).astype(np.float64))


def test_ones_zeros_and_negatives():
    for (M, N, K) in [(256, 256, 2048), (131, 70, 300)]:
        ones_a = np.ones((M, K), np.float16)
        ones_b = np.ones((K, N), np.float16)
        assert (run_fused(ones_a, ones_b).astype(np.float64) == K).all()
        assert (run_fused(-ones_a, ones_b).astype(np.float64) == 0).all()
        assert (run_fused(ones_a, np.zeros((K, N), np.float16)).astype(np.float64) == 0).all()


def test_empty_and_k_zero():
    import torch
    c = torch.full((4, 5), 7.0, dtype=torch.float16, device="cuda")
    assert gr.gemm_relu_f16(0, 0, c.data_ptr(), 0, 5, 3, torch.cuda.current_stream().cuda_stream) == gr.OK
    a = torch.empty((4, 0), dtype=torch.float16, device="cuda")
    b = torch.empty((0, 5), dtype=torch.float16, device="cuda")
    out = gr.gemm_relu(a, b, out=c)
    assert (host(out) == 0).all()
    c.fill_(7.0)
    out = gr.gemm_relu_splitk(a, b, 4, out=c)
    assert (host(out) == 0).all()


@pytest.mark.parametrize("M,N,K", [(1537, 1023, 777), (129, 264, 72), (17, 1000, 1000)])
def test_output_guard_band_untouched(M, N, K):
    import torch
    rng = np.random.default_rng(1)
    A = rng.standard_normal((M, K)).astype(np.float16)
    B = rng.standard_normal((K, N)).astype(np.float16)
    pad = 4096
    buf = torch.full((M * N + 2 * pad,), float("nan"), dtype=torch.float16, device="cuda")
    c = buf[pad:pad + M * N].view(M, N)
    gr.gemm_relu(dev(A), dev(B), out=c)
    if K % 8 == 0 and N % 8 == 0:
        gr.gemm_relu_splitk(dev(A), dev(B), 3, out=c)      # two-stage form
        gr.gemm_relu_splitk(dev(A), dev(B), 4, out=c)      # cluster form
    torch.cuda.synchronize()
    assert torch.isnan(buf[:pad]).all() and torch.isnan(buf[pad + M * N:]).all()
    assert not torch.isnan(c).any()


def test_error_growth_is_smooth(orc):
    """The rounding-versus-indexing criterion of the TileLang tutorial's
    numerics section: error against a wider reference that grows smoothly with
    the reduction length is rounding; a jump means a dropped or repeated tile.
    The mean error over positive outputs, relative to the output scale
    sqrt(K), must stay within a small band of its median over K."""
    rng = np.random.default_rng(3)
    rels = []
    for K in (64, 128, 256, 512, 1024, 2048, 4096, 8192):
        A = rng.standard_normal((128, K)).astype(np.float16)
        B = rng.standard_normal((K, 256)).astype(np.float16)
        g = run_fused(A, B).astype(np.float64)
        o = orc.gemm_relu_f16(A, B).astype(np.float64)
        pos = o > 0
        rels.append(float(np.abs(g - o)[pos].mean() / np.sqrt(K)))
    # smooth growth: at most 4x per doubling of K (with a floor for the many
    # exact small-K cases), and far below what one dropped 64-wide k tile gives
    # (a relative error of order 8 / sqrt(K), i.e. > 1e-2 here)
    for a, b in zip(rels, rels[1:]):
        assert b <= 4 * a + 1e-6, rels
    assert max(rels) < 1e-4, rels


# ----------------------------------------------------------------- stream-K

KERNELS = {"one_cta_256": 1, "one_cta_128": 2, "cta_pair": 3}


def _sampled_parity(orc, A, B, got, what, seed=7):
    M, K = A.shape
    N = B.shape[1]
    rows = sorted({r for mb in range((M + 127) // 128) for r in (mb * 128, min(M - 1, mb * 128 + 127))})
    for r0 in range(0, len(rows), 16):
        rr = rows[r0:r0 + 16]
        want = np.concatenate([orc.gemm_relu_f16_rows(A, B, r, 1) for r in rr])
        assert_parity(got[rr], want, abs_dot(A[rr], B), K, (what, "rows", rr[0]))
    rng = np.random.default_rng(seed)
    I = rng.integers(0, M, 2048)
    J = rng.integers(0, N, 2048)
    assert_parity(got[I, J], orc.gemm_relu_f16_at(A, B, I, J), abs_dot(A, B, I, J), K, (what, "samples"))


# Shapes whose tiles leave a thin partial last wave with a long K, so that
# both the CTA-pair and the single-CTA kernel (128 x 256 tiles) take a
# multi-wave stream-K schedule; 2300 x 2300 x 4000 has partial edge tiles and
# a partial last k block.
STREAMK_SHAPES = [(4096, 4096, 4096), (2304, 2304, 4096), (2300, 2300, 4000), (2560, 2560, 4096)]


@pytest.fixture(params=["one_cta_256", "cta_pair"])
def sk_kernel(request):
    """Stream-K runs on the single-CTA kernel and on CTA pairs."""
    gr.gemm_relu_debug_force_kernel(KERNELS[request.param])
    yield request.param
    gr.gemm_relu_debug_force_kernel(0)


@pytest.mark.parametrize("M,N,K", STREAMK_SHAPES)
def test_streamk_parity(orc, sk_kernel, M, N, K):
    import torch
    assert gr.gemm_relu_f16_streamk_workspace_bytes(M, N, K) > 0, "shape has no stream-K part"
    A, B = inputs.make(M, N, K, "normal", True, seed=M + N + K)
    a, b = dev(A), dev(B)
    ws = gr.streamk_workspace(M, N, K)
    ws.random_(0, 256)                                  # contents need no initialisation
    c = gr.gemm_relu_streamk(a, b, workspace=ws)
    got = host(c)
    assert gr.status() == gr.OK
    _sampled_parity(orc, A, B, got, (M, N, K))
    # bit-identical on a second call; close to the data-parallel kernel
    c2 = gr.gemm_relu_streamk(a, b, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(c.view(torch.int16), c2.view(torch.int16))
    ref = gr.gemm_relu(a, b)
    torch.testing.assert_close(c.float(), ref.float(), rtol=1e-2, atol=1e-3)


@pytest.mark.parametrize("M,N,K", STREAMK_SHAPES[1:])
def test_streamk_fixup_orders_give_identical_bits(orc, sk_kernel, M, N, K):
    """The fix-up of a cut tile gives the same bits whichever side finishes
    it: the first k blocks' side adding a pre-loaded piece (normal), adding a
    published piece from global memory after publishing its own first (the
    other side then being second), or the last k blocks' side finishing
    because it publishes late.  Every mode is also checked against the oracle
    on sampled rows and elements."""
    import torch
    A, B = inputs.make(M, N, K, "normal", True, seed=M + 2 * N + K)
    a, b = dev(A), dev(B)
    ws = gr.streamk_workspace(M, N, K)
    outs = {}
    try:
        for mode in (gr.SK_NORMAL, gr.SK_HEAD_PUBLISHES, gr.SK_TAIL_LATE, gr.SK_NORMAL):
            assert gr.gemm_relu_debug_streamk(mode) == gr.OK
            ws.random_(0, 256)
            c = gr.gemm_relu_streamk(a, b, workspace=ws)
            assert gr.status() == gr.OK
            if mode in outs:
                assert torch.equal(c.view(torch.int16), outs[mode].view(torch.int16)), mode
            outs[mode] = c
    finally:
        gr.gemm_relu_debug_streamk(gr.SK_NORMAL)
    for mode, c in outs.items():
        assert torch.equal(c.view(torch.int16), outs[gr.SK_NORMAL].view(torch.int16)), mode
        _sampled_parity(orc, A, B, host(c), (M, N, K, "fix-up mode", mode))


def test_streamk_concurrent_streams(sk_kernel):
    """Stream-K launches on two streams at once (distinct workspaces), beside
    a long library kernel of another stream that holds SMs meanwhile: no
    worker ever waits for another, so every launch completes with the same
    bits as when it runs alone."""
    import torch
    M, N, K = 2304, 2304, 4096
    assert gr.gemm_relu_f16_streamk_workspace_bytes(M, N, K) > 0
    A, B = inputs.make(M, N, K, "normal", True, seed=99)
    a, b = dev(A), dev(B)
    alone = gr.gemm_relu_streamk(a, b, workspace=gr.streamk_workspace(M, N, K))
    big_a = torch.randn(8192, 8192, device="cuda").half()
    s1, s2, s3 = (torch.cuda.Stream() for _ in range(3))
    # every buffer stays referenced until the end: the caching allocator
    # knows only the current stream, not the streams the kernels run on
    keep = [gr.streamk_workspace(M, N, K) for _ in range(8)]
    outs = [torch.empty((M, N), dtype=torch.float16, device="cuda") for _ in range(8)]
    big_c = torch.empty_like(big_a)
    torch.cuda.synchronize()
    gr.gemm_relu(big_a, big_a, out=big_c, stream=s3)   # ~0.6 ms on all SMs
    for i in range(8):
        gr.gemm_relu_streamk(a, b, out=outs[i], workspace=keep[i], stream=(s1, s2)[i % 2])
    torch.cuda.synchronize()
    assert gr.status() == gr.OK
    for c in outs:
        assert torch.equal(c.view(torch.int16), alone.view(torch.int16))


# Shapes whose stream-K schedule is sub-wave (fewer single-CTA tiles than SMs,
# long K), with the pieces per tile (0: the library's choice).  Two pieces cut
# each tile once; more give every tile middle pieces, settled through chains
# of cuts.
SUBWAVE_CASES = [
    (200, 3000, 4096, 0),    # 48 tiles of 64 k blocks: 2 pieces on 96 CTAs
    (128, 2048, 16384, 0),   # 16 tiles of 256 k blocks: 3 pieces on 48 CTAs
    (128, 4096, 8192, 4),    # 32 tiles of 128 k blocks: 4 pieces on 128 CTAs
]


@pytest.mark.parametrize("M,N,K,pieces", SUBWAVE_CASES)
def test_streamk_subwave_parity_and_fixup_orders(orc, M, N, K, pieces):
    """Every element against the oracle, and the same bits in every fix-up
    order: heads adding a published tail, heads always publishing, tails
    late (the rightmost worker of a tile carries the sum through each cut)
    and heads late (the workers left of each cut finish)."""
    import torch
    A, B = inputs.make(M, N, K, "normal", True, seed=M + 3 * N + K)
    a, b = dev(A), dev(B)
    outs = []
    try:
        assert gr.gemm_relu_debug_streamk_pieces(pieces) == gr.OK
        assert gr.gemm_relu_f16_streamk_workspace_bytes(M, N, K) > 0, "no stream-K part"
        ws = gr.streamk_workspace(M, N, K)
        for mode in (gr.SK_NORMAL, gr.SK_HEAD_PUBLISHES, gr.SK_TAIL_LATE, gr.SK_HEAD_LATE,
                     gr.SK_NORMAL):
            assert gr.gemm_relu_debug_streamk(mode) == gr.OK
            ws.random_(0, 256)                      # contents need no initialisation
            outs.append((mode, gr.gemm_relu_streamk(a, b, workspace=ws)))
            assert gr.status() == gr.OK
    finally:
        gr.gemm_relu_debug_streamk(gr.SK_NORMAL)
        gr.gemm_relu_debug_streamk_pieces(0)
    want = oracle_threaded(orc, A, B)
    assert_parity(host(outs[0][1]), want, abs_dot(A, B), K, (M, N, K, pieces, "stream-K"))
    for mode, c in outs[1:]:
        assert torch.equal(c.view(torch.int16), outs[0][1].view(torch.int16)), (M, N, K, mode)


def test_streamk_subwave_on_every_single_cta_width():
    """The sub-wave schedule on the single-CTA kernel forced to 128 x 256
    and to 128 x 128 tiles: repeat calls identical, and close to the plain
    launch."""
    import torch
    M, N, K = 384, 1536, 4096
    A, B = inputs.make(M, N, K, "normal", True, seed=5)
    a, b = dev(A), dev(B)
    try:
        for force in (KERNELS["one_cta_256"], KERNELS["one_cta_128"]):
            gr.gemm_relu_debug_force_kernel(force)
            assert gr.gemm_relu_f16_streamk_workspace_bytes(M, N, K) > 0, force
            ws = gr.streamk_workspace(M, N, K)
            c = gr.gemm_relu_streamk(a, b, workspace=ws)
            c2 = gr.gemm_relu_streamk(a, b, workspace=ws)
            ref = gr.gemm_relu(a, b)
            torch.cuda.synchronize()
            assert gr.status() == gr.OK
            assert torch.equal(c.view(torch.int16), c2.view(torch.int16)), force
            torch.testing.assert_close(c.float(), ref.float(), rtol=1e-2, atol=1e-3)
    finally:
        gr.gemm_relu_debug_force_kernel(0)


# ----------------------------------------------------------------- staged operands

# Row pitches that TMA cannot describe: the stream-K entry point copies A
# and/or B into aligned rows of its workspace and runs the TMA kernel, with
# predicated stores when C's rows are unaligned too.
STAGED_SHAPES = [
    # M, N, K, whether the copies run the single-CTA kernel with no tile cut
    # (then the bits equal the predicated-load kernel's)
    (1537, 1023, 777, True),    # the ragged workload: A and B copied, C stored predicated
    (1000, 1024, 777, True),    # A copied only; B and C aligned (C by TMA)
    (1024, 1001, 1024, True),   # B copied only, C predicated
    (129, 70, 300, True),       # one tile, edges everywhere
    (5000, 37, 13, True),       # K smaller than one k block, narrow N
    (2305, 1031, 333, False),   # CTA pairs, C predicated
    (2048, 2048, 1001, False),  # A copied only; CTA pairs with TMA stores of C
    (2305, 2049, 1031, False),  # CTA pairs with a stream-K schedule, C predicated
]


@pytest.mark.parametrize("M,N,K,same_bits", STAGED_SHAPES)
def test_staged_operands_full(orc, M, N, K, same_bits):
    """Every element of the staged path against the oracle, with the
    workspace and C inside guard bands that must stay untouched."""
    import torch
    n = gr.gemm_relu_f16_streamk_workspace_bytes(M, N, K)
    assert n > 0
    A, B = inputs.make(M, N, K, "normal", True, seed=M + N + 5 * K)
    a, b = dev(A), dev(B)
    pad = 4096
    wbuf = torch.full((n + 2 * pad,), 0x5A, dtype=torch.uint8, device="cuda")
    cbuf = torch.full((M * N + 2 * pad,), float("nan"), dtype=torch.float16, device="cuda")
    c = cbuf[pad:pad + M * N].view(M, N)
    gr.gemm_relu_streamk(a, b, out=c, workspace=wbuf[pad:pad + n])
    torch.cuda.synchronize()
    assert gr.status() == gr.OK
    assert (wbuf[:pad] == 0x5A).all() and (wbuf[pad + n:] == 0x5A).all()
    assert torch.isnan(cbuf[:pad]).all() and torch.isnan(cbuf[pad + M * N:]).all()
    want = oracle_threaded(orc, A, B)
    assert_parity(host(c), want, abs_dot(A, B), K, (M, N, K, "staged"))
    # same bits on a second call (and whatever the workspace held)
    c2 = gr.gemm_relu_streamk(a, b, workspace=wbuf[pad:pad + n].random_(0, 256))
    plain = gr.gemm_relu(a, b)
    torch.cuda.synchronize()
    assert torch.equal(c.view(torch.int16), c2.view(torch.int16))
    if same_bits:
        assert torch.equal(c.view(torch.int16), plain.view(torch.int16))


def test_staged_misaligned_bases(orc):
    """Aligned pitches but operands starting 2 bytes past a 16-byte boundary:
    without room in the workspace the predicated-load kernel runs, with room
    the operands are copied; both meet the contract against the oracle."""
    import torch
    M, N, K = 700, 1536, 512
    A, B = inputs.make(M, N, K, "normal", True, seed=11)
    abuf = torch.empty(M * K + 8, dtype=torch.float16, device="cuda")
    bbuf = torch.empty(K * N + 8, dtype=torch.float16, device="cuda")
    a = abuf[1:1 + M * K].view(M, K)
    b = bbuf[3:3 + K * N].view(K, N)
    a.copy_(torch.from_numpy(A))
    b.copy_(torch.from_numpy(B))
    assert gr.gemm_relu_f16_path(a.data_ptr(), b.data_ptr(), a.data_ptr(), M, N, K) == gr.PATH_LSU
    want = oracle_threaded(orc, A, B)
    tight = gr.streamk_workspace(M, N, K)
    roomy = torch.empty(2 * (M * K + K * N) + 4096, dtype=torch.uint8, device="cuda")
    outs = []
    for ws, what in ((tight, "predicated loads"), (roomy, "copied operands")):
        outs.append(gr.gemm_relu_streamk(a, b, workspace=ws))
        assert gr.status() == gr.OK
        assert_parity(host(outs[-1]), want, abs_dot(A, B), K, (M, N, K, what))
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_staged_workspace_errors():
    """Odd pitches need the workspace the query reports: a smaller or
    misaligned one is refused with GEMMRELU_ERR_WORKSPACE."""
    import torch
    M, N, K = 300, 200, 99
    n = gr.gemm_relu_f16_streamk_workspace_bytes(M, N, K)
    a = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    b = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    c = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    ws = torch.empty(n + 16, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    args = (a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K)
    assert gr.gemm_relu_f16_streamk(*args, ws.data_ptr(), n - 1, s) == gr.ERR_WORKSPACE
    assert gr.gemm_relu_f16_streamk(*args, None, 0, s) == gr.ERR_WORKSPACE
    assert gr.gemm_relu_f16_streamk(*args, ws.data_ptr() + 8, n, s) == gr.ERR_WORKSPACE
    assert gr.gemm_relu_f16_streamk(*args, ws.data_ptr(), n, s) == gr.OK
    torch.cuda.synchronize()


def test_streamk_falls_back_without_a_cut():
    import torch
    # 1024 x 2048 x 512: 32 pair tiles, fewer than the SM pairs, and the
    # pair kernel has no sub-wave schedule -> plain kernel, no workspace
    assert gr.gemm_relu_f16_streamk_workspace_bytes(1024, 2048, 512) == 0
    A, B = inputs.make(1024, 2048, 512, seed=3)
    a, b = dev(A), dev(B)
    c = torch.empty((1024, 2048), dtype=torch.float16, device="cuda")
    rc = gr.gemm_relu_f16_streamk(a.data_ptr(), b.data_ptr(), c.data_ptr(), 1024, 2048, 512,
                                  None, 0, torch.cuda.current_stream().cuda_stream)
    assert rc == gr.OK
    assert torch.equal(c.view(torch.int16), gr.gemm_relu(a, b).view(torch.int16))


# ----------------------------------------------------------------- every kernel variant

@pytest.fixture
def forced_kernel(request):
    gr.gemm_relu_debug_force_kernel(KERNELS[request.param])
    yield request.param
    gr.gemm_relu_debug_force_kernel(0)


@pytest.mark.parametrize("forced_kernel", sorted(KERNELS), indirect=True)
def test_each_kernel_sweep_and_workloads(orc, forced_kernel):
    _sweep(orc, TMA_SHAPES[::3] + [(256, 256, 64), (512, 768, 192), (300, 520, 136)], gr.PATH_TMA)
    for name in ("square1024", "square256"):
        w = inputs.WORKLOADS[name]
        A, B = inputs.make_workload(w)
        assert_parity(run_fused(A, B), orc.gemm_relu_f16(A, B), abs_dot(A, B), w.K,
                      (forced_kernel, name))


@pytest.mark.parametrize("forced_kernel", sorted(KERNELS), indirect=True)
def test_each_kernel_square4096_full(square4096, forced_kernel):
    """Every element of the 4096^3 output of each kernel, plain and with the
    stream-K schedule, against the oracle."""
    w, A, B, want, absab = square4096
    a, b = dev(A), dev(B)
    assert_parity(host(gr.gemm_relu(a, b)), want, absab, w.K, (forced_kernel, "square4096"))
    if gr.gemm_relu_f16_streamk_workspace_bytes(w.M, w.N, w.K) > 0:
        got = host(gr.gemm_relu_streamk(a, b, workspace=gr.streamk_workspace(w.M, w.N, w.K)))
        assert_parity(got, want, absab, w.K, (forced_kernel, "square4096 stream-K"))
    assert gr.status() == gr.OK


@pytest.mark.parametrize("forced_kernel", sorted(KERNELS), indirect=True)
def test_panel_height_changes_only_the_tile_order(forced_kernel):
    """The rasteriser's panel height reorders tiles and nothing else: every
    height gives the same bits on shapes whose last panel is partial.  With
    the stream-K schedule the height also decides which tiles are cut (and so
    summed in two parts): each height is deterministic and within the
    contract of the plain result."""
    import torch
    for (M, N, K) in [(2304, 1792, 384), (1664, 2560, 200), (2305, 1031, 333)]:
        # (the last: odd row pitches, the predicated-load kernel)
        A, B = inputs.make(M, N, K, seed=M + K)
        a, b = dev(A), dev(B)
        ws = gr.streamk_workspace(M, N, K)
        outs = []
        try:
            for rows in (0, 128, 256, 640, 1024, 4096):
                assert gr.gemm_relu_debug_set_panel(rows) == gr.OK
                outs.append((rows, gr.gemm_relu(a, b), gr.gemm_relu_streamk(a, b, workspace=ws),
                             gr.gemm_relu_streamk(a, b, workspace=ws)))
        finally:
            gr.gemm_relu_debug_set_panel(0)
        ref = outs[0][1].float()
        for rows, c, csk, csk2 in outs:
            assert torch.equal(c, outs[0][1]), (forced_kernel, M, N, K, rows)
            assert torch.equal(csk, csk2), (forced_kernel, M, N, K, rows, "stream-K repeat")
            err = (csk.float() - ref).abs()
            assert bool((err <= 1e-2 + 1e-2 * ref.abs()).all()), (forced_kernel, M, N, K, rows)
    assert gr.status() == gr.OK


@pytest.mark.parametrize("forced_kernel", ["cta_pair"], indirect=True)
def test_pair_integer_inputs_bit_exact(orc, forced_kernel):
    rng = np.random.default_rng(21)
    for (M, N, K) in [(520, 776, 64), (256, 256, 32), (1000, 264, 48)]:
        A = rng.integers(-4, 5, (M, K)).astype(np.float16)
        B = rng.integers(-4, 5, (K, N)).astype(np.float16)
        assert np.array_equal(run_fused(A, B).astype(np.float64),
                              orc.gemm_relu_f16(A, B).astype(np.float64))


# ----------------------------------------------------------------- GEMV (M <= 8)

# (M, N, K): every accumulator width (1, 2, 4, 8 rows), M between them, ragged N
# (not a multiple of the 256-column block) and K (not a multiple of 32),
# cluster sizes 1..8
GEMV_CASES = [(1, 8, 8), (1, 8192, 8192), (2, 264, 72), (3, 520, 1000), (4, 136, 4096),
              (5, 1032, 2056), (7, 256, 40), (8, 8192, 1024), (8, 2048, 8200), (6, 16392, 512)]


@pytest.fixture
def forced_gemv():
    gr.gemm_relu_debug_force_kernel(gr.FORCE_GEMV)
    yield
    gr.gemm_relu_debug_force_kernel(gr.FORCE_AUTO)


@pytest.mark.parametrize("M,N,K", GEMV_CASES)
def test_gemv_parity(orc, forced_gemv, M, N, K):
    import torch
    A, B = inputs.make(M, N, K, dist="normal", scale_by_sqrt_k=True, seed=M * 31 + N + K)
    a, b = dev(A), dev(B)
    c = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert gr.gemm_relu_f16_path(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K) == gr.PATH_TMA
    gr.gemm_relu(a, b, out=c)
    assert gr.status() == gr.OK
    assert_parity(host(c), orc.gemm_relu_f16(A, B), abs_dot(A, B), K, (M, N, K))
    again = gr.gemm_relu(a, b)
    assert torch.equal(c.view(torch.int16), again.view(torch.int16))      # fixed order


def test_gemv_integer_inputs_bit_exact(orc, forced_gemv):
    """Small integers: every partial sum is exact in fp32, so GEMV, oracle and
    exact arithmetic agree bit for bit, over all eight rows and ragged tiles."""
    rng = np.random.default_rng(3)
    M, N, K = 8, 776, 1000
    A = rng.integers(-4, 5, (M, K)).astype(np.float16)
    B = rng.integers(-4, 5, (K, N)).astype(np.float16)
    got = run_fused(A, B).astype(np.float64)
    assert np.array_equal(got, orc.gemm_relu_f16(A, B).astype(np.float64))


def test_decode_rows_routing(orc):
    """gemm_relu_f16 on decode-like rows: M <= 2 runs the GEMV kernel (same
    bits as forcing it), and so does M = 4 when the CTA pairs of a split
    would not fit in one wave (N = 16384); M = 4 or 8 with few column tiles
    runs K split in two on CTA pairs (same bits as gemm_relu_f16_splitk with
    split 2); all agree with the oracle and with the tensor-core tile kernel
    within the bounds."""
    import torch
    for M, N, K, route in [(2, 4096, 4096, "gemv"), (4, 16384, 512, "gemv"),
                           (4, 4096, 4096, "split2"), (8, 4096, 4096, "split2")]:
        A, B = inputs.make(M, N, K, dist="uniform", seed=70 + M)
        a, b = dev(A), dev(B)
        auto = gr.gemm_relu(a, b)
        try:
            gr.gemm_relu_debug_force_kernel(gr.FORCE_GEMV)
            gemv = gr.gemm_relu(a, b)
            gr.gemm_relu_debug_force_kernel(gr.FORCE_ONE_CTA_256)
            tile = gr.gemm_relu(a, b)
        finally:
            gr.gemm_relu_debug_force_kernel(gr.FORCE_AUTO)
        split2 = gr.gemm_relu_splitk(a, b, 2)
        assert gr.status() == gr.OK
        same = gemv if route == "gemv" else split2
        assert torch.equal(auto.view(torch.int16), same.view(torch.int16)), (M, N, route)
        want = orc.gemm_relu_f16(A, B)
        for name, got in (("auto", auto), ("gemv", gemv), ("tile", tile), ("split2", split2)):
            assert_parity(host(got), want, abs_dot(A, B), K, (M, name))

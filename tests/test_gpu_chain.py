"""The library's kernels chained on one stream with no host synchronisation
between them.

Every kernel is a programmatic dependent launch: its CTAs may start while the
previous grid still runs, and they wait for it before touching its data.  The
HBM-bound kernels (split-K, GEMV) also ask L2 for their first stages of B
before that wait.  These tests check that no launch moves past the data
dependence on the previous one:
  - read after write: a consumer reads, as A, as B or as the keys of the
    attention kernel, the output the previous launch wrote into a buffer
    that a fill had just set to NaN;
  - write after read: a producer overwrites a buffer the previous launch is
    still reading.
Integer-valued operands make every GEMM exact in fp32, so each GPU stage
equals the oracle's bit for bit and the next stage sees the same input on
both sides; the attention stage is held to the attention tests' bound.
"""
import numpy as np
import pytest

import tiled_tensor_core_03_gb300 as gr

from gpu_common import dev
from test_gpu_attention import _check as check_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.fixture
def split_form(request):
    gr.gemm_relu_debug_force_split(request.param)
    yield request.param
    gr.gemm_relu_debug_force_split(gr.SPLIT_AUTO)


def _ints(rng, shape, lo=-1, hi=1):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float16)


def _same_bits(got, want, what):
    g = np.ascontiguousarray(got).view(np.uint16)
    w = np.ascontiguousarray(want).view(np.uint16)
    bad = np.argwhere(g != w)
    assert bad.size == 0, (what, len(bad), bad[:4].tolist())


# P: T x D; its first S rows are also the keys [1, S, H, HD] of the attention
# stage.  T = 1024 so that the split-K calls contracting over T really split
# (a piece needs at least 256 k of its own).
T, D, S_ATT, H, HD = 1024, 1024, 256, 8, 128
_EXPECTED = {}


def _expected(orc, seed):
    """Inputs and the oracle's chain for one seed (computed once per seed)."""
    if seed not in _EXPECTED:
        rng = np.random.default_rng(seed)
        e = {"X": _ints(rng, (T, 128)), "W": _ints(rng, (128, D)),
             "X2": _ints(rng, (T, 128)), "W2": _ints(rng, (128, D)),
             "A1": _ints(rng, (16, T)), "a2": _ints(rng, (1, T)),
             "W3": _ints(rng, (D, 128)), "W5": _ints(rng, (D, 512)),
             "Q": (_ints(rng, (1, S_ATT, H, HD)).astype(np.float32) / 16).astype(np.float16),
             "V": rng.standard_normal((1, S_ATT, H, HD)).astype(np.float16)}
        e["P"] = orc.gemm_relu_f16(e["X"], e["W"])
        e["Y1"] = orc.gemm_relu_f16(e["A1"], e["P"])
        e["y2"] = orc.gemm_relu_f16(e["a2"], e["P"])
        e["Y3"] = orc.gemm_relu_f16(e["P"], e["W3"])
        e["Z"] = orc.gemm_relu_f16(e["Y1"], e["W5"])
        e["P2"] = orc.gemm_relu_f16(e["X2"], e["W2"])
        e["Y4"] = orc.gemm_relu_f16(e["A1"], e["P2"])
        _EXPECTED[seed] = e
    return _EXPECTED[seed]


@pytest.mark.parametrize("split_form", [gr.SPLIT_AUTO, gr.SPLIT_TWO_STAGE], indirect=True,
                         ids=["auto", "two_stage"])
@pytest.mark.parametrize("seed", [1, 2])
def test_chain_read_after_write_and_write_after_read(torch, orc, split_form, seed):
    e = _expected(orc, seed)
    x, w, x2, w2 = dev(e["X"]), dev(e["W"]), dev(e["X2"]), dev(e["W2"])
    a1, a2d, w3, w5 = dev(e["A1"]), dev(e["a2"]), dev(e["W3"]), dev(e["W5"])
    q, v = dev(e["Q"]), dev(e["V"])
    keys = e["P"][:S_ATT].reshape(1, S_ATT, H, HD)
    nan = float("nan")
    o0 = e.get("O")                     # the same for every split form
    for rep in range(4):
        p = torch.empty((T, D), dtype=torch.float16, device="cuda")
        y1 = torch.empty((16, D), dtype=torch.float16, device="cuda")
        p_seen = torch.empty_like(p)
        for t in (p, y1):
            t.fill_(nan)
        gr.gemm_relu(x, w, out=p)                            # producer
        g1 = gr.gemm_relu_splitk(a1, p, 4, out=y1)           # B from the previous launch
        g2 = gr.gemm_relu(a2d, p)                            # GEMV, B from two launches back
        g3 = gr.gemm_relu(p, w3)                             # A from an earlier launch
        gz = gr.gemm_relu_splitk(y1, w5, 2)                  # A from a split-K launch
        o = gr.flash_attention(q, p[:S_ATT].view(1, S_ATT, H, HD), v)  # keys, earlier launch
        p_seen.copy_(p)
        gr.gemm_relu(x2, w2, out=p)                          # overwrites what was just read
        g4 = gr.gemm_relu_splitk(a1, p, 2)                   # and reads the new contents
        assert gr.status() == gr.OK                          # synchronises
        _same_bits(p_seen.cpu().numpy(), e["P"], ("P", rep))
        _same_bits(g1.cpu().numpy(), e["Y1"], ("Y1", rep))
        _same_bits(g2.cpu().numpy(), e["y2"], ("y2", rep))
        _same_bits(g3.cpu().numpy(), e["Y3"], ("Y3", rep))
        _same_bits(gz.cpu().numpy(), e["Z"], ("Z", rep))
        _same_bits(g4.cpu().numpy(), e["Y4"], ("Y4", rep))
        _same_bits(p.cpu().numpy(), e["P2"], ("P2", rep))
        if o0 is None:                   # the oracle once; later runs give the same bits
            o0 = o.cpu().numpy()
            check_attention(orc, o0, e["Q"], keys, e["V"], False)
            e["O"] = o0
        else:
            _same_bits(o.cpu().numpy(), o0, ("O", rep))


def test_chain_long_run_of_dependent_splits(torch, orc):
    """Twelve split-K launches in a row, each reading the previous one's
    output as A and multiplying it by a permutation matrix (so the values
    stay bounded and a stale read shows as a wrong column order or a NaN).
    The outputs alternate between two buffers: every launch overwrites the
    buffer the launch before it was reading."""
    rng = np.random.default_rng(7)
    n = 1024                                         # 4 pieces of 256 k
    Ws = []
    for _ in range(3):
        W = np.zeros((n, n), np.float16)
        W[np.arange(n), rng.permutation(n)] = 1.0
        Ws.append(W)
    A0 = _ints(rng, (16, n), -4, 4)
    want = [A0]
    for i in range(12):
        want.append(orc.gemm_relu_f16(want[-1], Ws[i % 3]))
    ws = [dev(Wi) for Wi in Ws]
    bufs = [torch.full((16, n), float("nan"), dtype=torch.float16, device="cuda")
            for _ in range(2)]
    cur = dev(A0)
    for i in range(12):
        out = bufs[i % 2]
        gr.gemm_relu_splitk(cur, ws[i % 3], 4, out=out)
        cur = out
    assert gr.status() == gr.OK
    _same_bits(bufs[1].cpu().numpy(), want[12], "stage 12")
    _same_bits(bufs[0].cpu().numpy(), want[11], "stage 11")

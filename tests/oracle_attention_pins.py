"""Pins of the attention oracle to things other than itself.

Each pin takes an oracle.Oracle and raises AssertionError on a mismatch.  They
fix what the FlashAttention section of the TileLang tutorial pages defines --
O = softmax(Q K^T / sqrt(d)) V per (batch, head), keys j <= i only when causal,
fp16 output -- through:
  - an exact high-precision evaluation (mpmath, 60 digits) on tiny inputs,
    written independently of the C code;
  - closed forms: one key, the causal first row, constant scores (the mean of
    the visible V rows, exact in rationals), all-ones V, a dominant key;
  - invariants: a constant shift of one query's scores, a joint permutation of
    the keys and values (non-causal), heads and batches being independent.
"""
from fractions import Fraction

import numpy as np


def _rand(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def _f16_of_fraction(x):
    """binary16 nearest to a rational x (via the nearest double, then numpy's
    float64 -> float16 rounding, which is independent of the oracle)."""
    return np.float16(float(x))


def pin_mpmath_exact(o):
    """60-digit evaluation of the definition, rounded to fp16, equals the
    oracle bit for bit, causal and not, several head dims and scales."""
    import mpmath
    mpmath.mp.dps = 60
    for seed, (b, s, h, d), scale in [(1, (2, 5, 3, 8), 1.0), (2, (1, 7, 2, 4), 2.0),
                                      (3, (1, 3, 1, 16), 0.5), (4, (2, 4, 2, 5), 3.0)]:
        Q, K, V = _rand((b, s, h, d), seed, scale), _rand((b, s, h, d), seed + 10, scale), \
            _rand((b, s, h, d), seed + 20)
        for causal in (False, True):
            got = o.attention_f16(Q, K, V, causal)
            for bb in range(b):
                for hh in range(h):
                    for i in range(s):
                        vis = range(i + 1) if causal else range(s)
                        sc = [mpmath.fsum(mpmath.mpf(float(Q[bb, i, hh, c])) *
                                          mpmath.mpf(float(K[bb, j, hh, c])) for c in range(d))
                              / mpmath.sqrt(d) for j in vis]
                        w = [mpmath.exp(x) for x in sc]
                        z = mpmath.fsum(w)
                        for c in range(d):
                            num = mpmath.fsum(wj * mpmath.mpf(float(V[bb, j, hh, c]))
                                              for wj, j in zip(w, vis))
                            want = np.float16(float(num / z))
                            g = got[bb, i, hh, c]
                            assert g == want or (np.isnan(g) and np.isnan(want)), \
                                (seed, causal, bb, i, hh, c, g, want)


def pin_single_key(o):
    """seq = 1: the only key gets weight 1, so O = V exactly."""
    Q, K, V = _rand((2, 1, 3, 16), 5), _rand((2, 1, 3, 16), 6), _rand((2, 1, 3, 16), 7)
    for causal in (False, True):
        assert np.array_equal(o.attention_f16(Q, K, V, causal).view(np.uint16), V.view(np.uint16))


def pin_causal_first_row(o):
    """Causal: query 0 sees key 0 only, so O[:, 0] = V[:, 0] exactly; and the
    last query sees every key, so it equals the non-causal result."""
    Q, K, V = _rand((2, 9, 2, 8), 8), _rand((2, 9, 2, 8), 9), _rand((2, 9, 2, 8), 10)
    oc = o.attention_f16(Q, K, V, True)
    on = o.attention_f16(Q, K, V, False)
    assert np.array_equal(oc[:, 0].view(np.uint16), V[:, 0].view(np.uint16))
    assert np.array_equal(oc[:, -1].view(np.uint16), on[:, -1].view(np.uint16))
    assert not np.array_equal(oc[:, 1].view(np.uint16), on[:, 1].view(np.uint16))


def pin_constant_scores_give_mean(o):
    """K = 0: every score is 0, the weights are equal, and O[i] is the mean of
    the visible V rows (computed here in exact rationals)."""
    b, s, h, d = 1, 6, 2, 4
    Q = _rand((b, s, h, d), 11)
    K = np.zeros((b, s, h, d), np.float16)
    V = _rand((b, s, h, d), 12)
    for causal in (False, True):
        got = o.attention_f16(Q, K, V, causal)
        for i in range(s):
            n = i + 1 if causal else s
            for hh in range(h):
                for c in range(d):
                    mean = sum(Fraction(float(V[0, j, hh, c])) for j in range(n)) / n
                    assert got[0, i, hh, c] == _f16_of_fraction(mean), (causal, i, hh, c)


def pin_ones_value(o):
    """V = 1 everywhere: the weights sum to 1, so O = 1."""
    Q, K = _rand((2, 8, 2, 8), 13, 3.0), _rand((2, 8, 2, 8), 14, 3.0)
    V = np.ones((2, 8, 2, 8), np.float16)
    for causal in (False, True):
        assert (o.attention_f16(Q, K, V, causal) == np.float16(1.0)).all()


def pin_dominant_key(o):
    """Key p(i) scores 40 above every other key for query i: its weight is
    1 - O(e^-40), so O[i] = V[p(i)] to fp16 precision."""
    s, d = 6, 8
    perm = [3, 0, 5, 1, 4, 2]
    Q = np.zeros((1, s, 1, d), np.float16)
    K = np.zeros((1, s, 1, d), np.float16)
    for j in range(s):
        K[0, j, 0, j] = 1.0                       # key j = unit vector e_j
    for i in range(s):
        Q[0, i, 0, perm[i]] = 40.0 * np.sqrt(d)   # score 40 on key perm[i], 0 elsewhere
    V = _rand((1, s, 1, d), 15)
    got = o.attention_f16(Q, K, V, False)
    for i in range(s):
        assert np.array_equal(got[0, i, 0].view(np.uint16), V[0, perm[i], 0].view(np.uint16)), i


def pin_shift_invariance(o):
    """A constant added to all of one query's scores leaves its output alone:
    with K[..., 0] = 1 for every key, adding c to Q[..., 0] shifts every score
    of that query by c / sqrt(d).  Equal within one fp16 unit."""
    Q, K, V = _rand((1, 7, 2, 8), 16), _rand((1, 7, 2, 8), 17), _rand((1, 7, 2, 8), 18)
    K[..., 0] = 1.0
    Q2 = Q.copy()
    Q2[..., 0] = (Q2[..., 0].astype(np.float32) + 4.0).astype(np.float16)
    for causal in (False, True):
        a = o.attention_f16(Q, K, V, causal).astype(np.float64)
        b = o.attention_f16(Q2, K, V, causal).astype(np.float64)
        ulp = np.spacing(np.abs(a).astype(np.float16)).astype(np.float64)
        assert (np.abs(a - b) <= ulp).all()


def pin_permutation_invariance(o):
    """Non-causal: permuting the keys together with their values leaves O alone
    (within one fp16 unit: the summation order changes)."""
    Q, K, V = _rand((1, 9, 2, 8), 19), _rand((1, 9, 2, 8), 20), _rand((1, 9, 2, 8), 21)
    p = np.random.default_rng(22).permutation(9)
    a = o.attention_f16(Q, K, V, False).astype(np.float64)
    b = o.attention_f16(Q, K[:, p], V[:, p], False).astype(np.float64)
    ulp = np.spacing(np.abs(a).astype(np.float16)).astype(np.float64)
    assert (np.abs(a - b) <= ulp).all()


def pin_heads_and_batches_independent(o):
    """Each (batch, head) is its own problem: computing one of them alone (as
    a batch-1, head-1 problem) gives the same bits, and the rows entry point
    agrees with the full one."""
    Q, K, V = _rand((2, 5, 3, 8), 23), _rand((2, 5, 3, 8), 24), _rand((2, 5, 3, 8), 25)
    for causal in (False, True):
        full = o.attention_f16(Q, K, V, causal)
        for bb in range(2):
            for hh in range(3):
                one = o.attention_f16(Q[bb:bb + 1, :, hh:hh + 1].copy(),
                                      K[bb:bb + 1, :, hh:hh + 1].copy(),
                                      V[bb:bb + 1, :, hh:hh + 1].copy(), causal)
                assert np.array_equal(one[0, :, 0].view(np.uint16), full[bb, :, hh].view(np.uint16))
                rows = o.attention_f16_rows(Q, K, V, causal, bb, hh, 1, 3)
                assert np.array_equal(rows.view(np.uint16), full[bb, 1:4, hh].view(np.uint16))


PINS = [pin_mpmath_exact, pin_single_key, pin_causal_first_row, pin_constant_scores_give_mean,
        pin_ones_value, pin_dominant_key, pin_shift_invariance, pin_permutation_invariance,
        pin_heads_and_batches_independent]

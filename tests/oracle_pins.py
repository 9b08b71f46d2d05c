"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin takes an `oracle.Oracle` and raises AssertionError on a mismatch.
They are collected by tests/test_oracle.py, which also runs them against
deliberately broken copies of the oracle to show each planted mistake is
caught by at least one pin.

What pins what:
  decode / round-trip / midpoints / random doubles  -> the binary16 rounding,
      against numpy's own float64 -> float16 conversion (an independent
      library routine) and against the format definition;
  hand-worked goldens (tests/golden/*.json)         -> the whole path on
      values worked out by hand from the quickstart's definition;
  exact rational brute force                        -> the sum, the ReLU and
      the rounding, via Python Fractions and an independent nearest-value
      search over the table of all binary16 values;
  closed forms (identity, zeros, ones, rank 1, one k plane, K = 0);
  numpy fp64 matmul and int64 matmul                -> indexing and operand
      orientation on larger shapes;
  invariants                                        -> C >= 0, C = f16(max(P, 0)).
"""
import bisect
import json
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# ---------------------------------------------------------------- helpers


def _f16(x):
    return np.asarray(x, dtype=np.float16)


def _bits(x):
    return np.ascontiguousarray(_f16(x)).view(np.uint16)


def _same_values(a, b):
    """Equal as fp16 values (+0 == -0), NaN never expected."""
    a = np.asarray(a, dtype=np.float64)
    b = np.broadcast_to(np.asarray(b, dtype=np.float64), a.shape)
    return np.array_equal(a, b)


_TABLE_BITS = np.arange(0, 0x7C00, dtype=np.uint16)          # +0 .. 65504
_TABLE_VALS = [Fraction(float(v)) for v in _TABLE_BITS.view(np.float16).astype(np.float64)]


def exact_to_f16_nonneg(fr):
    """Round a non-negative Fraction to binary16 bits, nearest, ties to even.

    Independent of the oracle: a search in the sorted table of every finite
    non-negative binary16 value.  Beyond 65504 the next 'even' neighbour is
    2^16 (infinity), so the midpoint 65520 and above go to infinity.
    """
    assert fr >= 0
    if fr >= Fraction(65520):
        return 0x7C00
    idx = bisect.bisect_left(_TABLE_VALS, fr)
    if _TABLE_VALS[idx] == fr:
        return int(_TABLE_BITS[idx])
    lo, hi = idx - 1, idx
    dlo = fr - _TABLE_VALS[lo]
    dhi = _TABLE_VALS[hi] - fr
    if dlo < dhi:
        return int(_TABLE_BITS[lo])
    if dhi < dlo:
        return int(_TABLE_BITS[hi])
    return int(_TABLE_BITS[lo]) if (int(_TABLE_BITS[lo]) & 1) == 0 else int(_TABLE_BITS[hi])


def exact_gemm_relu_bits(A, B):
    A64 = _f16(A).astype(np.float64)
    B64 = _f16(B).astype(np.float64)
    M, K = A64.shape
    N = B64.shape[1]
    Af = [[Fraction(float(x)) for x in row] for row in A64]
    Bf = [[Fraction(float(x)) for x in row] for row in B64]
    out = np.zeros((M, N), dtype=np.uint16)
    for i in range(M):
        for j in range(N):
            s = sum((Af[i][k] * Bf[k][j] for k in range(K)), Fraction(0))
            out[i, j] = exact_to_f16_nonneg(max(s, Fraction(0)))
    return out


# ---------------------------------------------------------------- binary16 pins


def pin_decode_all_patterns(o):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([o.f16_to_f64(b) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_roundtrip_all_patterns(o):
    bits = np.arange(65536, dtype=np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    for b, v in zip(bits, vals):
        if np.isnan(v):
            continue
        assert o.f64_to_f16(v) == b, (hex(b), v)


def pin_midpoints(o):
    """Every midpoint between neighbouring positive binary16 values goes to the
    even significand; one fp64 ulp either side goes to the nearer neighbour.
    Checked against the format rule and against numpy's conversion."""
    bits = np.arange(0, 0x7BFF, dtype=np.uint16)                # pairs (b, b+1)
    lo = bits.view(np.float16).astype(np.float64)
    hi = (bits + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2.0                                       # exact in fp64
    even = np.where(bits % 2 == 0, bits, bits + 1).astype(np.uint16)
    assert np.array_equal(mid.astype(np.float16).view(np.uint16), even)
    up = np.nextafter(mid, np.inf)
    dn = np.nextafter(mid, -np.inf)
    for k in range(bits.size):
        assert o.f64_to_f16(mid[k]) == even[k], (hex(bits[k]), mid[k])
        assert o.f64_to_f16(up[k]) == bits[k] + 1, (hex(bits[k]), up[k])
        assert o.f64_to_f16(dn[k]) == bits[k], (hex(bits[k]), dn[k])
        assert o.f64_to_f16(-mid[k]) == (even[k] | 0x8000)


def pin_overflow_and_tiny(o):
    cases = {
        65504.0: 0x7BFF,
        65519.99: 0x7BFF,
        65520.0: 0x7C00,            # midpoint to 2^16 ties to 'even' infinity
        65536.0: 0x7C00,
        1e30: 0x7C00,
        float("inf"): 0x7C00,
        2.0 ** -24: 0x0001,         # smallest subnormal
        2.0 ** -25: 0x0000,         # half of it: tie to even zero
        np.nextafter(2.0 ** -25, 1.0): 0x0001,
        3 * 2.0 ** -25: 0x0002,     # 1.5 * 2^-24: tie to even 2 * 2^-24
        2.0 ** -14: 0x0400,         # smallest normal
        2.0 ** -14 - 2.0 ** -25: 0x0400,  # tie between 0x3ff and 0x400: even 0x400
        1.0: 0x3C00,
        0.0: 0x0000,
    }
    for x, want in cases.items():
        assert o.f64_to_f16(x) == want, (x, hex(o.f64_to_f16(x)), hex(want))
        assert o.f64_to_f16(-x) == (want | 0x8000), x


def pin_random_doubles(o, n=60000, seed=7):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n) * np.exp2(rng.uniform(-30, 17, n))
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    for k in range(n):
        assert o.f64_to_f16(x[k]) == want[k], (x[k], hex(want[k]))


# ---------------------------------------------------------------- GEMM pins


def pin_hand_goldens(o):
    for name in sorted(os.listdir(GOLDEN)):
        if not name.startswith("hand_"):
            continue
        with open(os.path.join(GOLDEN, name)) as f:
            g = json.load(f)
        A = _f16(g["A"])
        B = _f16(g["B"])
        want = _f16([[float(v) for v in row] for row in g["C"]])
        got = o.gemm_relu_f16(A, B)
        assert np.array_equal(got.view(np.uint16), want.view(np.uint16)), (name, got, want)
        if "pre_activation" in g:
            assert np.array_equal(o.gemm_f64(A, B), np.asarray(g["pre_activation"], np.float64))


def pin_exact_bruteforce(o, seed=11):
    rng = np.random.default_rng(seed)
    shapes = [(1, 1, 1), (2, 3, 4), (5, 4, 3), (3, 5, 7), (6, 6, 6), (4, 7, 8), (1, 8, 5)]
    scales = [1.0, 1e-3, 30.0, 200.0]
    for (M, N, K) in shapes:
        for sc in scales:
            A = _f16(rng.standard_normal((M, K)) * sc)
            B = _f16(rng.standard_normal((K, N)) * sc)
            want = exact_gemm_relu_bits(A, B)
            got = o.gemm_relu_f16(A, B).view(np.uint16)
            assert np.array_equal(got, want), ((M, N, K, sc), got, want)


def pin_closed_forms(o, seed=13):
    rng = np.random.default_rng(seed)
    for n in (1, 5, 16, 33):
        A = _f16(rng.standard_normal((n, n)) * 4)
        eye = np.eye(n, dtype=np.float16)
        # A . I = A, so ReLU(A . I) = ReLU(A), bit for bit.
        assert _same_values(o.gemm_relu_f16(A, eye), np.maximum(A, 0))
        assert _same_values(o.gemm_relu_f16(eye, A), np.maximum(A, 0))
        # a zero factor gives zero.
        assert _same_values(o.gemm_relu_f16(A, np.zeros((n, n), np.float16)), 0)
    for (M, N, K) in [(3, 4, 1), (2, 2, 7), (4, 3, 64), (2, 5, 2048)]:
        ones = o.gemm_relu_f16(np.ones((M, K), np.float16), np.ones((K, N), np.float16))
        assert _same_values(ones, np.full((M, N), K))
        neg = o.gemm_relu_f16(-np.ones((M, K), np.float16), np.ones((K, N), np.float16))
        assert _same_values(neg, 0)
    # rank one: K = 1 gives ReLU(u_i v_j), one rounding of an exact product.
    u = _f16(rng.standard_normal((9, 1)) * 50)
    v = _f16(rng.standard_normal((1, 11)) * 50)
    want = np.maximum(u.astype(np.float64) * v.astype(np.float64), 0).astype(np.float16)
    assert np.array_equal(o.gemm_relu_f16(u, v).view(np.uint16), want.view(np.uint16))
    # one non-zero k plane picks out one product.
    M, N, K = 6, 7, 10
    A = np.zeros((M, K), np.float16)
    B = np.zeros((K, N), np.float16)
    A[:, 3] = _f16(rng.standard_normal(M) * 3)
    B[3, :] = _f16(rng.standard_normal(N) * 3)
    B[4, :] = _f16(rng.standard_normal(N) * 3)     # pairs with a zero column of A
    want = np.maximum(np.outer(A[:, 3].astype(np.float64), B[3].astype(np.float64)), 0)
    assert np.array_equal(o.gemm_relu_f16(A, B).view(np.uint16),
                          want.astype(np.float16).view(np.uint16))
    # K = 0: the empty sum is 0.
    assert _same_values(o.gemm_relu_f16(np.zeros((3, 0), np.float16),
                                        np.zeros((0, 4), np.float16)), 0)


def pin_vs_numpy_fp64(o, seed=17):
    rng = np.random.default_rng(seed)
    for (M, N, K) in [(37, 29, 61), (64, 48, 130), (5, 90, 300)]:
        A = _f16(rng.standard_normal((M, K)))
        B = _f16(rng.standard_normal((K, N)))
        A64 = A.astype(np.float64)
        B64 = B.astype(np.float64)
        P = o.gemm_f64(A, B)
        ref = A64 @ B64
        bound = 1e-13 * (np.abs(A64) @ np.abs(B64)) + 1e-300
        assert (np.abs(P - ref) <= bound).all()
        C = o.gemm_relu_f16(A, B)
        R = np.maximum(ref, 0).astype(np.float16)
        # identical unless the two fp64 sums straddle an fp16 rounding boundary
        diff = np.abs(C.astype(np.float64) - R.astype(np.float64))
        ulp = np.spacing(np.abs(R).astype(np.float16)).astype(np.float64)
        assert (diff <= ulp).all()
        assert (C.view(np.uint16) != R.view(np.uint16)).mean() < 1e-3


def pin_integer_exact(o, seed=19):
    rng = np.random.default_rng(seed)
    for (M, N, K) in [(17, 23, 64), (40, 8, 31), (3, 100, 50)]:
        Ai = rng.integers(-4, 5, (M, K))
        Bi = rng.integers(-4, 5, (K, N))
        want = np.maximum(Ai @ Bi, 0).astype(np.float16)    # |sum| <= 1024: exact
        got = o.gemm_relu_f16(Ai.astype(np.float16), Bi.astype(np.float16))
        assert np.array_equal(got.view(np.uint16), want.view(np.uint16))


def pin_invariants(o, seed=23):
    rng = np.random.default_rng(seed)
    A = _f16(rng.standard_normal((31, 45)))
    B = _f16(rng.standard_normal((45, 27)))
    C = o.gemm_relu_f16(A, B)
    P = o.gemm_f64(A, B)
    assert (C.astype(np.float64) >= 0).all()
    assert not np.signbit(C.astype(np.float64)).any()          # ReLU gives +0
    want = np.array([[o.f64_to_f16(max(p, 0.0)) for p in row] for row in P], np.uint16)
    assert np.array_equal(C.view(np.uint16), want)
    # ReLU is idempotent: feeding C back through an identity changes nothing.
    eye = np.eye(C.shape[1], dtype=np.float16)
    assert np.array_equal(o.gemm_relu_f16(C, eye).view(np.uint16), C.view(np.uint16))
    # per-row and per-element entry points agree with the full product.
    rows = o.gemm_relu_f16_rows(A, B, 7, 9)
    assert np.array_equal(rows.view(np.uint16), C[7:16].view(np.uint16))
    I = rng.integers(0, 31, 50)
    J = rng.integers(0, 27, 50)
    at = o.gemm_relu_f16_at(A, B, I, J)
    assert np.array_equal(at.view(np.uint16), C[I, J].view(np.uint16))


PINS = [
    pin_decode_all_patterns,
    pin_roundtrip_all_patterns,
    pin_midpoints,
    pin_overflow_and_tiny,
    pin_random_doubles,
    pin_hand_goldens,
    pin_exact_bruteforce,
    pin_closed_forms,
    pin_vs_numpy_fp64,
    pin_integer_exact,
    pin_invariants,
]


def failing_pins(o):
    """Names of the pins that fail (or crash) for oracle `o`."""
    bad = []
    for pin in PINS:
        try:
            pin(o)
        except Exception:  # noqa: BLE001 - any failure counts
            bad.append(pin.__name__)
    return bad

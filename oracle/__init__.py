"""CPU oracles for C = fp16(max(A . B, 0)) and for attention forward
O = fp16(softmax(Q K^T / sqrt(d)) V) -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package entry point's smoke check and the benchmark's
CPU-baseline leg may import this package.  The product path (the CUDA library
and its Python binding) never imports, links or executes it.

The arithmetic lives in gemm_relu_oracle.c (fp64 triple loop, ReLU on the
accumulator, one round-to-nearest-even to binary16) and attention_oracle.c
(fp64 scores, softmax and weighted sum of V, one rounding); this module only
marshals numpy arrays through ctypes.
"""
import ctypes
import os

import numpy as np

from . import build_oracle

_lib = None


def load(path=None):
    """Load (building first if stale) the oracle shared library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if build_oracle.needs_build():
            build_oracle.build()
        _lib = _bind(ctypes.CDLL(build_oracle.LIB))
    return _lib


def _bind(lib):
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f64.restype = ctypes.c_double
    lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
    lib.oracle_f64_to_f16.restype = ctypes.c_uint16
    lib.oracle_gemm_f64.argtypes = [p, p, p, i64, i64, i64]
    lib.oracle_gemm_f64.restype = None
    lib.oracle_gemm_relu_f16.argtypes = [p, p, p, i64, i64, i64]
    lib.oracle_gemm_relu_f16.restype = None
    lib.oracle_gemm_relu_f16_rows.argtypes = [p, p, p, i64, i64, i64, i64]
    lib.oracle_gemm_relu_f16_rows.restype = None
    lib.oracle_gemm_relu_f16_at.argtypes = [p, p, i64, i64, i64, p, p, i64, p]
    lib.oracle_gemm_relu_f16_at.restype = None
    lib.oracle_attention_f16.argtypes = [p, p, p, p, i64, i64, i64, i64, ctypes.c_int]
    lib.oracle_attention_f16.restype = None
    lib.oracle_attention_f16_rows.argtypes = [p, p, p, p, i64, i64, i64, ctypes.c_int,
                                              i64, i64, i64, i64]
    lib.oracle_attention_f16_rows.restype = None
    return lib


def _h(x):
    """View an fp16 array as contiguous uint16 bits."""
    x = np.ascontiguousarray(x)
    assert x.dtype in (np.float16, np.uint16), x.dtype
    return x.view(np.uint16)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """numpy front end over one loaded oracle library."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    def f16_to_f64(self, bits):
        return self.lib.oracle_f16_to_f64(int(bits))

    def f64_to_f16(self, x):
        return self.lib.oracle_f64_to_f16(float(x))

    def gemm_f64(self, A, B):
        A, B = _h(A), _h(B)
        M, K = A.shape
        K2, N = B.shape
        assert K == K2
        P = np.empty((M, N), dtype=np.float64)
        self.lib.oracle_gemm_f64(_ptr(A), _ptr(B), _ptr(P), M, N, K)
        return P

    def gemm_relu_f16(self, A, B):
        A, B = _h(A), _h(B)
        M, K = A.shape
        K2, N = B.shape
        assert K == K2
        C = np.empty((M, N), dtype=np.uint16)
        self.lib.oracle_gemm_relu_f16(_ptr(A), _ptr(B), _ptr(C), M, N, K)
        return C.view(np.float16)

    def gemm_relu_f16_rows(self, A, B, row0, nrows):
        A, B = _h(A), _h(B)
        M, K = A.shape
        N = B.shape[1]
        assert 0 <= row0 and row0 + nrows <= M
        C = np.empty((nrows, N), dtype=np.uint16)
        self.lib.oracle_gemm_relu_f16_rows(_ptr(A), _ptr(B), _ptr(C), N, K, row0, nrows)
        return C.view(np.float16)

    def gemm_relu_f16_at(self, A, B, I, J):
        A, B = _h(A), _h(B)
        M, K = A.shape
        N = B.shape[1]
        I = np.ascontiguousarray(I, dtype=np.int64)
        J = np.ascontiguousarray(J, dtype=np.int64)
        assert I.shape == J.shape
        assert (I >= 0).all() and (I < M).all() and (J >= 0).all() and (J < N).all()
        out = np.empty(I.shape, dtype=np.uint16)
        self.lib.oracle_gemm_relu_f16_at(_ptr(A), _ptr(B), M, N, K, _ptr(I), _ptr(J),
                                         I.size, _ptr(out))
        return out.view(np.float16)

    # ------------------------------------------------------------ attention

    def attention_f16(self, Q, K, V, causal):
        """O = fp16(softmax(Q K^T / sqrt(d)) V) for [batch, seq, heads, dim] fp16
        arrays (key j visible to query i iff j <= i when causal)."""
        Q, K, V = _h(Q), _h(K), _h(V)
        assert Q.ndim == 4 and Q.shape == K.shape == V.shape, (Q.shape, K.shape, V.shape)
        b, s, h, d = Q.shape
        O = np.empty_like(Q)
        self.lib.oracle_attention_f16(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), b, s, h, d,
                                      1 if causal else 0)
        return O.view(np.float16)

    def attention_f16_rows(self, Q, K, V, causal, b, h, row0, nrows):
        """Rows [row0, row0 + nrows) of O for batch b, head h: (nrows, dim) fp16."""
        Q, K, V = _h(Q), _h(K), _h(V)
        B, s, H, d = Q.shape
        assert 0 <= b < B and 0 <= h < H and 0 <= row0 and row0 + nrows <= s
        O = np.zeros_like(Q)
        self.lib.oracle_attention_f16_rows(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), s, H, d,
                                           1 if causal else 0, b, h, row0, nrows)
        return O.view(np.float16)[b, row0:row0 + nrows, h, :].copy()

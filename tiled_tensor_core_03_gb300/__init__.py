"""Fused fp16 GEMM + ReLU for GB300 (sm_103a): Python binding of libgemmrelu.so.

    C = fp16(max(A @ B, 0)),  A: M x K, B: K x N, row-major fp16, fp32 accumulate.

The functions named like the C entry points (gemm_relu_f16, ...) take raw
device pointers and sizes exactly as the C ABI in include/gemm_relu.h does;
`gemm_relu` and `gemm_relu_splitk` accept torch tensors and only marshal
arguments (PyTorch supplies device memory and streams).  Every arithmetic
step runs in the library's CUDA kernels; if the library is missing this
module raises instead of computing anything another way.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgemmrelu.so")

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED_DEVICE = 2
ERR_WORKSPACE = 3
ERR_LAUNCH = 4
ERR_TIMEOUT = 5
ERR_CUDA = 6
ERR_SCRATCH_LIMIT = 7
NOALLOC_SCRATCH_BYTES = 8 << 20

PATH_NONE, PATH_TMA, PATH_LSU = 0, 1, 2
(KERNEL_PAIR, KERNEL_ONE_CTA_256, KERNEL_ONE_CTA_128, KERNEL_PREDICATED, KERNEL_GEMV,
 KERNEL_SPLITK_PAIR) = 1, 2, 3, 4, 5, 6
KERNEL_NAMES = {KERNEL_PAIR: "CTA-pair kernel (256 x 256 tiles)",
                KERNEL_ONE_CTA_256: "single-CTA kernel (128 x 256 tiles)",
                KERNEL_ONE_CTA_128: "single-CTA kernel (128 x 128 tiles)",
                KERNEL_PREDICATED: "predicated-load kernel (128 x 128 tiles)",
                KERNEL_GEMV: "GEMV kernel",
                KERNEL_SPLITK_PAIR: "split-K CTA-pair form (split 2)"}

_lib = None


class GemmReluError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} (status {code})" if what else strerror(code))


def lib():
    """Load libgemmrelu.so (built by __graft_entry__.build() or _build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        L.gemm_relu_f16.argtypes = [vp, vp, vp, i64, i64, i64, vp]
        L.gemm_relu_f16.restype = i32
        L.gemm_relu_f16_splitk_workspace_bytes.argtypes = [i64, i64, i64, i32]
        L.gemm_relu_f16_splitk_workspace_bytes.restype = sz
        L.gemm_relu_f16_splitk.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp, sz, vp]
        L.gemm_relu_f16_splitk.restype = i32
        L.gemm_relu_f16_streamk_workspace_bytes.argtypes = [i64, i64, i64]
        L.gemm_relu_f16_streamk_workspace_bytes.restype = sz
        L.gemm_relu_f16_streamk.argtypes = [vp, vp, vp, i64, i64, i64, vp, sz, vp]
        L.gemm_relu_f16_streamk.restype = i32
        L.gemm_relu_f16_splitk_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp]
        L.gemm_relu_f16_splitk_noalloc.restype = i32
        L.gemm_relu_status.argtypes = [vp]
        L.gemm_relu_status.restype = i32
        L.gemm_relu_strerror.argtypes = [i32]
        L.gemm_relu_strerror.restype = ctypes.c_char_p
        L.gemm_relu_f16_path.argtypes = [vp, vp, vp, i64, i64, i64]
        L.gemm_relu_f16_path.restype = i32
        L.gemm_relu_f16_kernel.argtypes = [vp, vp, vp, i64, i64, i64]
        L.gemm_relu_f16_kernel.restype = i32
        L.gemm_relu_tile_coord.argtypes = [i64, i64, i64, i32, ctypes.POINTER(i64),
                                           ctypes.POINTER(i64)]
        L.gemm_relu_tile_coord.restype = i32
        L.gemm_relu_debug_force_kernel.argtypes = [i32]
        L.gemm_relu_debug_force_kernel.restype = i32
        L.gemm_relu_debug_force_split.argtypes = [i32]
        L.gemm_relu_debug_force_split.restype = i32
        L.flash_attention_f16.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i32, vp]
        L.flash_attention_f16.restype = i32
        L.gemm_relu_debug_streamk.argtypes = [i32]
        L.gemm_relu_debug_streamk.restype = i32
        L.gemm_relu_debug_streamk_pieces.argtypes = [i32]
        L.gemm_relu_debug_streamk_pieces.restype = i32
        L.gemm_relu_debug_streamk_plan.argtypes = [i64, i64, i64, i32, i32, ctypes.POINTER(i64),
                                                   ctypes.POINTER(i64), ctypes.POINTER(i32)]
        L.gemm_relu_debug_streamk_plan.restype = i32
        L.gemm_relu_debug_set_panel.argtypes = [i32]
        L.gemm_relu_debug_set_panel.restype = i32
        L.gemm_relu_debug_set.argtypes = [i32, i64]
        L.gemm_relu_debug_set.restype = i32
        _lib = L
    return _lib


# ------------------------------------------------------------------ C-ABI names


def gemm_relu_f16(A, B, C, M, N, K, stream=None):
    return lib().gemm_relu_f16(A, B, C, M, N, K, stream)


def gemm_relu_f16_streamk_workspace_bytes(M, N, K):
    return lib().gemm_relu_f16_streamk_workspace_bytes(M, N, K)


def gemm_relu_f16_streamk(A, B, C, M, N, K, workspace, workspace_bytes, stream=None):
    return lib().gemm_relu_f16_streamk(A, B, C, M, N, K, workspace, workspace_bytes, stream)


def gemm_relu_f16_splitk_workspace_bytes(M, N, K, split_k):
    return lib().gemm_relu_f16_splitk_workspace_bytes(M, N, K, split_k)


def gemm_relu_f16_splitk(A, B, C, M, N, K, split_k, workspace, workspace_bytes, stream=None):
    return lib().gemm_relu_f16_splitk(A, B, C, M, N, K, split_k, workspace, workspace_bytes,
                                      stream)


def gemm_relu_f16_splitk_noalloc(A, B, C, M, N, K, split_k, stream=None):
    """Split-K without a caller workspace, for callers that may not allocate
    device memory; uses the library's fixed 8 MiB device scratch array."""
    return lib().gemm_relu_f16_splitk_noalloc(A, B, C, M, N, K, split_k, stream)


def flash_attention_f16(Q, K, V, O, batch, seq, heads, head_dim, causal, stream=None):
    return lib().flash_attention_f16(Q, K, V, O, batch, seq, heads, head_dim, int(causal),
                                     stream)


def gemm_relu_status(stream=None):
    return lib().gemm_relu_status(stream)


def gemm_relu_strerror(code):
    return lib().gemm_relu_strerror(code).decode()


strerror = gemm_relu_strerror


def gemm_relu_f16_path(A, B, C, M, N, K):
    return lib().gemm_relu_f16_path(A, B, C, M, N, K)


def gemm_relu_f16_kernel(A, B, C, M, N, K):
    return lib().gemm_relu_f16_kernel(A, B, C, M, N, K)


def gemm_relu_tile_coord(tile, m_tiles, n_tiles, panel):
    mb, nb = ctypes.c_int64(), ctypes.c_int64()
    rc = lib().gemm_relu_tile_coord(tile, m_tiles, n_tiles, panel, ctypes.byref(mb),
                                    ctypes.byref(nb))
    if rc != 0:
        raise ValueError("tile out of range")
    return mb.value, nb.value


# codes of gemm_relu_debug_force_kernel (not the gemm_relu_f16_kernel codes above)
FORCE_AUTO, FORCE_ONE_CTA_256, FORCE_ONE_CTA_128, FORCE_PAIR, FORCE_GEMV = 0, 1, 2, 3, 4


def gemm_relu_debug_force_kernel(which):
    return lib().gemm_relu_debug_force_kernel(int(which))


SPLIT_AUTO, SPLIT_TWO_STAGE = 0, 1


def gemm_relu_debug_force_split(which):
    return lib().gemm_relu_debug_force_split(int(which))


SK_NORMAL, SK_HEAD_PUBLISHES, SK_TAIL_LATE, SK_HEAD_LATE = 0, 1, 2, 3


def gemm_relu_debug_streamk(mode):
    return lib().gemm_relu_debug_streamk(int(mode))


def gemm_relu_debug_streamk_pieces(pieces):
    return lib().gemm_relu_debug_streamk_pieces(int(pieces))


def streamk_plan(M, N, K, sms, path=PATH_TMA):
    """(dp_tiles, ctas, pair) of gemm_relu_f16_streamk's schedule on a GPU of
    `sms` SMs; dp_tiles -1: no stream-K part.  Host-only."""
    dp, ctas, pair = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
    rc = lib().gemm_relu_debug_streamk_plan(M, N, K, path, sms, ctypes.byref(dp),
                                            ctypes.byref(ctas), ctypes.byref(pair))
    if rc != OK:
        raise ValueError(strerror(rc))
    return dp.value, ctas.value, bool(pair.value)


def gemm_relu_debug_set_panel(rows):
    return lib().gemm_relu_debug_set_panel(int(rows))


def gemm_relu_debug_set(drop_arrive=0, wait_limit_ns=0):
    return lib().gemm_relu_debug_set(int(drop_arrive), int(wait_limit_ns))


# ------------------------------------------------------------------ torch helpers


def _stream_ptr(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check_operands(a, b):
    import torch
    if a.dtype != torch.float16 or b.dtype != torch.float16:
        raise TypeError("A and B must be torch.float16")
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"shapes {tuple(a.shape)} and {tuple(b.shape)} do not multiply")
    if not (a.is_cuda and b.is_cuda and a.device == b.device):
        raise ValueError("A and B must be CUDA tensors on the same device")
    if not (a.is_contiguous() and b.is_contiguous()):
        raise ValueError("A and B must be contiguous row-major")


def _out(a, b, out):
    import torch
    M, N = a.shape[0], b.shape[1]
    if out is None:
        return torch.empty((M, N), dtype=torch.float16, device=a.device)
    if out.shape != (M, N) or out.dtype != torch.float16 or not out.is_contiguous() \
            or out.device != a.device:
        raise ValueError("out must be a contiguous float16 (M, N) tensor on A's device")
    return out


def gemm_relu(a, b, out=None, stream=None):
    """C = relu(a @ b) in fp16 with fp32 accumulation (one fused kernel)."""
    _check_operands(a, b)
    c = _out(a, b, out)
    M, K = a.shape
    N = b.shape[1]
    rc = gemm_relu_f16(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, _stream_ptr(stream))
    if rc != OK:
        raise GemmReluError(rc, "gemm_relu_f16")
    return c


def streamk_workspace(M, N, K, device=None):
    """A device workspace sized for gemm_relu_streamk (uint8 tensor, may be tiny)."""
    import torch
    n = gemm_relu_f16_streamk_workspace_bytes(M, N, K)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def gemm_relu_streamk(a, b, out=None, workspace=None, stream=None):
    """Same result as gemm_relu (up to fp32 summation order in the tiles the
    schedule cuts), with a stream-K schedule for a partial wave and operands
    whose rows TMA cannot describe copied into aligned rows of `workspace`."""
    _check_operands(a, b)
    c = _out(a, b, out)
    M, K = a.shape
    N = b.shape[1]
    if workspace is None:
        workspace = streamk_workspace(M, N, K, a.device)
    rc = gemm_relu_f16_streamk(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                               workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                               _stream_ptr(stream))
    if rc != OK:
        raise GemmReluError(rc, "gemm_relu_f16_streamk")
    return c


def splitk_workspace(M, N, K, split_k, device=None):
    """A device workspace sized for gemm_relu_splitk (uint8 tensor, may be empty)."""
    import torch
    n = gemm_relu_f16_splitk_workspace_bytes(M, N, K, split_k)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def gemm_relu_splitk(a, b, split_k, out=None, workspace=None, stream=None):
    """Same result as gemm_relu, with K split into `split_k` pieces whose fp32
    partials are summed in fixed order (inside a thread-block cluster for a
    split of 2, 4 or 8, else by a second kernel) -- for skinny, memory-bound
    shapes; bit-reproducible."""
    _check_operands(a, b)
    c = _out(a, b, out)
    M, K = a.shape
    N = b.shape[1]
    if workspace is None:
        workspace = splitk_workspace(M, N, K, split_k, a.device)
    rc = gemm_relu_f16_splitk(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, split_k,
                              workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                              _stream_ptr(stream))
    if rc != OK:
        raise GemmReluError(rc, "gemm_relu_f16_splitk")
    return c


def status(stream=None):
    """Synchronise and return (and clear) the device watchdog status."""
    return gemm_relu_status(_stream_ptr(stream))


def flash_attention(q, k, v, causal=False, out=None, stream=None):
    """O = softmax(q k^T / sqrt(d)) v for fp16 CUDA tensors shaped
    [batch, seq, heads, d] (d = 64 or 128), causal or not."""
    import torch
    for t in (q, k, v):
        if t.dtype != torch.float16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q, k, v must be contiguous 4-D float16 CUDA tensors [b, s, h, d]")
    if not (q.shape == k.shape == v.shape):
        raise ValueError("q, k and v must have the same shape")
    if out is None:
        out = torch.empty_like(q)
    b, s, h, d = q.shape
    rc = flash_attention_f16(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), b, s, h, d,
                             causal, _stream_ptr(stream))
    if rc != OK:
        raise GemmReluError(rc, "flash_attention_f16")
    return out

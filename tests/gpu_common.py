"""Shared helpers for the GPU parity tests (device transfer, error metrics)."""
import numpy as np

import tiled_tensor_core_03_gb300 as gr

ATOL = 1e-2
RTOL = 1e-2


def dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t):
    import torch
    torch.cuda.synchronize()
    return t.cpu().numpy()


def run_fused(A, B):
    return host(gr.gemm_relu(dev(A), dev(B)))


def run_split(A, B, split_k, workspace=None):
    a, b = dev(A), dev(B)
    return host(gr.gemm_relu_splitk(a, b, split_k, workspace=workspace))


def abs_dot(A, B, I=None, J=None):
    """sum_k |A[i,k]| |B[k,j]| in fp64 (the scale of the fp32 accumulation error)."""
    A64 = np.abs(A.astype(np.float64))
    B64 = np.abs(B.astype(np.float64))
    if I is None:
        return A64 @ B64
    return np.einsum("tk,kt->t", A64[I], B64[:, J])


def compare(g, o, absab, K):
    """Contract check (|g-o| <= atol + rtol|o|) and the scale-aware bound
    |g-o| <= ulp16(max(|g|,|o|)) + K * 2^-22 * sum_k |a||b|  (fp32 accumulation
    with slack, plus the two fp16 roundings).  Returns a dict of findings."""
    g = np.asarray(g, dtype=np.float16).astype(np.float64)
    o = np.asarray(o, dtype=np.float16).astype(np.float64)
    err = np.abs(g - o)
    contract = err <= ATOL + RTOL * np.abs(o)
    ulp = np.spacing(np.maximum(np.abs(g), np.abs(o)).astype(np.float16)).astype(np.float64)
    strict = err <= ulp + K * 2.0 ** -22 * absab
    rel = err / np.maximum(np.abs(o), 1e-30)
    return {
        "contract_ok": bool(contract.all()),
        "strict_ok": bool(strict.all()),
        "max_abs": float(err.max()) if err.size else 0.0,
        "max_rel": float(rel[o != 0].max()) if (o != 0).any() else 0.0,
        "n_bad_contract": int((~contract).sum()),
        "n_bad_strict": int((~strict).sum()),
        "nonneg": bool((g >= 0).all()),
        "finite": bool(np.isfinite(g).all()),
    }


def assert_parity(g, o, absab, K, what=""):
    r = compare(g, o, absab, K)
    assert r["finite"] and r["nonneg"], (what, r)
    assert r["contract_ok"], (what, r)
    assert r["strict_ok"], (what, r)
    return r


def oracle_threaded(orc, A, B, threads=None):
    """The oracle's full output, its rows split over host threads (the oracle
    library releases the GIL; every row is computed on its own, in the same
    order as a single call would)."""
    import os
    import threading
    M = A.shape[0]
    threads = threads or os.cpu_count() or 1
    out = np.empty((M, B.shape[1]), dtype=np.float16)
    step = (M + threads - 1) // threads

    def work(r0):
        n = min(step, M - r0)
        if n > 0:
            out[r0:r0 + n] = orc.gemm_relu_f16_rows(A, B, r0, n)
    pool = [threading.Thread(target=work, args=(r0,)) for r0 in range(0, M, step)]
    for t in pool:
        t.start()
    for t in pool:
        t.join()
    return out

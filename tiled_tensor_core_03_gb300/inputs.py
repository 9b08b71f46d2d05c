"""Seeded synthetic inputs for the fused GEMM + ReLU workloads.

This module draws random matrices and rounds them to fp16; it holds none of
the GEMM's arithmetic.  Both the CUDA path and the CPU oracle are fed from
here, so they see the same fp16 bits.

Workloads (the pages' example shapes plus the edge and roofline cases):
  square256  M=N=K=256,   A,B ~ N(0,1),            seed 0
  square1024 M=N=K=1024,  A,B ~ N(0,1),            seed 1  (the quickstart shape)
  ragged     1537x1023x777, A,B ~ U[-1,1],         seed 2
  square4096 M=N=K=4096,  A,B ~ N(0,1)/sqrt(K),    seed 3
  skinny     M=16, N=K=8192, A,B ~ N(0,1)/sqrt(K), seed 4, split-K 8

The pages draw fp16 inputs with torch.randn ("TileLang 编程基本知识点", §二) and
ask for a normal distribution rather than zeros (same page, §六 ③).  Here the
draw is numpy default_rng(seed): standard normal (or uniform) in fp32, scaled,
then rounded to fp16 (round-to-nearest-even, numpy's astype).  A is drawn
first, then B, from the same generator.
"""
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dist: str          # "normal" | "uniform"
    scale_by_sqrt_k: bool
    seed: int
    split_k: int = 1

    @property
    def flops(self):
        return 2 * self.M * self.N * self.K

    @property
    def bytes(self):
        """Algorithmic HBM bytes: A and B read once, C written once (fp16)."""
        return 2 * (self.M * self.K + self.K * self.N + self.M * self.N)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("square256", 256, 256, 256, "normal", False, 0),
        Workload("square1024", 1024, 1024, 1024, "normal", False, 1),
        Workload("ragged", 1537, 1023, 777, "uniform", False, 2),
        Workload("square4096", 4096, 4096, 4096, "normal", True, 3),
        Workload("skinny", 16, 8192, 8192, "normal", True, 4, split_k=8),
        # the skinny shape taken to one row (a decode step): the GEMV path
        Workload("decode1", 1, 8192, 8192, "normal", True, 5),
    ]
}


def draw(shape, dist, scale, rng):
    if dist == "normal":
        x = rng.standard_normal(shape, dtype=np.float32)
    elif dist == "uniform":
        x = rng.uniform(-1.0, 1.0, size=shape).astype(np.float32)
    elif dist == "int4":
        x = rng.integers(-4, 5, size=shape).astype(np.float32)
    else:
        raise ValueError(dist)
    if scale != 1.0:
        x *= np.float32(scale)
    return x.astype(np.float16)


def make(M, N, K, dist="normal", scale_by_sqrt_k=False, seed=0):
    """Return (A, B) as C-contiguous fp16 numpy arrays of shapes (M,K), (K,N)."""
    rng = np.random.default_rng(seed)
    scale = 1.0 / np.sqrt(K) if (scale_by_sqrt_k and K > 0) else 1.0
    A = draw((M, K), dist, scale, rng)
    B = draw((K, N), dist, scale, rng)
    return np.ascontiguousarray(A), np.ascontiguousarray(B)


def make_workload(w):
    if isinstance(w, str):
        w = WORKLOADS[w]
    return make(w.M, w.N, w.K, w.dist, w.scale_by_sqrt_k, w.seed)

"""Seeded synthetic operands for the fp16 NT GEMM.

This module draws inputs only; it holds none of the product's arithmetic.
Both the CUDA path and the CPU oracle receive what it returns, so it is the
one piece the two sides share.

Recipe for every workload: ``numpy.random.Generator(PCG64(seed))`` draws A
[M,K] then B [N,K] in row-major order as float64, and ``astype(float16)``
rounds them (round to nearest even).  The value families are

  eighths   integers in [-8, 8] divided by 8 (exact in fp16)
  normal    standard normal divided by sqrt(K)
  uniform   uniform on [-1, 1)

The page "wgmma_gemm.cu" draws {-8..8}/8 operands from a 32-bit LCG
(multiplier 1664525, increment 1013904223, seed 20260901, value
((state >> 24) mod 17 - 8) / 8, A first then B); ``lcg_eighths`` reproduces
that stream for a 256^3 cross-check.
"""
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dist: str
    seed: int
    note: str = ""

    @property
    def flops(self):
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self):
        """A and B read once, C written once (fp16)."""
        return 2 * (self.M * self.K + self.N * self.K + self.M * self.N)


# The five workloads of this GEMM, smallest first.
WORKLOADS = [
    Workload("square_256", 256, 256, 256, "eighths", 1001, "exact integer-valued case"),
    Workload("square_4096", 4096, 4096, 4096, "normal", 1002, "N(0,1)/sqrt(K)"),
    Workload("square_8192", 8192, 8192, 8192, "uniform", 1003, "compute-bound headline case"),
    Workload("ragged_3000x5000x4096", 3000, 5000, 4096, "eighths", 1004, "ragged M and N edges"),
    Workload("skinny_128x16384x16384", 128, 16384, 16384, "normal", 1005, "bandwidth-leaning"),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def _draw(rng, dist, shape, K):
    if dist == "eighths":
        return rng.integers(-8, 9, size=shape).astype(np.float64) / 8.0
    if dist == "normal":
        return rng.standard_normal(size=shape) / np.sqrt(float(K))
    if dist == "uniform":
        return rng.uniform(-1.0, 1.0, size=shape)
    raise ValueError("unknown distribution %r" % dist)


def make_operands(M, N, K, dist, seed):
    """A [M,K] and B [N,K] as C-contiguous float16 numpy arrays."""
    rng = np.random.Generator(np.random.PCG64(seed))
    A = _draw(rng, dist, (M, K), K).astype(np.float16)
    B = _draw(rng, dist, (N, K), K).astype(np.float16)
    return A, B


def workload_operands(w):
    return make_operands(w.M, w.N, w.K, w.dist, w.seed)


def lcg_eighths(M, N, K, seed=20260901):
    """{-8..8}/8 operands from the day78 page's 32-bit LCG, A then B."""
    total = M * K + N * K
    out = np.empty(total, dtype=np.float16)
    state = seed & 0xFFFFFFFF
    for i in range(total):
        state = (state * 1664525 + 1013904223) & 0xFFFFFFFF
        out[i] = ((state >> 24) % 17 - 8) / 8.0
    return out[: M * K].reshape(M, K), out[M * K:].reshape(N, K)


# ---- structured operands with known products (used by parity pins) ----

def identity(n):
    return np.eye(n, dtype=np.float16)


def permutation(n, seed):
    """A permutation matrix P (fp16) and its permutation p: P[i, p[i]] = 1."""
    p = np.random.Generator(np.random.PCG64(seed)).permutation(n)
    P = np.zeros((n, n), dtype=np.float16)
    P[np.arange(n), p] = 1.0
    return P, p


def rank1(M, N, K, seed):
    """a_ik = u_i v_k, b_jk = w_j v_k with dyadic u, v, w (all exact in fp16).

    Returns A, B and the factors (u, w, v) as float64.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    u = rng.choice(np.array([-2.0, -1.0, -0.5, 0.5, 1.0, 2.0]), size=M)
    w = rng.choice(np.array([-2.0, -1.0, -0.5, 0.5, 1.0, 2.0]), size=N)
    v = rng.integers(-8, 9, size=K).astype(np.float64) / 8.0
    A = np.outer(u, v).astype(np.float16)
    B = np.outer(w, v).astype(np.float16)
    return A, B, (u, w, v)

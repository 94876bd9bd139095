"""GB300 (sm_103a) dense fp16 GEMM, C[M,N] = A[M,K] . B[N,K]^T.

The compute path is the C-ABI library built from ``csrc/`` (declared in
``include/gemm_f16.h``); ``gemm`` is a thin ctypes binding over it with the
same entry-point names.  ``inputs`` draws the seeded synthetic operands.
Importing this package loads nothing; the library is loaded on first use and
a missing library is an error, never a fallback.
"""
__all__ = ["inputs", "gemm"]

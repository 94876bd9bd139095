"""CPU oracle for C[M,N] = A[M,K] . B[N,K]^T (fp16 in, fp16 out).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
baseline leg of bench.py may import this package.  The product path (the
CUDA library and its Python binding) never imports, loads or calls it.

Arithmetic lives in gemm_oracle.c (natural-order double dot products, one
binary16 round-to-nearest-even rounding; see its header for the passages it
follows).  This module only marshals numpy arrays into that library and
states the acceptance bound of the parity tests (tolerance.py).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def load_library(path):
    """ctypes handle of an oracle library with its signatures declared."""
    L = ctypes.CDLL(path)
    _declare(L)
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = load_library(_build.build())
    return _lib


def _declare(L):
    i64, u16p, f64p, i64p = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    L.oracle_f16_to_f64.restype = ctypes.c_double
    L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    L.oracle_f64_to_f16.restype = ctypes.c_uint16
    L.oracle_f64_to_f16.argtypes = [ctypes.c_double]
    L.oracle_f16_to_f64_array.argtypes = [i64, u16p, f64p]
    L.oracle_f64_to_f16_array.argtypes = [i64, f64p, u16p]
    L.oracle_gemm_nt.restype = ctypes.c_int
    L.oracle_gemm_nt.argtypes = [i64, i64, i64, u16p, u16p, u16p, f64p, f64p]
    L.oracle_gemm_nt_entries.restype = ctypes.c_int
    L.oracle_gemm_nt_entries.argtypes = [i64, i64, i64, u16p, u16p, i64, i64p, i64p, u16p, f64p, f64p]
    L.oracle_gemm_nn_f32.restype = ctypes.c_int
    L.oracle_gemm_nn_f32.argtypes = [i64, i64, i64, u16p, u16p, ctypes.c_void_p, f64p, f64p]
    L.oracle_gemm_nn_f32_entries.restype = ctypes.c_int
    L.oracle_gemm_nn_f32_entries.argtypes = [i64, i64, i64, u16p, u16p, i64, i64p, i64p, ctypes.c_void_p,
                                             f64p, f64p]
    L.oracle_f64_to_f32_array.argtypes = [i64, f64p, ctypes.c_void_p]
    L.oracle_num_threads.restype = ctypes.c_int


def _bits(x):
    """View an fp16 (or uint16) array as contiguous uint16 bits."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16)
    if x.dtype == np.uint16:
        return x
    raise TypeError("expected float16 or uint16 array, got %s" % x.dtype)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def f16_to_f64(bits):
    bits = _bits(np.asarray(bits))
    out = np.empty(bits.shape, dtype=np.float64)
    lib().oracle_f16_to_f64_array(bits.size, _ptr(bits), _ptr(out))
    return out


def f64_to_f16(values):
    values = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(values.shape, dtype=np.uint16)
    lib().oracle_f64_to_f16_array(values.size, _ptr(values), _ptr(out))
    return out


def gemm_nt(A, B, want_exact=False):
    """Full product.  A [M,K], B [N,K] fp16 (or uint16 bits).

    Returns (C_bits uint16 [M,N], absum float64 [M,N]) and, if want_exact,
    also the unrounded double sums.
    """
    a, b = _bits(A), _bits(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError("A must be [M,K] and B [N,K]")
    M, K = a.shape
    N = b.shape[0]
    c = np.empty((M, N), dtype=np.uint16)
    absum = np.empty((M, N), dtype=np.float64)
    exact = np.empty((M, N), dtype=np.float64) if want_exact else None
    rc = lib().oracle_gemm_nt(M, N, K, _ptr(a), _ptr(b), _ptr(c), _ptr(absum),
                              _ptr(exact) if want_exact else None)
    if rc != 0:
        raise MemoryError("oracle_gemm_nt failed (%d)" % rc)
    return (c, absum, exact) if want_exact else (c, absum)


def gemm_nt_entries(A, B, rows, cols, want_exact=False):
    """Only the entries (rows[e], cols[e]) of A . B^T."""
    a, b = _bits(A), _bits(B)
    M, K = a.shape
    N = b.shape[0]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols differ in shape")
    c = np.empty(rows.shape, dtype=np.uint16)
    absum = np.empty(rows.shape, dtype=np.float64)
    exact = np.empty(rows.shape, dtype=np.float64) if want_exact else None
    rc = lib().oracle_gemm_nt_entries(M, N, K, _ptr(a), _ptr(b), rows.size, _ptr(rows), _ptr(cols),
                                      _ptr(c), _ptr(absum), _ptr(exact) if want_exact else None)
    if rc != 0:
        raise ValueError("oracle_gemm_nt_entries failed (%d)" % rc)
    return (c, absum, exact) if want_exact else (c, absum)


def gemm_nn_f32(A, B_kn, want_exact=False):
    """D = A . B with A [M,K] and B [K,N] fp16 (or uint16 bits), fp32 result.

    Returns (D float32 [M,N], absum float64 [M,N]) and, if want_exact, the
    unrounded double sums.
    """
    a, b = _bits(A), _bits(B_kn)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[0]:
        raise ValueError("A must be [M,K] and B [K,N]")
    M, K = a.shape
    N = b.shape[1]
    d = np.empty((M, N), dtype=np.float32)
    absum = np.empty((M, N), dtype=np.float64)
    exact = np.empty((M, N), dtype=np.float64) if want_exact else None
    rc = lib().oracle_gemm_nn_f32(M, N, K, _ptr(a), _ptr(b), _ptr(d), _ptr(absum),
                                  _ptr(exact) if want_exact else None)
    if rc != 0:
        raise MemoryError("oracle_gemm_nn_f32 failed (%d)" % rc)
    return (d, absum, exact) if want_exact else (d, absum)


def gemm_nn_f32_entries(A, B_kn, rows, cols):
    a, b = _bits(A), _bits(B_kn)
    M, K = a.shape
    N = b.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    d = np.empty(rows.shape, dtype=np.float32)
    absum = np.empty(rows.shape, dtype=np.float64)
    rc = lib().oracle_gemm_nn_f32_entries(M, N, K, _ptr(a), _ptr(b), rows.size, _ptr(rows), _ptr(cols), _ptr(d),
                                          _ptr(absum), None)
    if rc != 0:
        raise ValueError("oracle_gemm_nn_f32_entries failed (%d)" % rc)
    return d, absum


def f64_to_f32(values):
    values = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(values.shape, dtype=np.float32)
    lib().oracle_f64_to_f32_array(values.size, _ptr(values), _ptr(out))
    return out


def num_threads():
    return int(lib().oracle_num_threads())


from .tolerance import check_parity, check_parity_f32, ulp16, ulp32  # noqa: E402,F401

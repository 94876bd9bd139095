"""Acceptance bound of the parity tests (test infrastructure only).

Every element must satisfy

    |c_gpu - c_ref| <= 1e-3 * sum_k |a_ik * b_jk| + ulp16(c_ref)

where c_ref is the oracle's binary16 result, the sum of absolute products
comes from the oracle in double, and ulp16(x) is the binary16 spacing at
|x|: 2^(e-10) for a normal |x| in [2^e, 2^(e+1)), 2^-24 below 2^-14.

Why this bound: the tensor cores accumulate in fp32 in an unspecified order
("wgmma_gemm.cu", the tolerance comment next to kRelTolerance, and the
fp32 accumulator of "1. WGMMA", section "The Full Kernel").  An fp32 sum of
K products in any order is off from the exact sum by at most about
K * 2^-24 * sum|a*b|, far inside 1e-3 * sum|a*b| for the sizes used, and
the final cast can land one binary16 step away from the oracle's single
rounding of the double sum.  An Inf or NaN from the GPU always fails.
"""
import numpy as np


def ulp16(ref_values):
    """binary16 spacing at |x| for finite double values x."""
    x = np.abs(np.asarray(ref_values, dtype=np.float64))
    _, e2 = np.frexp(x)          # x = m * 2^e2, m in [0.5, 1)
    e = e2.astype(np.int64) - 1  # floor(log2 x) for x > 0
    spacing = np.ldexp(1.0, (np.maximum(e, -14) - 10).astype(np.int64))
    spacing = np.where(x < 2.0 ** -14, 2.0 ** -24, spacing)
    return spacing


class ParityReport:
    def __init__(self, ok, failures, first, worst_ratio, max_abs_err, n):
        self.ok = ok
        self.failures = failures
        self.first = first
        self.worst_ratio = worst_ratio
        self.max_abs_err = max_abs_err
        self.n = n

    def __repr__(self):
        return ("ParityReport(ok=%s, failures=%d/%d, first=%s, worst_ratio=%.3g, max_abs_err=%.3g)"
                % (self.ok, self.failures, self.n, self.first, self.worst_ratio, self.max_abs_err))


def check_parity(c_gpu_bits, c_ref_bits, absum, rel=1e-3, index_shape=None):
    """Compare GPU binary16 output bits with the oracle's, element by element.

    Returns a ParityReport naming the first failing index, the worst ratio
    |err| / bound, the largest absolute error and the failure count.
    """
    from . import f16_to_f64
    g = f16_to_f64(np.asarray(c_gpu_bits)).ravel()
    r = f16_to_f64(np.asarray(c_ref_bits)).ravel()
    s = np.asarray(absum, dtype=np.float64).ravel()
    if not (g.size == r.size == s.size):
        raise ValueError("shape mismatch")
    finite_ref = np.isfinite(r)
    bound = rel * s + np.where(finite_ref, ulp16(np.where(finite_ref, r, 0.0)), 0.0)
    err = np.abs(g - r)
    ok_elem = np.isfinite(g) & finite_ref & (err <= bound)
    # an infinite reference (unreachable on the configured inputs) must be met exactly
    ok_elem |= (~finite_ref) & (g == r)
    bad = np.flatnonzero(~ok_elem)
    first = None
    if bad.size:
        idx = int(bad[0])
        pos = np.unravel_index(idx, index_shape) if index_shape is not None else idx
        first = (pos, float(g[idx]), float(r[idx]), float(bound[idx]))
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, np.where(err > 0, np.inf, 0.0))
    ratio = np.where(np.isfinite(g), ratio, np.inf)
    worst = float(ratio.max()) if ratio.size else 0.0
    fin = np.isfinite(g) & finite_ref
    max_abs = float(err[fin].max()) if fin.any() else 0.0
    return ParityReport(bad.size == 0, int(bad.size), first, worst, max_abs, g.size)


def ulp32(ref_values):
    """binary32 spacing at |x| for finite double values x: 2^(e-23) for a
    normal |x| in [2^e, 2^(e+1)), 2^-149 below 2^-126."""
    x = np.abs(np.asarray(ref_values, dtype=np.float64))
    _, e2 = np.frexp(x)
    e = e2.astype(np.int64) - 1
    spacing = np.ldexp(1.0, (np.maximum(e, -126) - 23).astype(np.int64))
    return np.where(x < 2.0 ** -126, 2.0 ** -149, spacing)


def check_parity_f32(d_gpu, d_ref, absum, rel=1e-3, index_shape=None):
    """The fp32-output form of the bound: |d_gpu - d_ref| <= 1e-3 * sum|a*b|
    + ulp32(d_ref) for every element; Inf/NaN from the GPU fails."""
    g = np.asarray(d_gpu, dtype=np.float32).astype(np.float64).ravel()
    r = np.asarray(d_ref, dtype=np.float32).astype(np.float64).ravel()
    s = np.asarray(absum, dtype=np.float64).ravel()
    bound = rel * s + ulp32(r)
    err = np.abs(g - r)
    ok_elem = np.isfinite(g) & (err <= bound)
    bad = np.flatnonzero(~ok_elem)
    first = None
    if bad.size:
        idx = int(bad[0])
        pos = np.unravel_index(idx, index_shape) if index_shape is not None else idx
        first = (pos, float(g[idx]), float(r[idx]), float(bound[idx]))
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, np.where(err > 0, np.inf, 0.0))
    ratio = np.where(np.isfinite(g), ratio, np.inf)
    fin = np.isfinite(g)
    return ParityReport(bad.size == 0, int(bad.size), first, float(ratio.max()) if ratio.size else 0.0,
                        float(err[fin].max()) if fin.any() else 0.0, g.size)

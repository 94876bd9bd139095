"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test fixes part of the oracle to something independent of it: the
IEEE 754 binary16 definition (hand-written golden cases and an independent
conversion routine), exact rational arithmetic, closed forms (identity,
permutation and rank-1 operands) and exact integer products.  Together they
catch a dropped or repeated term, a wrong sign, a transposed operand, a
wrong index stride and a wrong rounding rule.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from dense_fp16_gemm_03_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16)


# --------------------------------------------------------------------------
# binary16 conversions

def test_f16_to_f64_exhaustive_against_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # the sign of zero survives
    assert np.signbit(ours[0x8000]) and not np.signbit(ours[0])


def test_f64_to_f16_round_trip_every_finite_value():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(vals)
    back = oracle.f64_to_f16(vals[finite])
    assert np.array_equal(back, bits[finite])
    assert oracle.f64_to_f16(np.array([np.inf]))[0] == 0x7C00
    assert oracle.f64_to_f16(np.array([-np.inf]))[0] == 0xFC00
    nan_bits = oracle.f64_to_f16(np.array([np.nan]))[0]
    assert (nan_bits & 0x7C00) == 0x7C00 and (nan_bits & 0x3FF) != 0


def test_f64_to_f16_golden_cases():
    path = os.path.join(GOLDEN, "f16_rounding_cases.txt")
    n = 0
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        hex_value, expected = line.split()[:2]
        x = float.fromhex(hex_value)
        got = int(oracle.f64_to_f16(np.array([x]))[0])
        assert got == int(expected, 16), (hex_value, hex(got), expected)
        n += 1
    assert n >= 20


def test_f64_to_f16_midpoints_ties_to_even():
    """Every midpoint between neighbouring finite binary16 values rounds to
    the neighbour whose last fraction bit is 0; a hair either side of the
    midpoint rounds to the nearer neighbour."""
    pos = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)   # +0 .. 65504
    lo = pos[:-1]
    hi = pos[1:]
    lo_v = lo.view(np.float16).astype(np.float64)
    hi_v = hi.view(np.float16).astype(np.float64)
    mid = (lo_v + hi_v) / 2.0                                       # exact in double
    even = np.where((lo & 1) == 0, lo, hi)
    for sign in (1.0, -1.0):
        sbit = np.uint16(0x8000) if sign < 0 else np.uint16(0)
        got = oracle.f64_to_f16(sign * mid)
        assert np.array_equal(got, even | sbit)
        below = oracle.f64_to_f16(sign * np.nextafter(mid, 0.0))
        above = oracle.f64_to_f16(sign * np.nextafter(mid, np.inf))
        assert np.array_equal(below, lo | sbit)
        assert np.array_equal(above, hi | sbit)


def test_f64_to_f16_random_against_numpy():
    rng = np.random.Generator(np.random.PCG64(7))
    mant = rng.uniform(1.0, 2.0, size=400_000)
    expo = rng.integers(-30, 18, size=400_000)
    sign = rng.choice([-1.0, 1.0], size=400_000)
    x = sign * np.ldexp(mant, expo)
    ours = oracle.f64_to_f16(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


# --------------------------------------------------------------------------
# the product

def _parse_matrix(text):
    return np.array([[float(v) for v in row.split(",")] for row in text.split(";")])


def test_hand_worked_cases():
    path = os.path.join(GOLDEN, "tiny_gemm_cases.txt")
    cases, cur = [], None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "case":
            cur = {}
            cases.append(cur)
        else:
            cur[key] = _parse_matrix(rest)
    assert len(cases) == 3
    for c in cases:
        A = c["A"].astype(np.float16)
        B = c["B"].astype(np.float16)
        C, absum = oracle.gemm_nt(A, B)
        assert np.array_equal(oracle.f16_to_f64(C), c["C"])


def _random_moderate_f16(rng, shape):
    """fp16 values with random 11-bit significands and exponents in [-4, 4):
    products and sums of up to 17 of them are exact in double."""
    mant = rng.integers(1024, 2048, size=shape).astype(np.float64)
    expo = rng.integers(-4, 4, size=shape)
    sign = rng.choice([-1.0, 1.0], size=shape)
    return (sign * np.ldexp(mant, expo - 10)).astype(np.float16)


@pytest.mark.parametrize("seed", range(40))
def test_brute_force_exact_rationals(seed):
    rng = np.random.Generator(np.random.PCG64(100 + seed))
    M, N, K = (int(v) for v in rng.integers(1, 18, size=3))
    A = _random_moderate_f16(rng, (M, K))
    B = _random_moderate_f16(rng, (N, K))
    if seed % 5 == 0:                      # sprinkle exact zeros
        A[rng.random((M, K)) < 0.3] = 0
    C, absum, exact = oracle.gemm_nt(A, B, want_exact=True)
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            sa = Fraction(0)
            for k in range(K):
                p = Fraction(float(A[i, k])) * Fraction(float(B[j, k]))
                s += p
                sa += abs(p)
            assert Fraction(exact[i, j]) == s
            assert Fraction(absum[i, j]) == sa
            expect = np.float64(float(s)).astype(np.float16).view(np.uint16)
            assert C[i, j] == expect, (i, j, float(s))


def test_entries_match_full_product():
    rng = np.random.Generator(np.random.PCG64(3))
    A = (rng.standard_normal((37, 70)) / 8).astype(np.float16)
    B = (rng.standard_normal((29, 70)) / 8).astype(np.float16)
    C, absum = oracle.gemm_nt(A, B)
    rows = rng.integers(0, 37, size=200)
    cols = rng.integers(0, 29, size=200)
    Ce, ae = oracle.gemm_nt_entries(A, B, rows, cols)
    assert np.array_equal(Ce, C[rows, cols])
    assert np.array_equal(ae, absum[rows, cols])
    with pytest.raises(ValueError):
        oracle.gemm_nt_entries(A, B, np.array([37]), np.array([0]))


def test_identity_operands():
    rng = np.random.Generator(np.random.PCG64(11))
    K = 48
    B = (rng.standard_normal((33, K))).astype(np.float16)
    C, _ = oracle.gemm_nt(inputs.identity(K), B)          # A = I: C = B^T
    assert np.array_equal(oracle.f16_to_f64(C), B.T.astype(np.float64))
    A = (rng.standard_normal((21, K))).astype(np.float16)
    C, _ = oracle.gemm_nt(A, inputs.identity(K))          # B = I: C = A
    assert np.array_equal(oracle.f16_to_f64(C), A.astype(np.float64))


def test_permutation_operands():
    rng = np.random.Generator(np.random.PCG64(12))
    K = 40
    P, p = inputs.permutation(K, seed=5)
    B = (rng.standard_normal((19, K))).astype(np.float16)
    C, _ = oracle.gemm_nt(P, B)            # C[i, j] = B[j, p[i]]
    assert np.array_equal(oracle.f16_to_f64(C), B[:, p].T.astype(np.float64))
    C2, _ = oracle.gemm_nt(B, P)           # C[i, j] = B[i, p[j]]
    assert np.array_equal(oracle.f16_to_f64(C2), B[:, p].astype(np.float64))


@pytest.mark.parametrize("shape", [(5, 7, 9), (16, 24, 64), (33, 17, 300)])
def test_rank1_closed_form(shape):
    M, N, K = shape
    A, B, (u, w, v) = inputs.rank1(M, N, K, seed=M + N + K)
    C, absum = oracle.gemm_nt(A, B)
    S = float(np.sum(v * v))                       # exact: multiples of 1/64
    expect = np.outer(u, w) * S                    # exact dyadic doubles
    assert np.array_equal(C, expect.astype(np.float16).view(np.uint16))
    assert np.array_equal(absum, np.abs(np.outer(u, w)) * S)


@pytest.mark.parametrize("shape", [(37, 53, 200), (64, 64, 256), (9, 130, 1000)])
def test_integer_operands_exact(shape):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "eighths", seed=M * N)
    Ai = (A.astype(np.float64) * 8).astype(np.int64)
    Bi = (B.astype(np.float64) * 8).astype(np.int64)
    exact_int = Ai @ Bi.T                          # exact, in units of 1/64
    C, absum = oracle.gemm_nt(A, B)
    expect = (exact_int.astype(np.float64) / 64.0).astype(np.float16).view(np.uint16)
    assert np.array_equal(C, expect)
    assert np.array_equal(absum, (np.abs(Ai) @ np.abs(Bi).T).astype(np.float64) / 64.0)


def test_lcg_stream_matches_page_recipe():
    """The day78 page's LCG: first values computed by hand from its recurrence."""
    A, B = inputs.lcg_eighths(2, 2, 2)
    state = 20260901
    vals = []
    for _ in range(8):
        state = (state * 1664525 + 1013904223) % 2 ** 32
        vals.append(((state >> 24) % 17 - 8) / 8)
    assert list(A.ravel().astype(float)) == vals[:4]
    assert list(B.ravel().astype(float)) == vals[4:]


# --------------------------------------------------------------------------
# the acceptance bound

def test_ulp16_values():
    assert oracle.ulp16(np.array([1.0]))[0] == 2.0 ** -10
    assert oracle.ulp16(np.array([0.99]))[0] == 2.0 ** -11
    assert oracle.ulp16(np.array([-65504.0]))[0] == 32.0
    assert oracle.ulp16(np.array([0.0]))[0] == 2.0 ** -24
    assert oracle.ulp16(np.array([2.0 ** -14]))[0] == 2.0 ** -24
    assert oracle.ulp16(np.array([2.0 ** -15]))[0] == 2.0 ** -24
    assert oracle.ulp16(np.array([3.0]))[0] == 2.0 ** -9


def test_check_parity_bounds():
    ref = np.array([1.0, 2.0, -0.5, 0.0], dtype=np.float16).view(np.uint16)
    absum = np.zeros(4)
    # exactly one ulp away everywhere passes with a zero absum
    one_ulp = np.array([1.0 + 2 ** -10, 2.0 - 2 ** -10, -0.5 - 2 ** -11, 2 ** -24]).astype(np.float16)
    assert oracle.check_parity(one_ulp.view(np.uint16), ref, absum).ok
    two_ulp = np.array([1.0 + 2 ** -9, 2.0, -0.5, 0.0]).astype(np.float16)
    rep = oracle.check_parity(two_ulp.view(np.uint16), ref, absum)
    assert not rep.ok and rep.failures == 1 and rep.first[0] == 0
    # the absum term widens the bound
    assert oracle.check_parity(two_ulp.view(np.uint16), ref, np.array([2.0, 0, 0, 0])).ok
    for bad in (np.inf, np.nan):
        g = np.array([bad, 2.0, -0.5, 0.0]).astype(np.float16).view(np.uint16)
        assert not oracle.check_parity(g, ref, np.full(4, 1e9)).ok


# --------------------------------------------------------------------------
# the fp32-output product with B stored [K, N] ("wgmma_gemm.cu" layout)

def test_f64_to_f32_golden_cases():
    path = os.path.join(GOLDEN, "f32_rounding_cases.txt")
    n = 0
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        src, expect = line.split()[:2]
        got = float(oracle.f64_to_f32(np.array([float.fromhex(src)]))[0])
        assert got == float.fromhex(expect), (src, got.hex(), expect)
        n += 1
    assert n >= 10


@pytest.mark.parametrize("shape", [(37, 53, 200), (64, 64, 256), (9, 130, 1000)])
def test_nn_f32_integer_operands_exact(shape):
    M, N, K = shape
    A, Bnk = inputs.make_operands(M, N, K, "eighths", seed=M + 3 * N)
    B = np.ascontiguousarray(Bnk.T)                 # [K, N]
    Ai = (A.astype(np.float64) * 8).astype(np.int64)
    Bi = (B.astype(np.float64) * 8).astype(np.int64)
    D, absum = oracle.gemm_nn_f32(A, B)
    assert D.dtype == np.float32
    assert np.array_equal(D, ((Ai @ Bi).astype(np.float64) / 64.0).astype(np.float32))
    assert np.array_equal(absum, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64) / 64.0)


@pytest.mark.parametrize("seed", range(12))
def test_nn_f32_brute_force_exact_rationals(seed):
    rng = np.random.Generator(np.random.PCG64(500 + seed))
    M, N, K = (int(v) for v in rng.integers(1, 14, size=3))
    A = _random_moderate_f16(rng, (M, K))
    B = _random_moderate_f16(rng, (K, N))
    D, absum, exact = oracle.gemm_nn_f32(A, B, want_exact=True)
    for i in range(M):
        for j in range(N):
            s = sum(Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(K))
            assert Fraction(exact[i, j]) == s
            assert D[i, j] == np.float32(float(s))


def test_nn_f32_agrees_with_nt_sums():
    """D = A . B and C = A . (B^T)^T are the same sums: the unrounded double
    results of the two oracle entries coincide, and the fp16 result is the
    fp16 rounding of the same value."""
    rng = np.random.Generator(np.random.PCG64(9))
    A = (rng.standard_normal((31, 96)) / 4).astype(np.float16)
    Bkn = (rng.standard_normal((96, 45)) / 4).astype(np.float16)
    D, absum_nn, exact_nn = oracle.gemm_nn_f32(A, Bkn, want_exact=True)
    C, absum_nt, exact_nt = oracle.gemm_nt(A, np.ascontiguousarray(Bkn.T), want_exact=True)
    assert np.array_equal(exact_nn, exact_nt) and np.array_equal(absum_nn, absum_nt)
    assert np.array_equal(oracle.f64_to_f16(exact_nn), C)
    assert np.array_equal(D, exact_nn.astype(np.float32))


def test_nn_f32_identity_and_entries():
    rng = np.random.Generator(np.random.PCG64(10))
    A = rng.standard_normal((20, 48)).astype(np.float16)
    D, _ = oracle.gemm_nn_f32(A, inputs.identity(48))          # B = I: D = A exactly
    assert np.array_equal(D, A.astype(np.float32))
    B = rng.standard_normal((48, 33)).astype(np.float16)
    D, _ = oracle.gemm_nn_f32(inputs.identity(48), B)          # A = I: D = B exactly
    assert np.array_equal(D, B.astype(np.float32))
    D, absum = oracle.gemm_nn_f32(A, B)
    rows, cols = rng.integers(0, 20, size=50), rng.integers(0, 33, size=50)
    De, ae = oracle.gemm_nn_f32_entries(A, B, rows, cols)
    assert np.array_equal(De, D[rows, cols]) and np.array_equal(ae, absum[rows, cols])


def test_check_parity_f32_bounds():
    ref = np.array([1.0, -2.0, 0.0], dtype=np.float32)
    ok = np.array([1.0 + 2 ** -23, -2.0 + 2 ** -22, 2 ** -149], dtype=np.float32)
    assert oracle.check_parity_f32(ok, ref, np.zeros(3)).ok
    bad = np.array([1.0 + 2 ** -21, -2.0, 0.0], dtype=np.float32)
    rep = oracle.check_parity_f32(bad, ref, np.zeros(3))
    assert not rep.ok and rep.first[0] == 0
    assert oracle.check_parity_f32(bad, ref, np.array([0.01, 0, 0])).ok
    assert oracle.ulp32(np.array([1.0]))[0] == 2.0 ** -23

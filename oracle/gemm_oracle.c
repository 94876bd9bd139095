/*
 * CPU oracle for the dense fp16 GEMM  C[M,N] = A[M,K] . B[N,K]^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; it exists so that tests, the smoke check and the CPU
 * baseline leg of the benchmark have an independent, obviously correct
 * statement of what the GPU path must compute.  It shares no code, header,
 * table or constant with the CUDA library.
 *
 * What it follows:
 *  - "1. WGMMA: Hopper's Asynchronous Tensor Core" (tilus tutorial),
 *    section "The Full Kernel": A is viewed as [m, k] and B as [n, k], both
 *    fp16; the product is taken against B transposed, accumulated in fp32
 *    and cast to fp16 before the store to C [m, n].
 *  - "wgmma_gemm.cu" (day78 page), function gemmCpu: the reference product
 *    is a plain triple loop that accumulates each dot product in double.
 *
 * Definition implemented here (no blocking, no reordering):
 *     C[i][j] = fp16_rne( sum_{k=0}^{K-1} double(A[i][k]) * double(B[j][k]) )
 * with the sum taken in double in natural k order and a single rounding
 * from double to binary16, round-to-nearest-even, subnormals included,
 * overflow to +-inf.  Alongside it the oracle returns
 *     absum[i][j] = sum_k |double(A[i][k]) * double(B[j][k])|
 * which scales the acceptance bound of the parity tests.
 *
 * The binary16 <-> double conversions are written here from the IEEE 754
 * binary16 interchange format (1 sign bit, 5 exponent bits with bias 15,
 * 10 fraction bits) and its round-to-nearest-ties-to-even rule.
 *
 * A second entry computes the layout of "wgmma_gemm.cu" (B as [K, N],
 * fp32 result); see oracle_gemm_nn_f32.
 *
 * Parity pins (checked by tests marked "not gpu"): exhaustive conversion
 * checks against an independent library, brute force with exact rational
 * arithmetic, identity and permutation operands, rank-1 closed forms,
 * integer-valued operands against an exact int64 product.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (see build.py).
 * -ffp-contract=off keeps every product and sum a separately rounded
 * double operation, as the definition states.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* binary16 -> double (exact: every binary16 value is a double value). */
double oracle_f16_to_f64(uint16_t h)
{
    int negative = (h >> 15) & 1;
    int biased_exp = (h >> 10) & 0x1f;
    int fraction = h & 0x3ff;
    double magnitude;
    if (biased_exp == 0) {
        /* zero or subnormal: fraction * 2^(1-15) * 2^-10 = fraction * 2^-24 */
        magnitude = ldexp((double)fraction, -24);
    } else if (biased_exp == 31) {
        magnitude = fraction ? NAN : INFINITY;
    } else {
        /* normal: (1 + fraction/2^10) * 2^(biased_exp-15) */
        magnitude = ldexp((double)(1024 + fraction), biased_exp - 15 - 10);
    }
    return negative ? -magnitude : magnitude;
}

/* ------------------------------------------------------------------ */
/* double -> binary16, one rounding, round to nearest, ties to even.   */
uint16_t oracle_f64_to_f16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7c00u);
    if (a == 0.0) return sign;

    /* a = frac * 2^e2 with frac in [0.5, 1): floor(log2(a)) = e2 - 1 */
    int e2;
    (void)frexp(a, &e2);
    int unbiased = e2 - 1;
    /* Grid spacing of binary16 at a: 2^(E-10) in the normal range,
       2^-24 below the smallest normal 2^-14. */
    int spacing_exp = (unbiased < -14) ? -24 : unbiased - 10;
    if (unbiased > 15) return (uint16_t)(sign | 0x7c00u); /* >= 2^16 */

    double scaled = ldexp(a, -spacing_exp);   /* exact: power-of-two scale */
    double whole = floor(scaled);             /* scaled < 2^11: exact      */
    double rest = scaled - whole;             /* exact                     */
    uint32_t n = (uint32_t)whole;
    if (rest > 0.5 || (rest == 0.5 && (n & 1u))) n += 1u;

    if (spacing_exp == -24) {
        /* subnormal range; n == 1024 is exactly the smallest normal,
           whose encoding (exponent field 1, fraction 0) is also 1024. */
        return (uint16_t)(sign | n);
    }
    int exponent = unbiased;
    if (n == 2048u) {           /* rounded up into the next binade */
        n = 1024u;
        exponent += 1;
    }
    if (exponent > 15) return (uint16_t)(sign | 0x7c00u); /* overflow */
    return (uint16_t)(sign | ((uint32_t)(exponent + 15) << 10) | (n - 1024u));
}

void oracle_f16_to_f64_array(int64_t count, const uint16_t *src, double *dst)
{
    for (int64_t i = 0; i < count; ++i) dst[i] = oracle_f16_to_f64(src[i]);
}

void oracle_f64_to_f16_array(int64_t count, const double *src, uint16_t *dst)
{
    for (int64_t i = 0; i < count; ++i) dst[i] = oracle_f64_to_f16(src[i]);
}

/* ------------------------------------------------------------------ */
/* One output element: natural-order double dot product of row i of A  */
/* and row j of B (both K-contiguous), then one rounding to binary16.   */
static void dot_entry(int64_t K, const uint16_t *a_row, const uint16_t *b_row,
                      const double *decode, uint16_t *c_out, double *absum_out,
                      double *sum_out)
{
    double sum = 0.0;
    double abs_sum = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double product = decode[a_row[k]] * decode[b_row[k]];
        sum += product;
        abs_sum += fabs(product);
    }
    *c_out = oracle_f64_to_f16(sum);
    if (absum_out) *absum_out = abs_sum;
    if (sum_out) *sum_out = sum;
}

/* The 65536-entry decode table is oracle_f16_to_f64 evaluated once per
   code point; it only saves re-decoding the same bits K times. */
static double *make_decode_table(void)
{
    double *t = (double *)malloc(sizeof(double) * 65536);
    if (!t) return NULL;
    for (uint32_t h = 0; h < 65536u; ++h) t[h] = oracle_f16_to_f64((uint16_t)h);
    return t;
}

/* Full product.  A: M*K binary16 bits, row-major; B: N*K, row-major;
   C: M*N binary16 bits, row-major.  absum / exact may be NULL, else M*N
   doubles.  Returns 0 on success, -1 if the decode table can't be made. */
int oracle_gemm_nt(int64_t M, int64_t N, int64_t K, const uint16_t *A,
                   const uint16_t *B, uint16_t *C, double *absum, double *exact)
{
    double *decode = make_decode_table();
    if (!decode) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            dot_entry(K, A + i * K, B + j * K, decode, C + i * N + j,
                      absum ? absum + i * N + j : NULL,
                      exact ? exact + i * N + j : NULL);
        }
    }
    free(decode);
    return 0;
}

/* Selected entries (rows[e], cols[e]) only, for sampled checks of sizes
   whose full product is too slow on the CPU. */
int oracle_gemm_nt_entries(int64_t M, int64_t N, int64_t K, const uint16_t *A,
                           const uint16_t *B, int64_t count, const int64_t *rows,
                           const int64_t *cols, uint16_t *C, double *absum,
                           double *exact)
{
    for (int64_t e = 0; e < count; ++e) {
        if (rows[e] < 0 || rows[e] >= M || cols[e] < 0 || cols[e] >= N) return -2;
    }
    double *decode = make_decode_table();
    if (!decode) return -1;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t e = 0; e < count; ++e) {
        dot_entry(K, A + rows[e] * K, B + cols[e] * K, decode, C + e,
                  absum ? absum + e : NULL, exact ? exact + e : NULL);
    }
    free(decode);
    return 0;
}

/* ------------------------------------------------------------------ */
/* The layout of the "wgmma_gemm.cu" page (function gemmCpu and the D   */
/* store of its kernel): D[M,N] = A[M,K] . B[K,N] with B row-major      */
/* [K,N] (N contiguous) and an fp32 result:                             */
/*     D[i][j] = fp32_rne( sum_{k} double(A[i][k]) * double(B[k][j]) )  */
/* summed in double in natural k order; the cast to float is the C      */
/* language's IEEE 754 double -> binary32 conversion (round to nearest  */
/* even in the default floating-point environment).  absum as above.    */
static void dot_entry_kn(int64_t N, int64_t K, const uint16_t *a_row, const uint16_t *b_col,
                         const double *decode, float *d_out, double *absum_out, double *sum_out)
{
    double sum = 0.0;
    double abs_sum = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double product = decode[a_row[k]] * decode[b_col[k * N]];
        sum += product;
        abs_sum += fabs(product);
    }
    *d_out = (float)sum;
    if (absum_out) *absum_out = abs_sum;
    if (sum_out) *sum_out = sum;
}

int oracle_gemm_nn_f32(int64_t M, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B,
                       float *D, double *absum, double *exact)
{
    double *decode = make_decode_table();
    if (!decode) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            dot_entry_kn(N, K, A + i * K, B + j, decode, D + i * N + j,
                         absum ? absum + i * N + j : NULL, exact ? exact + i * N + j : NULL);
        }
    }
    free(decode);
    return 0;
}

int oracle_gemm_nn_f32_entries(int64_t M, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B,
                               int64_t count, const int64_t *rows, const int64_t *cols, float *D,
                               double *absum, double *exact)
{
    for (int64_t e = 0; e < count; ++e) {
        if (rows[e] < 0 || rows[e] >= M || cols[e] < 0 || cols[e] >= N) return -2;
    }
    double *decode = make_decode_table();
    if (!decode) return -1;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t e = 0; e < count; ++e) {
        dot_entry_kn(N, K, A + rows[e] * K, B + cols[e], decode, D + e, absum ? absum + e : NULL,
                     exact ? exact + e : NULL);
    }
    free(decode);
    return 0;
}

void oracle_f64_to_f32_array(int64_t count, const double *src, float *dst)
{
    for (int64_t i = 0; i < count; ++i) dst[i] = (float)src[i];
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * sgemm_oracle.c -- fp64 CPU oracle for the row-major single-precision GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * definition that the CUDA library is checked against.  It shares no code,
 * header, table or helper with the CUDA path and is never linked into it.
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg may load it.
 *
 * What it computes (the definition of GEMM on the page "GPU GEMM 优化完全拆解
 * （一）：从朴素 Kernel 到共享内存分块", section "什么是 GEMM", with the
 * read-modify-write of C that the naive kernel on the same page and on "CUDA
 * 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS", section "1. Kernel 1", performs):
 *
 *     C[i][j] = fp32( alpha * S[i][j] + beta * C0[i][j] )
 *     S[i][j] = sum over k = 0 .. K-1, in ascending k, of
 *               (double) A[i][k] * (double) B[k][j]
 *
 * with A M x K (element (i,k) at A[i*lda + k]), B K x N (B[k*ldb + j]) and C
 * M x N (C[i*ldc + j]), all row-major.  Every float*float product is exact in
 * double (24 + 24 significant bits <= 53), so the only error before the final
 * rounding to float is the fp64 summation, at most about K * 2^-53 relative.
 *
 * Readings of points the pages leave open (the BLAS convention):
 *   - beta == 0: the beta*C0 term is omitted and C0 is not read (NaN in C0
 *     does not reach the result; C0 may be NULL).
 *   - alpha == 0 or K == 0: the alpha*S term is omitted and A, B are not read.
 *   - the final result is alpha*S + beta*C0 evaluated in double and rounded
 *     once to float (round to nearest even).
 *
 * The loops run in i-k-j order: one double accumulator row per output row,
 * so each S[i][j] is still summed in ascending k.  OpenMP splits the rows.
 *
 * The reduced-precision products (the library's sgemm_tf32 and sgemm_bf16)
 * are defined as the same sum over operands first rounded to TF32 or BF16 by
 * oracle_round_tf32 / oracle_round_bf16 below; the caller rounds A and B and
 * passes the rounded copies to the functions above (C0 is not rounded).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads the OpenMP runtime will use for a parallel region (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Fused epilogue (the library's sgemm_fused): after alpha*S + beta*C0 the
 * bias of the column is added and an activation applied, all in double,
 * before the single rounding to float:
 *     C[i][j] = fp32( act( alpha*S[i][j] + beta*C0[i][j] + bias[j] ) )
 * bias == NULL adds nothing.  The activations (the pages choose none; these
 * are the ones of the transformer FFN blocks the prefill shapes come from):
 *   ORACLE_ACT_NONE  identity
 *   ORACLE_ACT_RELU  x < 0 ? 0 : x                   (NaN stays NaN)
 *   ORACLE_ACT_GELU  x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3)))
 *                    (the tanh form of GELU)
 *   ORACLE_ACT_SILU  x / (1 + exp(-x))
 */
enum { ORACLE_ACT_NONE = 0, ORACLE_ACT_RELU = 1, ORACLE_ACT_GELU = 2, ORACLE_ACT_SILU = 3 };

static double activate(double x, int act)
{
    switch (act) {
    case ORACLE_ACT_RELU:
        return x < 0.0 ? 0.0 : x;
    case ORACLE_ACT_GELU:
        return 0.5 * x * (1.0 + tanh(0.79788456080286535588 * (x + 0.044715 * x * x * x)));
    case ORACLE_ACT_SILU:
        return x / (1.0 + exp(-x));
    default:
        return x;
    }
}

/*
 * Rows rows[0..nrows-1] of C = act(alpha*A@B + beta*C0 + bias), written
 * densely to out[r*ldo + j] for r < nrows, j < N.  C0 is indexed by the true
 * row number.  Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_sgemm_rows_fused(int64_t M, int64_t N, int64_t K, float alpha,
                            const float *A, int64_t lda, const float *B, int64_t ldb,
                            float beta, const float *C0, int64_t ldc,
                            const float *bias, int act,
                            const int64_t *rows, int64_t nrows,
                            float *out, int64_t ldo, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0 || ldo < N || act < 0 || act > ORACLE_ACT_SILU)
        return -1;
    const int use_ab = (alpha != 0.0f) && (K > 0);
    const int use_c = (beta != 0.0f);
    if (use_ab && (A == NULL || B == NULL || lda < K || ldb < N))
        return -1;
    if (use_c && (C0 == NULL || ldc < N))
        return -1;
    if (nrows > 0 && (rows == NULL || out == NULL))
        return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M)
            return -1;
    if (N == 0 || nrows == 0)
        return 0;

    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
#endif
    {
        double *acc = (double *)malloc((size_t)N * sizeof(double));
        if (acc == NULL) {
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t r = 0; r < nrows; ++r) {
                const int64_t i = rows[r];
                for (int64_t j = 0; j < N; ++j)
                    acc[j] = 0.0;
                if (use_ab) {
                    for (int64_t k = 0; k < K; ++k) {
                        const double a = (double)A[i * lda + k];
                        const float *brow = B + k * ldb;
                        for (int64_t j = 0; j < N; ++j)
                            acc[j] += a * (double)brow[j];
                    }
                }
                float *orow = out + r * ldo;
                for (int64_t j = 0; j < N; ++j) {
                    double v = use_ab ? (double)alpha * acc[j] : 0.0;
                    if (use_c)
                        v += (double)beta * (double)C0[i * ldc + j];
                    if (bias != NULL)
                        v += (double)bias[j];
                    orow[j] = (float)activate(v, act);
                }
            }
            free(acc);
        }
    }
    return failed ? -1 : 0;
}

/* Rows of C = alpha*A@B + beta*C0 (no bias, no activation). */
int oracle_sgemm_rows(int64_t M, int64_t N, int64_t K, float alpha,
                      const float *A, int64_t lda, const float *B, int64_t ldb,
                      float beta, const float *C0, int64_t ldc,
                      const int64_t *rows, int64_t nrows,
                      float *out, int64_t ldo, int nthreads)
{
    return oracle_sgemm_rows_fused(M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc, NULL,
                                   ORACLE_ACT_NONE, rows, nrows, out, ldo, nthreads);
}

/* All M rows of C = alpha*A@B + beta*C0 into out[i*ldo + j]. */
int oracle_sgemm(int64_t M, int64_t N, int64_t K, float alpha,
                 const float *A, int64_t lda, const float *B, int64_t ldb,
                 float beta, const float *C0, int64_t ldc,
                 float *out, int64_t ldo, int nthreads)
{
    if (M < 0)
        return -1;
    int64_t *rows = (int64_t *)malloc((size_t)(M > 0 ? M : 1) * sizeof(int64_t));
    if (rows == NULL)
        return -1;
    for (int64_t i = 0; i < M; ++i)
        rows[i] = i;
    int rc = oracle_sgemm_rows(M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc,
                               rows, M, out, ldo, nthreads);
    free(rows);
    return rc;
}

/*
 * TF32 keeps FP32's sign bit, its 8-bit exponent and the top 10 of its 23
 * stored mantissa bits.  out[i] = x[i] rounded to the nearest TF32 value,
 * ties away from zero.  On the bit pattern: add half the weight of the 13
 * dropped bits (0x1000) to the magnitude, then clear those 13 bits.  A carry
 * out of the mantissa moves the value to the next binade, and past the
 * largest finite TF32 value to infinity, as any round-to-nearest does.
 * Infinities are unchanged; a NaN stays a NaN (its quiet bit is set, so that
 * clearing the low bits cannot turn it into an infinity).
 */
void oracle_round_tf32(const float *x, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u;
        memcpy(&u, &x[i], sizeof u);
        if ((u & 0x7f800000u) == 0x7f800000u) {
            if (u & 0x007fffffu)
                u |= 0x00400000u;
        } else {
            u = (u + 0x1000u) & 0xffffe000u;
        }
        memcpy(&out[i], &u, sizeof u);
    }
}

/*
 * BF16 keeps FP32's sign bit, its 8-bit exponent and the top 7 of its 23
 * stored mantissa bits.  out[i] = x[i] rounded to the nearest BF16 value,
 * ties to the value whose last kept bit is 0 (round to nearest even, the
 * IEEE default).  On the bit pattern: add 0x7fff plus the last kept bit to
 * the magnitude, then clear the 16 dropped bits.  Carries and overflow behave
 * as for TF32 above; infinities are unchanged and a NaN stays a NaN.
 * out[i] holds the BF16 value as a float (its low 16 bits zero).
 */
void oracle_round_bf16(const float *x, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u;
        memcpy(&u, &x[i], sizeof u);
        if ((u & 0x7f800000u) == 0x7f800000u) {
            if (u & 0x007fffffu)
                u |= 0x00400000u;
        } else {
            u = (u + 0x7fffu + ((u >> 16) & 1u)) & 0xffff0000u;
        }
        memcpy(&out[i], &u, sizeof u);
    }
}

/*
 * gemm_oracle.c -- the plain, slow CPU definition of the dense GEMM
 *
 *     C  <-  alpha * (A x B) + beta * C
 *
 * with A (M x K), B (K x N) and C (M x N), all row-major with leading
 * dimensions lda, ldb, ldc ("GEMM Worklog I: Naive to Tiled", opening
 * equation; "A GEMM Kernel, Step by Step", section "The ladder we are
 * climbing", which states the same call for SGEMM).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle the CUDA path is checked
 * against.  Only the test suite, the package's smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header or constant with
 * the CUDA library, and the library never calls it.
 *
 * What it computes, for every i < M and j < N:
 *   acc[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]       in fp64, k increasing
 *   ref[i][j] = alpha * acc[i][j] + beta * C[i][j]       in fp64
 *   den[i][j] = |alpha| * sum_k |A[i][k]| * |B[k][j]| + |beta| * |C[i][j]|
 * and returns ref both in fp64 and rounded once to fp32.  den is the scale of
 * the error bound used by the tests.
 *
 * Readings where the pages are silent (each one is a choice, listed in the
 * design notes):
 *   - beta == 0: C is not read, so NaN or garbage in C does not propagate
 *     (the BLAS convention).
 *   - alpha == 0 or K == 0: the product term is absent and A, B are not read;
 *     the result is beta * C (or 0 when beta == 0 too).
 *   - bf16 inputs are widened exactly: a bf16 value is the IEEE binary32 whose
 *     upper 16 bits are the bf16 bit pattern and whose lower 16 bits are zero.
 *
 * Loop order is i-k-j with an fp64 row accumulator: the order of the k-sum of
 * every single element is still k = 0, 1, ..., K-1.  Rows are independent, so
 * the OpenMP split over rows does not change any result.  Build with
 * -ffp-contract=off so that no compiler fuses the multiply and the add, which
 * keeps the fp64 result identical on x86-64 and aarch64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARGS 1
#define ORACLE_NO_MEMORY 2

/* bf16 -> binary32 -> binary64; both widenings are exact. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t word = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

static int check_args(int64_t M, int64_t N, int64_t K, int64_t lda,
                      int64_t ldb, int64_t ldc, int64_t ldo)
{
    if (M < 0 || N < 0 || K < 0) return ORACLE_BAD_ARGS;
    if (lda < (K > 1 ? K : 1)) return ORACLE_BAD_ARGS;
    if (ldb < (N > 1 ? N : 1)) return ORACLE_BAD_ARGS;
    if (ldc < (N > 1 ? N : 1)) return ORACLE_BAD_ARGS;
    if (ldo < (N > 1 ? N : 1)) return ORACLE_BAD_ARGS;
    return ORACLE_OK;
}

/* Final step of one row: scale the product sum by alpha, add beta * C_old,
 * and write the fp64 value, its fp32 rounding and the error scale.  `acc`
 * and `mag` are ignored when `have_product` is 0. */
static void finish_row(int64_t N, double alpha, double beta, int have_product,
                       const double *acc, const double *mag,
                       const float *c_row, float *out_row, double *out64_row,
                       double *den_row)
{
    for (int64_t j = 0; j < N; ++j) {
        double value = 0.0;
        double scale = 0.0;
        if (have_product) {
            value = alpha * acc[j];
            scale = fabs(alpha) * mag[j];
        }
        if (beta != 0.0) {
            double c_old = (double)c_row[j];
            value = value + beta * c_old;
            scale = scale + fabs(beta) * fabs(c_old);
        }
        if (out_row) out_row[j] = (float)value;
        if (out64_row) out64_row[j] = value;
        if (den_row) den_row[j] = scale;
    }
}

/*
 * fp32 SGEMM oracle.  A, B, C are binary32, results are written to
 * out (fp32, leading dimension ldo), out64 (fp64, ldo) and den (fp64, ldo);
 * any of the three may be NULL.  C may be NULL when beta == 0.  nthreads <= 0
 * means "all available".
 */
int oracle_sgemm(int64_t M, int64_t N, int64_t K, double alpha,
                 const float *A, int64_t lda, const float *B, int64_t ldb,
                 double beta, const float *C, int64_t ldc,
                 float *out, double *out64, double *den, int64_t ldo,
                 int nthreads)
{
    int rc = check_args(M, N, K, lda, ldb, ldc, ldo);
    if (rc != ORACLE_OK) return rc;
    if (beta != 0.0 && C == NULL && M > 0 && N > 0) return ORACLE_BAD_ARGS;
    const int have_product = (alpha != 0.0 && K > 0);
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *acc = (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double));
        double *mag = (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double));
        if (acc == NULL || mag == NULL) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t i = 0; i < M; ++i) {
            if (acc == NULL || mag == NULL) continue;
            if (have_product) {
                for (int64_t j = 0; j < N; ++j) { acc[j] = 0.0; mag[j] = 0.0; }
                const float *a_row = A + i * lda;
                for (int64_t k = 0; k < K; ++k) {
                    const double a = (double)a_row[k];
                    const double abs_a = fabs(a);
                    const float *b_row = B + k * ldb;
                    for (int64_t j = 0; j < N; ++j) {
                        const double b = (double)b_row[j];
                        acc[j] = acc[j] + a * b;
                        mag[j] = mag[j] + abs_a * fabs(b);
                    }
                }
            }
            finish_row(N, alpha, beta, have_product, acc, mag,
                       beta != 0.0 ? C + i * ldc : NULL,
                       out ? out + i * ldo : NULL,
                       out64 ? out64 + i * ldo : NULL,
                       den ? den + i * ldo : NULL);
        }
        free(acc);
        free(mag);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * bf16-input oracle: A and B hold bf16 bit patterns (uint16), widened exactly
 * before the fp64 arithmetic; C, out, out64 and den are as in oracle_sgemm.
 */
int oracle_bf16gemm(int64_t M, int64_t N, int64_t K, double alpha,
                    const uint16_t *A, int64_t lda, const uint16_t *B,
                    int64_t ldb, double beta, const float *C, int64_t ldc,
                    float *out, double *out64, double *den, int64_t ldo,
                    int nthreads)
{
    int rc = check_args(M, N, K, lda, ldb, ldc, ldo);
    if (rc != ORACLE_OK) return rc;
    if (beta != 0.0 && C == NULL && M > 0 && N > 0) return ORACLE_BAD_ARGS;
    const int have_product = (alpha != 0.0 && K > 0);
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *acc = (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double));
        double *mag = (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double));
        if (acc == NULL || mag == NULL) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t i = 0; i < M; ++i) {
            if (acc == NULL || mag == NULL) continue;
            if (have_product) {
                for (int64_t j = 0; j < N; ++j) { acc[j] = 0.0; mag[j] = 0.0; }
                const uint16_t *a_row = A + i * lda;
                for (int64_t k = 0; k < K; ++k) {
                    const double a = bf16_bits_to_double(a_row[k]);
                    const double abs_a = fabs(a);
                    const uint16_t *b_row = B + k * ldb;
                    for (int64_t j = 0; j < N; ++j) {
                        const double b = bf16_bits_to_double(b_row[j]);
                        acc[j] = acc[j] + a * b;
                        mag[j] = mag[j] + abs_a * fabs(b);
                    }
                }
            }
            finish_row(N, alpha, beta, have_product, acc, mag,
                       beta != 0.0 ? C + i * ldc : NULL,
                       out ? out + i * ldo : NULL,
                       out64 ? out64 + i * ldo : NULL,
                       den ? den + i * ldo : NULL);
        }
        free(acc);
        free(mag);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* Number of threads an "all available" call would use. */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

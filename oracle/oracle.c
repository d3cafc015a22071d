/*
 * Reference oracle for dense row-major matrix multiplication.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may
 * include, link, load or call this file.  It is used by the test suite,
 * by the package's smoke check, and by the benchmark's CPU-baseline leg.
 * It shares no code, header, table or helper with the CUDA kernels.
 *
 * What it computes is the plain definition of the product, taken from
 *   "第八课：GPU 如何完成矩阵乘法" (Lesson 8: how a GPU does matrix
 *   multiplication), section 一 "矩阵乘法在算什么": for A (M x K) and
 *   B (K x N), C (M x N) has C[i][j] = sum over k = 0..K-1 of A[i][k]*B[k][j];
 *   the same element formula opens "SGEMM 优化旅程", Level 1, and the
 *   naive kernel of "4. 矩阵乘法（GEMM）优化", section 4.1.
 * Row-major addressing with leading dimensions: element (r, c) of a matrix
 * with leading dimension ld sits at index r*ld + c (the pages use the
 * compact case ld = number of columns; "4. 矩阵乘法（GEMM）优化" 4.1 and
 * Lesson 8 section 四).
 *
 * Precision: every fp32 input is widened to double; the product of two
 * widened fp32 values is exact in double (at most 48 significant bits),
 * so the only rounding is in the k-ascending double additions.  The
 * oracle's own error is therefore at most about K * 2^-53 * S, where
 * S = sum_k |A[i][k]|*|B[k][j]| (oracle_abs_gemm_f64 below).
 *
 * Build: plain C11, -O2 -ffp-contract=off, no fast-math (oracle/build.py).
 * OpenMP, if the compiler offers it, only splits the independent rows i.
 * Pins: tests/test_oracle.py checks this file against hand-computed
 * products (tests/golden/), exact rational brute force, identity and zero
 * matrices, the transpose identity, the K-slab decomposition of Lesson 8
 * section 九, and numpy's float64 matmul within the rounding bound.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of threads the row loops below may use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Cap the thread count used by later calls (n <= 0 leaves it unchanged). */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * One output row: out[j] = sum_{k ascending} A[i][k]*B[k][j] for j < N.
 * With take_abs != 0 the terms are |A[i][k]|*|B[k][j]| instead.
 * The k loop is outside the j loop, but for every fixed (i, j) the terms
 * are still added in ascending k, exactly as the element formula reads.
 */
static void one_row(int64_t i, int N, int K,
                    const float *A, int64_t lda,
                    const float *B, int64_t ldb,
                    double *out, int take_abs)
{
    for (int j = 0; j < N; ++j) out[j] = 0.0;
    for (int k = 0; k < K; ++k) {
        double a = (double)A[i * lda + k];
        if (take_abs) a = fabs(a);
        const float *brow = B + (int64_t)k * ldb;
        if (take_abs) {
            for (int j = 0; j < N; ++j) out[j] += a * fabs((double)brow[j]);
        } else {
            for (int j = 0; j < N; ++j) out[j] += a * (double)brow[j];
        }
    }
}

/*
 * C[i*ldc + j] = sum_k A[i*lda + k] * B[k*ldb + j], for i < M, j < N,
 * accumulated in double.  C is written only inside its M x N region.
 * K == 0 gives the empty sum, zero.
 */
void oracle_gemm_f64(int M, int N, int K,
                     const float *A, int lda,
                     const float *B, int ldb,
                     double *C, int ldc)
{
    int64_t m;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 4)
#endif
    for (m = 0; m < M; ++m)
        one_row(m, N, K, A, lda, B, ldb, C + m * (int64_t)ldc, 0);
}

/* S[i*lds + j] = sum_k |A[i][k]| * |B[k][j]| in double: the scale that
 * every floating-point error bound of the product is stated against. */
void oracle_abs_gemm_f64(int M, int N, int K,
                         const float *A, int lda,
                         const float *B, int ldb,
                         double *S, int lds)
{
    int64_t m;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 4)
#endif
    for (m = 0; m < M; ++m)
        one_row(m, N, K, A, lda, B, ldb, S + m * (int64_t)lds, 1);
}

/*
 * Only the rows rows[0..nrows-1] of C (and, if S is not NULL, of S):
 * out row r holds C[rows[r]][0..N-1], rows are stored compactly (stride N).
 * For products too large to evaluate whole on the CPU.
 */
void oracle_gemm_rows_f64(int nrows, const int64_t *rows, int N, int K,
                          const float *A, int lda,
                          const float *B, int ldb,
                          double *C, double *S)
{
    int64_t r;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (r = 0; r < nrows; ++r) {
        one_row(rows[r], N, K, A, lda, B, ldb, C + r * (int64_t)N, 0);
        if (S) one_row(rows[r], N, K, A, lda, B, ldb, S + r * (int64_t)N, 1);
    }
}

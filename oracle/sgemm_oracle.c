/*
 * CPU oracle for single-precision GEMM, C = alpha * A * B + beta * C, row-major.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the independent reference that the CUDA library
 * is checked against. Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * may load it; the library itself never calls it and shares no code with it.
 *
 * What it computes (the plain definition, no blocking, fusion or reordering):
 *   - "Lecture 4 - GPU Acceleration" (CMU 11-868 notes), section 5.2 "Interface":
 *     the BLAS sgemm statement C = alpha * op(A) * op(B) + beta * C, here with op = N.
 *   - "SGEMM six-level optimisation: evolution of the core code", section 2 (kernel K1):
 *     each output element is one dot product over k of A's row and B's column, scaled by
 *     alpha and added to beta times the old C; operands are row-major, A is M x K, B is
 *     K x N, element (x, i) of A sits at A[x * lda + i].
 *   - Same lecture, section 5.3: a leading dimension is the distance between the starts
 *     of two consecutive rows (row-major here), so a sub-matrix is a pointer plus an ld.
 *
 * Arithmetic: every float input is widened to double; a product of two widened floats is
 * exact in double (24 + 24 significant bits < 53), only the running sums round. The
 * result R and the magnitude sum S are returned in double, never rounded to float.
 *   R_ij = alpha * sum_k a_ik * b_kj + beta * c_ij
 *   S_ij = sum_k |a_ik * b_kj|        (used by the tests' error bound)
 *
 * BLAS reference conventions (the plainest reading of the "BLAS-style" statement; the
 * pages' own kernels always read C, which the BLAS reading does not require):
 *   - beta == 0: C is not read (NaN or garbage in C does not propagate);
 *   - alpha == 0 or K == 0: A and B are not read, R = beta * C (0 when beta == 0), S = 0;
 *   - M == 0 or N == 0: nothing to compute.
 *
 * Loop order is i, then k, then j (a row of R accumulates one scaled row of B per k),
 * which visits the same products and adds them in the same k order as the i-j-k form.
 * Rows are independent, so OpenMP splits the row list across threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One output row i, all N columns, into r[0..N) and s[0..N). */
static void oracle_row(int64_t i, int64_t N, int64_t K, double alpha, const float *A,
                       int64_t lda, const float *B, int64_t ldb, double beta,
                       const float *C, int64_t ldc, double *r, double *s) {
    for (int64_t j = 0; j < N; ++j) {
        r[j] = 0.0;
        s[j] = 0.0;
    }
    if (alpha != 0.0) {
        for (int64_t k = 0; k < K; ++k) {
            const double a = (double)A[i * lda + k];
            const float *brow = B + k * ldb;
            for (int64_t j = 0; j < N; ++j) {
                const double p = a * (double)brow[j];
                r[j] += p;
                s[j] += fabs(p);
            }
        }
    }
    for (int64_t j = 0; j < N; ++j) {
        const double ab = alpha * r[j];
        const double bc = (beta == 0.0) ? 0.0 : beta * (double)C[i * ldc + j];
        r[j] = ab + bc;
    }
}

/* Rows listed in `rows` (nrows of them, each in [0, M)); R and S are nrows x N, packed. */
int oracle_sgemm_f64_rows(int64_t M, int64_t N, int64_t K, double alpha, const float *A,
                          int64_t lda, const float *B, int64_t ldb, double beta,
                          const float *C, int64_t ldc, const int64_t *rows, int64_t nrows,
                          double *R, double *S) {
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (K == 0) alpha = 0.0; /* empty sum: A and B are not read */
    for (int64_t t = 0; t < nrows; ++t)
        if (rows[t] < 0 || rows[t] >= M) return -2;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < nrows; ++t)
        oracle_row(rows[t], N, K, alpha, A, lda, B, ldb, beta, C, ldc, R + t * N, S + t * N);
    return 0;
}

/* Every row: R and S are M x N, packed. */
int oracle_sgemm_f64(int64_t M, int64_t N, int64_t K, double alpha, const float *A,
                     int64_t lda, const float *B, int64_t ldb, double beta, const float *C,
                     int64_t ldc, double *R, double *S) {
    if (M < 0 || N < 0 || K < 0) return -1;
    if (K == 0) alpha = 0.0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i)
        oracle_row(i, N, K, alpha, A, lda, B, ldb, beta, C, ldc, R + i * N, S + i * N);
    return 0;
}

/* Single elements (ii[t], jj[t]): one dot product each, for sampled checks at any size. */
int oracle_sgemm_f64_entries(int64_t M, int64_t N, int64_t K, double alpha, const float *A,
                             int64_t lda, const float *B, int64_t ldb, double beta,
                             const float *C, int64_t ldc, const int64_t *ii,
                             const int64_t *jj, int64_t n, double *R, double *S) {
    if (M < 0 || N < 0 || K < 0 || n < 0) return -1;
    if (K == 0) alpha = 0.0;
    for (int64_t t = 0; t < n; ++t)
        if (ii[t] < 0 || ii[t] >= M || jj[t] < 0 || jj[t] >= N) return -2;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        const int64_t i = ii[t], j = jj[t];
        double r = 0.0, s = 0.0;
        if (alpha != 0.0) {
            for (int64_t k = 0; k < K; ++k) {
                const double p = (double)A[i * lda + k] * (double)B[k * ldb + j];
                r += p;
                s += fabs(p);
            }
        }
        const double bc = (beta == 0.0) ? 0.0 : beta * (double)C[i * ldc + j];
        R[t] = alpha * r + bc;
        S[t] = s;
    }
    return 0;
}

/* Threads the OpenMP runtime will use for the loops above. */
int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

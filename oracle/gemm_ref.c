/*
 * fp64 reference GEMM (test infrastructure, CPU only).
 *
 * TEST INFRASTRUCTURE: only the tests, __graft_entry__.smoke() and the
 * cpu_baseline / --impl reference legs of bench.py call this code. It shares
 * nothing with the CUDA path.
 *
 * Computes the plain definition of the GEMM from "Stream-K: Work-centric
 * Parallel Decomposition for Dense Matrix-Matrix Multiplication on the GPU",
 * §A3 (Background): C = alpha*A*B + beta*C, A is m x k, B is k x n, with every
 * product and sum in double precision. Stream-K only re-associates the k sum
 * (§3.3, §4), so this definition does not depend on any schedule.
 *
 * Layouts:
 *   a_layout 0: A(i,l) = A[i*lda + l]      (row-major, "K-major")
 *   a_layout 1: A(i,l) = A[i + l*lda]      (column-major, "M-major")
 *   b_layout 0: B(l,j) = B[j*ldb + l]      (stored n x k, "K-major")
 *   b_layout 1: B(l,j) = B[l*ldb + j]      (stored k x n, "N-major")
 *   C and C0 are row-major: C(i,j) = C[i*ldc + j].
 * beta == 0 means C0 is not read (BLAS convention: NaN in C0 does not leak).
 */
#include <stddef.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static inline double a_at(const double *A, long lda, int a_layout, long i, long l) {
  return a_layout == 0 ? A[i * lda + l] : A[i + l * lda];
}

static inline double b_at(const double *B, long ldb, int b_layout, long l, long j) {
  return b_layout == 0 ? B[j * ldb + l] : B[l * ldb + j];
}

/* One entry of the definition: alpha * sum_l A(i,l) B(l,j) + beta * C0(i,j). */
static double entry(long i, long j, long k, double alpha, const double *A, long lda,
                    int a_layout, const double *B, long ldb, int b_layout, double beta,
                    const double *C0, long ldc0) {
  double s = 0.0;
  for (long l = 0; l < k; ++l)
    s += a_at(A, lda, a_layout, i, l) * b_at(B, ldb, b_layout, l, j);
  double c = alpha * s;
  if (beta != 0.0)
    c += beta * C0[i * ldc0 + j];
  return c;
}

/* Full m x n result. Output rows are independent; OpenMP splits them. */
void oracle_gemm(long m, long n, long k, double alpha, const double *A, long lda,
                 int a_layout, const double *B, long ldb, int b_layout, double beta,
                 const double *C0, long ldc0, double *C, long ldc) {
#pragma omp parallel for schedule(dynamic, 1)
  for (long i = 0; i < m; ++i)
    for (long j = 0; j < n; ++j)
      C[i * ldc + j] = entry(i, j, k, alpha, A, lda, a_layout, B, ldb, b_layout, beta, C0, ldc0);
}

/* Selected entries (rows[s], cols[s]) of the same definition. */
void oracle_gemm_entries(long k, double alpha, const double *A, long lda, int a_layout,
                         const double *B, long ldb, int b_layout, double beta,
                         const double *C0, long ldc0, long count, const long *rows,
                         const long *cols, double *out) {
#pragma omp parallel for schedule(static)
  for (long s = 0; s < count; ++s)
    out[s] = entry(rows[s], cols[s], k, alpha, A, lda, a_layout, B, ldb, b_layout, beta, C0, ldc0);
}

/* Threads the OpenMP runtime will use (reported beside oracle timings). */
int oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

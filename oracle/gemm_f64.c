/* gemm_f64.c -- the oracle's contraction: a plain fp64 triple loop.
 *
 * TEST INFRASTRUCTURE ONLY (part of the oracle; the CUDA library never links
 * or calls it, and it includes nothing of the library).
 *
 * Page "matmul ve matmul_residual -- Tiled Matrix Multiply (Forward)"
 * (03_linear_forward), "Ne Yapar?": Y[M,N] = A[M,K] @ B[K,N], every operand
 * row-major. Written out as the definition, in i-k-j order:
 *
 *   Y[i,j] = sum over k = 0 .. K-1 of A[i,k] * B[k,j]      (k ascending)
 *   S[i,j] = sum over k = 0 .. K-1 of |A[i,k] * B[k,j]|     (the normaliser of
 *            the acceptance bound; the same products, in the same loop)
 *
 * Each output row starts at +0.0 and takes its K terms in ascending k, so the
 * rounding order is fixed and no blocking, vectorised reduction or other
 * reordering of the sum takes place. Rows are independent; with OpenMP they
 * are shared out between threads, which changes nothing in any row's sum.
 * S may be NULL (Y only).
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

void oracle_gemm_f64(const double* A, const double* B, double* Y, double* S, int64_t M,
                     int64_t N, int64_t K) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
  for (int64_t i = 0; i < M; ++i) {
    double* y = Y + i * N;
    double* s = S ? S + i * N : 0;
    for (int64_t j = 0; j < N; ++j) y[j] = 0.0;
    if (s)
      for (int64_t j = 0; j < N; ++j) s[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double a = A[i * K + k];
      const double* b = B + k * N;
      for (int64_t j = 0; j < N; ++j) y[j] += a * b[j];
      if (s)
        for (int64_t j = 0; j < N; ++j) s[j] += fabs(a * b[j]);
    }
  }
}

/* Threads the loop above runs on (1 without OpenMP). */
int oracle_gemm_threads(void) {
#ifdef _OPENMP
  int n = 1;
#pragma omp parallel
  {
#pragma omp single
    n = omp_get_num_threads();
  }
  return n;
#else
  return 1;
#endif
}

/*
 * CPU oracle for the row-major FP32 matrix product C = A * B.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline / reference arm may load or run this code. The
 * product path (the CUDA library under dense_fp32_matrix_gb300/) never calls
 * it and shares no code, header or helper with it.
 *
 * What it computes (the plain definition, no blocking, no reordering):
 *
 *   C_ij = sum_{k=0}^{K-1} A_ik * B_kj          for 0 <= i < M, 0 <= j < N
 *   S_ij = sum_{k=0}^{K-1} |A_ik * B_kj|        (scale for the error bound)
 *
 *   - "CUDA 算子优化：GEMM" (llm-tech.com.cn), section "矩阵乘法": the
 *     element formula C_ij = sum_k A_ik B_kj with A M x K, B K x N.
 *   - "GEMM from naive to tiled" (arganzheng.life), section 二.1 "FLOPs 与最小
 *     访存": each output is K products summed, all three matrices row-major.
 *   - hotelren.com/news/4711315, section 1.1: row-major element (i, j) lives
 *     at i * ld + j; section 4.2: the leading dimension ld is passed apart
 *     from the logical width.
 *
 * Precision: every product of two fp32 values is exact in fp64 (24 + 24
 * significant bits fit in 53), and the K products are summed in fp64 in
 * ascending k. The caller rounds to fp32 once when it needs an fp32 result.
 *
 * Two loop orders, both with k ascending for every (i, j):
 *   oracle_gemm_inner: i-j-k, one dot product per output ("inner product"
 *     view, hotelren.com section 1.2);
 *   oracle_gemm_outer: i-k-j, the rank-1 update sum_k A[:,k] (x) B[k,:]
 *     ("outer product" view, hotelren.com section 1.3; "SGEMM 纯 CUDA 优化总结"
 *     Q4). The page notes the rewrite does not change the mathematical
 *     result; with exact products and the same per-output summation order the
 *     two functions must agree bit for bit, which the tests check.
 *
 * Degenerate sizes (the pages are silent; plainest reading of the sum):
 *   M == 0 or N == 0: nothing to compute. K == 0: every C_ij = S_ij = 0.
 *
 * Every function returns 0 on success and -1 on an invalid argument
 * (negative size, leading dimension below the row width, null pointer where
 * elements are read or written).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static int bad_args(int64_t M, int64_t N, int64_t K, const float *A,
                    int64_t lda, const float *B, int64_t ldb) {
  if (M < 0 || N < 0 || K < 0) return 1;
  if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1)) return 1;
  if (M > 0 && K > 0 && A == NULL) return 1;
  if (K > 0 && N > 0 && B == NULL) return 1;
  return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* i-j-k: C[i*ldc + j] = sum_k A[i*lda + k] * B[k*ldb + j]. S may be NULL. */
int oracle_gemm_inner(int64_t M, int64_t N, int64_t K, const float *A,
                      int64_t lda, const float *B, int64_t ldb, double *C,
                      int64_t ldc, double *S, int64_t lds) {
  if (bad_args(M, N, K, A, lda, B, ldb)) return -1;
  if (M > 0 && N > 0 && (C == NULL || ldc < N)) return -1;
  if (S != NULL && M > 0 && N > 0 && lds < N) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      double acc = 0.0, mag = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double p = (double)A[i * lda + k] * (double)B[k * ldb + j];
        acc += p;
        mag += fabs(p);
      }
      C[i * ldc + j] = acc;
      if (S != NULL) S[i * lds + j] = mag;
    }
  }
  return 0;
}

/* i-k-j: for each row i, C[i,:] = sum_k A[i,k] * B[k,:] (rank-1 updates). */
int oracle_gemm_outer(int64_t M, int64_t N, int64_t K, const float *A,
                      int64_t lda, const float *B, int64_t ldb, double *C,
                      int64_t ldc, double *S, int64_t lds) {
  if (bad_args(M, N, K, A, lda, B, ldb)) return -1;
  if (M > 0 && N > 0 && (C == NULL || ldc < N)) return -1;
  if (S != NULL && M > 0 && N > 0 && lds < N) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < M; ++i) {
    double *c = C + i * ldc;
    double *s = S != NULL ? S + i * lds : NULL;
    for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
    if (s != NULL)
      for (int64_t j = 0; j < N; ++j) s[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double a = (double)A[i * lda + k];
      const float *b = B + k * ldb;
      if (s != NULL) {
        for (int64_t j = 0; j < N; ++j) {
          double p = a * (double)b[j];
          c[j] += p;
          s[j] += fabs(p);
        }
      } else {
        for (int64_t j = 0; j < N; ++j) c[j] += a * (double)b[j];
      }
    }
  }
  return 0;
}

/* The rows listed in `rows` (each 0 <= rows[r] < M), outer-product order.
 * Output row r of C (and S, when not NULL) is dense with width N. */
int oracle_gemm_rows(int64_t M, int64_t N, int64_t K, const float *A,
                     int64_t lda, const float *B, int64_t ldb,
                     const int64_t *rows, int64_t nrows, double *C, double *S) {
  if (bad_args(M, N, K, A, lda, B, ldb)) return -1;
  if (nrows < 0 || (nrows > 0 && (rows == NULL || (N > 0 && C == NULL))))
    return -1;
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= M) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t i = rows[r];
    double *c = C + r * N;
    double *s = S != NULL ? S + r * N : NULL;
    for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
    if (s != NULL)
      for (int64_t j = 0; j < N; ++j) s[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double a = (double)A[i * lda + k];
      const float *b = B + k * ldb;
      for (int64_t j = 0; j < N; ++j) {
        double p = a * (double)b[j];
        c[j] += p;
        if (s != NULL) s[j] += fabs(p);
      }
    }
  }
  return 0;
}

/* Single entries (ii[e], jj[e]) as dot products, k ascending. */
int oracle_gemm_entries(int64_t M, int64_t N, int64_t K, const float *A,
                        int64_t lda, const float *B, int64_t ldb,
                        const int64_t *ii, const int64_t *jj, int64_t n,
                        double *c, double *s) {
  if (bad_args(M, N, K, A, lda, B, ldb)) return -1;
  if (n < 0 || (n > 0 && (ii == NULL || jj == NULL || c == NULL))) return -1;
  for (int64_t e = 0; e < n; ++e)
    if (ii[e] < 0 || ii[e] >= M || jj[e] < 0 || jj[e] >= N) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t e = 0; e < n; ++e) {
    const int64_t i = ii[e], j = jj[e];
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      double p = (double)A[i * lda + k] * (double)B[k * ldb + j];
      acc += p;
      mag += fabs(p);
    }
    c[e] = acc;
    if (s != NULL) s[e] = mag;
  }
  return 0;
}

/*
 * The general form C = alpha * op(A) * op(B) + beta * C0, in fp64:
 *
 *   op(A)_ik = A[i*lda + k]  (op_a == 0, A stored M x K)
 *            = A[k*lda + i]  (op_a == 1, A stored K x M: op(A) = A^T)
 *   op(B)_kj = B[k*ldb + j]  (op_b == 0, B stored K x N)
 *            = B[j*ldb + k]  (op_b == 1, B stored N x K: op(B) = B^T)
 *   C_ij = alpha * (sum_k op(A)_ik op(B)_kj) + beta * C0_ij
 *   S_ij = |alpha| * (sum_k |op(A)_ik op(B)_kj|) + |beta * C0_ij|
 *
 * The pages print only alpha = 1, beta = 0 and row-major operands; the
 * transposed forms and the scalars are the BLAS reading of the cuBLAS call
 * they discuss ("GEMM from naive to tiled", sections 二.2 and 九.2): with
 * beta == 0, C0 is not read (it may hold anything, NaN included); with
 * alpha == 0 (or K == 0), A and B are not read. The K products are exact in
 * fp64 and summed in ascending k as above; the sum is then scaled once.
 */
int oracle_gemm_ex(int op_a, int op_b, int64_t M, int64_t N, int64_t K,
                   double alpha, const float *A, int64_t lda, const float *B,
                   int64_t ldb, double beta, const float *C0, int64_t ldc0,
                   double *C, int64_t ldc, double *S, int64_t lds) {
  if ((op_a != 0 && op_a != 1) || (op_b != 0 && op_b != 1)) return -1;
  if (M < 0 || N < 0 || K < 0) return -1;
  const int64_t a_cols = op_a ? M : K, b_cols = op_b ? K : N;
  if (lda < (a_cols > 1 ? a_cols : 1) || ldb < (b_cols > 1 ? b_cols : 1))
    return -1;
  const int read_ab = alpha != 0.0 && K > 0;
  if (read_ab && M > 0 && N > 0 && (A == NULL || B == NULL)) return -1;
  if (beta != 0.0 && M > 0 && N > 0 && (C0 == NULL || ldc0 < N)) return -1;
  if (M > 0 && N > 0 && (C == NULL || ldc < N)) return -1;
  if (S != NULL && M > 0 && N > 0 && lds < N) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      double acc = 0.0, mag = 0.0;
      if (read_ab) {
        for (int64_t k = 0; k < K; ++k) {
          const double a = op_a ? (double)A[k * lda + i] : (double)A[i * lda + k];
          const double b = op_b ? (double)B[j * ldb + k] : (double)B[k * ldb + j];
          const double p = a * b;
          acc += p;
          mag += fabs(p);
        }
      }
      double c = alpha * acc, s = fabs(alpha) * mag;
      if (beta != 0.0) {
        const double t = beta * (double)C0[i * ldc0 + j];
        c += t;
        s += fabs(t);
      }
      C[i * ldc + j] = c;
      if (S != NULL) S[i * lds + j] = s;
    }
  }
  return 0;
}

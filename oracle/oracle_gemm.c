/*
 * oracle_gemm.c -- the CPU oracle for dense GEMM, C = A * B.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only tests/,
 * __graft_entry__.smoke() and bench.py's cpu_baseline / reference legs load
 * this library. It shares no source, header, helper or table with the CUDA
 * library under dense_gemm_14_gb300/csrc, and neither side includes or links
 * the other.
 *
 * What it computes: the plain definition of the matrix product,
 *     C[i][j] = sum over k of A[i][k] * B[k][j],
 * for a row-major M x K matrix A and a row-major K x N matrix B, as stated in
 * gpu-hpc-book ch.06 "高级 cuda 特性 —— 从矩阵乘法(gemm)说起" (Advanced CUDA
 * features, starting from GEMM), section "缓存缺失与带宽约束分析" item (4),
 * and in "Kernel 优化指南" (cuda-kernel-academy module 02), "GEMM 优化路径",
 * Level 1 (one output element = one dot product over K, row-major indexing
 * A[row*K+k], B[k*N+col]). Tiling, double buffering and tensor cores in those
 * pages reorder this sum; they do not change it, so the oracle is the sum
 * itself, taken in the order i, k, j with no blocking.
 *
 * Precision: every input element is decoded exactly to double. A product of
 * two fp32 values (24 + 24 significant bits) or two bf16 / fp16 values is
 * exact in double, so the only rounding is in the running sum, whose relative
 * error is at most K * 2^-53. Alongside C it returns Cabs = |A| * |B| (the same
 * sum over absolute values), which scales the element-wise error bound.
 *
 * The pages do not fix the 16-bit formats (the plainest reading: IEEE binary16
 * and bfloat16 = the top half of an IEEE binary32). The decoders below are
 * written from those format definitions; fp16 subnormals, infinities and NaN
 * are decoded, not flushed.
 *
 * Errors: every entry point returns 0 on success and a negative value for an
 * invalid argument or a failed allocation; nothing aborts or prints.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2 };

/* bfloat16: the 16 high bits of an IEEE binary32 value. */
double oracle_decode_bf16(uint16_t bits) {
  uint32_t w = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_decode_f16(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int expo = (bits >> 10) & 0x1f;
  int frac = bits & 0x3ff;
  double mag;
  if (expo == 0) {
    mag = ldexp((double)frac, -24); /* subnormal: frac * 2^-10 * 2^-14 */
  } else if (expo == 31) {
    mag = frac ? NAN : INFINITY;
  } else {
    mag = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/2^10) * 2^(e-15) */
  }
  return sign ? -mag : mag;
}

static double decode_one(int dtype, const void *base, int64_t idx) {
  if (dtype == ORACLE_F32) return (double)((const float *)base)[idx];
  uint16_t b = ((const uint16_t *)base)[idx];
  return dtype == ORACLE_BF16 ? oracle_decode_bf16(b) : oracle_decode_f16(b);
}

static int check_args(int64_t M, int64_t N, int64_t K, int dtype,
                      const void *A, int64_t lda, const void *B, int64_t ldb) {
  if (M < 0 || N < 0 || K < 0) return -1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F16) return -1;
  if (lda < K || ldb < N) return -1;
  if ((M > 0 && K > 0 && !A) || (K > 0 && N > 0 && !B)) return -1;
  return 0;
}

/* Decodes a rows x cols row-major matrix (leading dimension ld) to double. */
int oracle_decode_matrix(int dtype, const void *X, int64_t rows, int64_t cols,
                         int64_t ld, double *out) {
  if (rows < 0 || cols < 0 || ld < cols) return -1;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      out[r * cols + c] = decode_one(dtype, X, r * ld + c);
  return 0;
}

/*
 * Full product. C (and Cabs, if not NULL) are M x N row-major doubles with
 * leading dimension ldc. nthreads <= 0 means the OpenMP default. Rows of C are
 * independent, so the i loop may run on several threads; within a row the sum
 * runs over k in increasing order.
 */
int oracle_gemm(int64_t M, int64_t N, int64_t K, int dtype,
                const void *A, int64_t lda, const void *B, int64_t ldb,
                double *C, double *Cabs, int64_t ldc, int nthreads) {
  if (check_args(M, N, K, dtype, A, lda, B, ldb) || ldc < N) return -1;
  if (M == 0 || N == 0) return 0;
  if (!C) return -1;

  double *Bd = NULL;
  if (K > 0) {
    Bd = (double *)malloc((size_t)K * (size_t)N * sizeof(double));
    if (!Bd) return -2;
    oracle_decode_matrix(dtype, B, K, N, ldb, Bd);
  }
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int64_t i = 0; i < M; ++i) {
    double *c = C + i * ldc;
    double *cabs = Cabs ? Cabs + i * ldc : NULL;
    for (int64_t j = 0; j < N; ++j) {
      c[j] = 0.0;
      if (cabs) cabs[j] = 0.0;
    }
    for (int64_t k = 0; k < K; ++k) {
      const double a = decode_one(dtype, A, i * lda + k);
      const double *b = Bd + k * N;
      for (int64_t j = 0; j < N; ++j) c[j] += a * b[j];
      if (cabs) {
        const double aa = fabs(a);
        for (int64_t j = 0; j < N; ++j) cabs[j] += aa * fabs(b[j]);
      }
    }
  }
  free(Bd);
  return 0;
}

/*
 * Selected entries only: out[t] = C[rows[t]][cols[t]] for t < count, each a
 * separate dot product over k (for spot checks of products too large to form
 * whole). outabs may be NULL.
 */
int oracle_gemm_entries(int64_t M, int64_t N, int64_t K, int dtype,
                        const void *A, int64_t lda, const void *B, int64_t ldb,
                        int64_t count, const int64_t *rows, const int64_t *cols,
                        double *out, double *outabs, int nthreads) {
  if (check_args(M, N, K, dtype, A, lda, B, ldb) || count < 0) return -1;
  for (int64_t t = 0; t < count; ++t)
    if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 16) num_threads(nthreads)
#endif
  for (int64_t t = 0; t < count; ++t) {
    double s = 0.0, sa = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double a = decode_one(dtype, A, rows[t] * lda + k);
      const double b = decode_one(dtype, B, k * ldb + cols[t]);
      s += a * b;
      sa += fabs(a) * fabs(b);
    }
    out[t] = s;
    if (outabs) outabs[t] = sa;
  }
  return 0;
}

/*
 * The extended product of the pages' wgmma description (gpu-hpc-book ch.06
 * "Tensor Cores" / "wgmma": D = A*B + D, with A and B optionally transposed
 * and negated, and D scaled by 0 or 1), written for general scalars:
 *     C[i][j] = alpha * sum_k opA[i][k] * opB[k][j] + beta * C0[i][j]
 * where opA[i][k] = A[i*lda + k] (transa == 0) or A[k*lda + i] (transa != 0),
 * and   opB[k][j] = B[k*ldb + j] (transb == 0) or B[j*ldb + k] (transb != 0).
 * C0 is fp32 (ldc0) and is not read when beta == 0. Cabs (if not NULL) is
 * |alpha| * sum |opA||opB| + |beta| * |C0| (0 for the second term when
 * beta == 0), the scale of the error bound. The sum runs over k in order, in
 * double; alpha * sum and beta * C0 are formed in double and added last.
 */
int oracle_gemm_ex(int64_t M, int64_t N, int64_t K, int dtype, int transa, int transb,
                   double alpha, const void *A, int64_t lda, const void *B, int64_t ldb,
                   double beta, const float *C0, int64_t ldc0, double *C, double *Cabs,
                   int64_t ldc, int nthreads) {
  if (M < 0 || N < 0 || K < 0) return -1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F16) return -1;
  if (lda < (transa ? M : K) || ldb < (transb ? K : N) || ldc < N) return -1;
  if (M == 0 || N == 0) return 0;
  if (!C || (K > 0 && (!A || !B)) || (beta != 0.0 && (!C0 || ldc0 < N))) return -1;

  /* opB decoded once, K x N row-major */
  double *Bd = NULL;
  if (K > 0) {
    Bd = (double *)malloc((size_t)K * (size_t)N * sizeof(double));
    if (!Bd) return -2;
    for (int64_t k = 0; k < K; ++k)
      for (int64_t j = 0; j < N; ++j)
        Bd[k * N + j] = decode_one(dtype, B, transb ? j * ldb + k : k * ldb + j);
  }
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int64_t i = 0; i < M; ++i) {
    double *c = C + i * ldc;
    double *cabs = Cabs ? Cabs + i * ldc : NULL;
    for (int64_t j = 0; j < N; ++j) {
      c[j] = 0.0;
      if (cabs) cabs[j] = 0.0;
    }
    for (int64_t k = 0; k < K; ++k) {
      const double a = decode_one(dtype, A, transa ? k * lda + i : i * lda + k);
      const double *b = Bd + k * N;
      for (int64_t j = 0; j < N; ++j) c[j] += a * b[j];
      if (cabs) {
        const double aa = fabs(a);
        for (int64_t j = 0; j < N; ++j) cabs[j] += aa * fabs(b[j]);
      }
    }
    for (int64_t j = 0; j < N; ++j) {
      const double c0 = beta != 0.0 ? (double)C0[i * ldc0 + j] : 0.0;
      c[j] = alpha * c[j] + (beta != 0.0 ? beta * c0 : 0.0);
      if (cabs) cabs[j] = fabs(alpha) * cabs[j] + (beta != 0.0 ? fabs(beta) * fabs(c0) : 0.0);
    }
  }
  free(Bd);
  return 0;
}

/*
 * The tf32 value the tensor cores take from an fp32 input: the binary32
 * pattern with its 13 low fraction bits cleared (truncation toward zero to 10
 * fraction bits, every exponent kept). The pages fix the format, not the
 * rounding; this is the hardware's reading of an fp32 operand. Applied to the
 * n values in place; infinities stay; a NaN whose payload lies only in the
 * cleared bits becomes an infinity, as it does in the hardware.
 */
int oracle_truncate_tf32(float *x, int64_t n) {
  if (n < 0 || (n > 0 && !x)) return -1;
  for (int64_t i = 0; i < n; ++i) {
    uint32_t w;
    memcpy(&w, &x[i], sizeof w);
    w &= ~0x1fffu;
    memcpy(&x[i], &w, sizeof w);
  }
  return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

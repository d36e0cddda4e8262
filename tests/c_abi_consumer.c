/*
 * A C (not C++) consumer of libgemm14.so through include/gemm14.h alone: the
 * device-pointer entry points with cudaMalloc'd buffers, the stream-K
 * workspace call, and the host-buffer call with tickets. Integer-valued
 * inputs make every product exact, so each result is compared bit for bit
 * with a plain int64 triple loop. Exit status 0 when every check passes.
 */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gemm14.h"

#define CHECK(cond, what)                                  \
  do {                                                     \
    if (!(cond)) {                                         \
      fprintf(stderr, "FAILED: %s (line %d)\n", what, __LINE__); \
      return 1;                                            \
    }                                                      \
  } while (0)

/* bf16 bits of a small integer (exact: |v| <= 256) */
static uint16_t bf16_of(int v) {
  float f = (float)v;
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

static int64_t lcg(uint64_t* s) {
  *s = *s * 6364136223846793005ull + 1442695040888963407ull;
  return (int64_t)((*s >> 33) % 7) - 3; /* in [-3, 3] */
}

/* C_ref = A B for int matrices (row-major, dense) */
static void ref_product(const int* A, const int* B, int64_t* C, int M, int N, int K) {
  for (int i = 0; i < M; ++i)
    for (int j = 0; j < N; ++j) {
      int64_t s = 0;
      for (int k = 0; k < K; ++k) s += (int64_t)A[i * K + k] * B[k * N + j];
      C[i * N + j] = s;
    }
}

static int same(const float* got, const int64_t* want, int n) {
  for (int i = 0; i < n; ++i)
    if (got[i] != (float)want[i]) {
      fprintf(stderr, "element %d: %.1f, want %lld\n", i, got[i], (long long)want[i]);
      return 0;
    }
  return 1;
}

int main(void) {
  const int M = 301, N = 257, K = 129;
  uint64_t seed = 14;
  int* Ai = malloc(sizeof(int) * M * K);
  int* Bi = malloc(sizeof(int) * K * N);
  int64_t* Cr = malloc(sizeof(int64_t) * M * N);
  float* Af = malloc(sizeof(float) * M * K);
  float* Bf = malloc(sizeof(float) * K * N);
  uint16_t* Ah = malloc(sizeof(uint16_t) * M * K);
  uint16_t* Bh = malloc(sizeof(uint16_t) * K * N);
  float* C = malloc(sizeof(float) * M * N);
  CHECK(Ai && Bi && Cr && Af && Bf && Ah && Bh && C, "host allocation");
  for (int i = 0; i < M * K; ++i) Ai[i] = (int)lcg(&seed), Af[i] = (float)Ai[i], Ah[i] = bf16_of(Ai[i]);
  for (int i = 0; i < K * N; ++i) Bi[i] = (int)lcg(&seed), Bf[i] = (float)Bi[i], Bh[i] = bf16_of(Bi[i]);
  ref_product(Ai, Bi, Cr, M, N, K);

  CHECK(gemm14_version() > 0, "version");
  /* host-side argument checks need no device */
  CHECK(gemm_f32(-1, N, K, NULL, K, NULL, N, NULL, N, NULL) == GEMM14_ERR_INVALID_ARG,
        "negative M rejected");

  void *dA, *dB, *dA16, *dB16, *dC, *ws;
  CHECK(cudaMalloc(&dA, sizeof(float) * M * K) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc(&dB, sizeof(float) * K * N) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc(&dA16, 2 * M * K) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc(&dB16, 2 * K * N) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc(&dC, sizeof(float) * M * N) == cudaSuccess, "cudaMalloc");
  cudaMemcpy(dA, Af, sizeof(float) * M * K, cudaMemcpyHostToDevice);
  cudaMemcpy(dB, Bf, sizeof(float) * K * N, cudaMemcpyHostToDevice);
  cudaMemcpy(dA16, Ah, 2 * M * K, cudaMemcpyHostToDevice);
  cudaMemcpy(dB16, Bh, 2 * K * N, cudaMemcpyHostToDevice);

  /* fp32 (unaligned pitches K = 129, N = 257: the element-wise loader) */
  CHECK(gemm_f32(M, N, K, dA, K, dB, N, dC, N, NULL) == GEMM14_OK, "gemm_f32");
  CHECK(gemm14_check_device_error(NULL) == GEMM14_OK, "device error word");
  cudaMemcpy(C, dC, sizeof(float) * M * N, cudaMemcpyDeviceToHost);
  CHECK(same(C, Cr, M * N), "gemm_f32 exact");

  /* bf16 with a workspace of the size asked for these operands */
  size_t wsb = gemm14_workspace_bytes_ex(GEMM14_DTYPE_BF16, 0, 0, M, N, K, dA16, K, dB16, N, dC,
                                         N, 0);
  CHECK(wsb > 0, "workspace for unaligned bf16 operands (re-pitch)");
  CHECK(cudaMalloc(&ws, wsb) == cudaSuccess && cudaMemset(ws, 0, wsb) == cudaSuccess, "workspace");
  CHECK(gemm14_gemm_ex(GEMM14_DTYPE_BF16, 0, 0, M, N, K, 1.0f, dA16, K, dB16, N, 0.0f, dC, N, ws,
                       wsb, NULL) == GEMM14_OK, "gemm14_gemm_ex bf16");
  CHECK(gemm14_check_device_error(NULL) == GEMM14_OK, "device error word");
  cudaMemcpy(C, dC, sizeof(float) * M * N, cudaMemcpyDeviceToHost);
  CHECK(same(C, Cr, M * N), "bf16 exact");

  /* the host-buffer call: operands and result in (pageable) host memory */
  memset(C, 0, sizeof(float) * M * N);
  uint64_t ticket = 0;
  CHECK(gemm14_gemm_host(GEMM14_DTYPE_F32, 0, 0, M, N, K, 1.0f, Af, K, Bf, N, 0.0f, C, N, 0,
                         &ticket) == GEMM14_OK, "gemm14_gemm_host");
  CHECK(gemm14_host_wait(ticket) == GEMM14_OK, "gemm14_host_wait");
  CHECK(same(C, Cr, M * N), "host-buffer product exact");
  CHECK(gemm14_host_synchronize() == GEMM14_OK, "gemm14_host_synchronize");

  cudaFree(dA); cudaFree(dB); cudaFree(dA16); cudaFree(dB16); cudaFree(dC); cudaFree(ws);
  free(Ai); free(Bi); free(Cr); free(Af); free(Bf); free(Ah); free(Bh); free(C);
  printf("c_abi_consumer: all checks passed\n");
  return 0;
}

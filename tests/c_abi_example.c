/*
 * A plain C program on the library's C ABI (include/gemm_gb300.h), with the
 * CUDA runtime for device memory: C = A * B^T for bf16 A (M x K) and B
 * (N x K) with fp32 C, through gemm_run on device buffers and gemm_run_host on
 * host buffers, checked against a double-precision loop on the host.
 * Prints "ok <max relative error>" and returns 0, or prints the failure and
 * returns 1.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "gemm_gb300.h"

static uint16_t to_bf16(float x) {  /* round to nearest even */
  uint32_t u;
  memcpy(&u, &x, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static double from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float x;
  memcpy(&x, &u, 4);
  return (double)x;
}

int main(void) {
  const int64_t M = 300, N = 264, K = 200;
  uint16_t* A = malloc(M * K * 2);
  uint16_t* B = malloc(N * K * 2);
  float* C = malloc(M * N * 4);
  float* C2 = malloc(M * N * 4);
  if (!A || !B || !C || !C2) return 1;
  uint32_t seed = 12345u;
  for (int64_t i = 0; i < M * K; ++i) {
    seed = seed * 1664525u + 1013904223u;
    A[i] = to_bf16((float)((int32_t)(seed >> 9) % 2001 - 1000) / 1000.0f);
  }
  for (int64_t i = 0; i < N * K; ++i) {
    seed = seed * 1664525u + 1013904223u;
    B[i] = to_bf16((float)((int32_t)(seed >> 9) % 2001 - 1000) / 1000.0f);
  }
  gemm_handle_t h;
  gemm_status_t s = gemm_create(&h, 0);
  if (s != GEMM_OK) {
    printf("gemm_create: %s\n", gemm_status_string(s));
    return 1;
  }
  void *dA, *dB, *dC;
  if (cudaMalloc(&dA, M * K * 2) != cudaSuccess || cudaMalloc(&dB, N * K * 2) != cudaSuccess ||
      cudaMalloc(&dC, M * N * 4) != cudaSuccess)
    return 1;
  cudaMemcpy(dA, A, M * K * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(dB, B, N * K * 2, cudaMemcpyHostToDevice);
  s = gemm_run(h, GEMM_OP_N, GEMM_OP_T, M, N, K, 1.0f, dA, K, dB, K, 0.0f, dC, N, GEMM_BF16_F32, NULL);
  if (s == GEMM_OK) s = gemm_run_host(h, GEMM_OP_N, GEMM_OP_T, M, N, K, 1.0f, A, K, B, K, 0.0f, C2, N,
                                      GEMM_BF16_F32, NULL);
  if (s != GEMM_OK) {
    printf("gemm_run: %s\n", gemm_status_string(s));
    return 1;
  }
  cudaDeviceSynchronize();
  cudaMemcpy(C, dC, M * N * 4, cudaMemcpyDeviceToHost);
  double worst = 0.0;
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      double r = 0.0, m = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double p = from_bf16(A[i * K + k]) * from_bf16(B[j * K + k]);
        r += p;
        m += fabs(p);
      }
      const double e1 = fabs(C[i * N + j] - r) / (m + 1e-30), e2 = fabs(C2[i * N + j] - r) / (m + 1e-30);
      if (e1 > worst) worst = e1;
      if (e2 > worst) worst = e2;
    }
  }
  gemm_destroy(h);
  cudaFree(dA);
  cudaFree(dB);
  cudaFree(dC);
  if (!(worst <= 1e-3)) {
    printf("error %g\n", worst);
    return 1;
  }
  printf("ok %g\n", worst);
  return 0;
}

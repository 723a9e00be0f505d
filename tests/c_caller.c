/*
 * c_caller.c -- a plain C program that uses librd through include/rd.h only:
 * device buffers from the CUDA runtime, one grouped forward on the default
 * stream, the result copied back and checked against a direct loop on the
 * host.  Built and run by tests/test_gpu_c_caller.py.  Prints "c caller ok"
 * and exits 0 on success.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "rd.h"

static uint16_t to_bf16(float x) {  /* round to nearest even (finite inputs) */
  uint32_t u;
  memcpy(&u, &x, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static float from_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float x;
  memcpy(&x, &u, 4);
  return x;
}

#define CK(x)                                                  \
  do {                                                         \
    cudaError_t e_ = (x);                                      \
    if (e_ != cudaSuccess) {                                   \
      printf("cuda error %s at line %d\n", cudaGetErrorString(e_), __LINE__); \
      return 1;                                                \
    }                                                          \
  } while (0)

int main(void) {
  enum { M = 64, K = 32, N = 48, G = 3 };
  const int32_t sizes[G] = {20, 0, 40}; /* rows 60..63 belong to no group: +0 */
  uint16_t* lhs = malloc(sizeof(uint16_t) * M * K);
  uint16_t* rhs = malloc(sizeof(uint16_t) * G * K * N);
  uint16_t* out = malloc(sizeof(uint16_t) * M * N);
  unsigned s = 12345u;
  for (int i = 0; i < M * K; ++i) {
    s = s * 1664525u + 1013904223u;
    lhs[i] = to_bf16((float)((int)(s >> 24) - 128) / 64.0f);
  }
  for (int i = 0; i < G * K * N; ++i) {
    s = s * 1664525u + 1013904223u;
    rhs[i] = to_bf16((float)((int)(s >> 24) - 128) / 512.0f);
  }
  void *d_lhs, *d_rhs, *d_out;
  int32_t *d_sizes, *d_status;
  CK(cudaMalloc(&d_lhs, sizeof(uint16_t) * M * K));
  CK(cudaMalloc(&d_rhs, sizeof(uint16_t) * G * K * N));
  CK(cudaMalloc(&d_out, sizeof(uint16_t) * M * N));
  CK(cudaMalloc((void**)&d_sizes, sizeof(sizes)));
  CK(cudaMalloc((void**)&d_status, sizeof(int32_t)));
  CK(cudaMemcpy(d_lhs, lhs, sizeof(uint16_t) * M * K, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_rhs, rhs, sizeof(uint16_t) * G * K * N, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_sizes, sizes, sizeof(sizes), cudaMemcpyHostToDevice));
  CK(cudaMemset(d_status, 0, sizeof(int32_t)));
  CK(cudaMemset(d_out, 0x3C, sizeof(uint16_t) * M * N)); /* a sentinel, overwritten */

  /* a rejected call: g_local past g_total */
  rd_status st = rd_ragged_dot(d_lhs, d_rhs, d_out, M, K, N, d_sizes, G, 1, G, NULL, RD_EPI_NONE,
                               d_status, NULL);
  if (st != RD_ERR_INVALID_ARG) {
    printf("expected RD_ERR_INVALID_ARG, got %s\n", rd_status_string(st));
    return 1;
  }
  st = rd_ragged_dot(d_lhs, d_rhs, d_out, M, K, N, d_sizes, G, 0, G, NULL, RD_EPI_NONE, d_status,
                     NULL);
  if (st != RD_OK) {
    printf("rd_ragged_dot: %s\n", rd_status_string(st));
    return 1;
  }
  CK(cudaDeviceSynchronize());
  int32_t status = -1;
  CK(cudaMemcpy(out, d_out, sizeof(uint16_t) * M * N, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(&status, d_status, sizeof(int32_t), cudaMemcpyDeviceToHost));
  if (status != 0) {
    printf("status word %d\n", status);
    return 1;
  }
  int bad = 0, row = 0;
  for (int j = 0; j < G; ++j) {
    for (int r = 0; r < sizes[j]; ++r, ++row) {
      for (int c = 0; c < N; ++c) {
        double acc = 0.0, mag = 0.0;
        for (int q = 0; q < K; ++q) {
          const double p = (double)from_bf16(lhs[row * K + q]) * from_bf16(rhs[(j * K + q) * N + c]);
          acc += p;
          mag += fabs(p);
        }
        const double got = from_bf16(out[row * N + c]);
        if (fabs(got - acc) > 1e-2 * fabs(acc) + 1e-3 * mag + 1e-6) ++bad;
      }
    }
  }
  for (; row < M; ++row)
    for (int c = 0; c < N; ++c)
      if (out[row * N + c] != 0) ++bad; /* rows outside the groups: +0 */
  if (bad) {
    printf("%d outputs wrong\n", bad);
    return 1;
  }
  cudaFree(d_lhs);
  cudaFree(d_rhs);
  cudaFree(d_out);
  cudaFree(d_sizes);
  cudaFree(d_status);
  free(lhs);
  free(rhs);
  free(out);
  printf("c caller ok\n");
  return 0;
}

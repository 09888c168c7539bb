/* A plain C client of libcoda: allocates device memory with the CUDA
 * runtime, runs a ragged GEMM and the LM-head cross-entropy through the
 * C ABI of include/coda.h, and checks both against double-precision loops
 * on the host. No Python and no PyTorch on this path.
 * Prints "OK" and exits 0 on success; any failure exits 1 with a message. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "coda.h"

#define FAIL(...)                     \
  do {                                \
    fprintf(stderr, __VA_ARGS__);     \
    fprintf(stderr, "\n");            \
    exit(1);                          \
  } while (0)
#define CUDA_OK(x)                                                        \
  do {                                                                    \
    cudaError_t e_ = (x);                                                 \
    if (e_ != cudaSuccess) FAIL("%s: %s", #x, cudaGetErrorString(e_));    \
  } while (0)
#define CODA_OK_(x)                                                           \
  do {                                                                        \
    coda_status_t s_ = (x);                                                   \
    if (s_ != CODA_OK) FAIL("%s: status %d (%s)", #x, (int)s_,               \
                            coda_last_error_string());                        \
  } while (0)

/* float -> bf16 with round-to-nearest-even (finite inputs), and back */
static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
static double from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static uint32_t lcg_state = 12345u;
static float uniform_pm1(void) { /* in [-1, 1) */
  lcg_state = lcg_state * 1664525u + 1013904223u;
  return (float)((lcg_state >> 8) & 0xFFFFFF) / 8388608.0f - 1.0f;
}

static void* dev_copy(const void* h, size_t bytes) {
  void* d = NULL;
  CUDA_OK(cudaMalloc(&d, bytes));
  CUDA_OK(cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice));
  return d;
}

static void check_gemm(void) {
  const int M = 300, N = 264, K = 200; /* ragged against 256-row and 256-column tiles */
  uint16_t* A = malloc(sizeof(uint16_t) * M * K);
  uint16_t* B = malloc(sizeof(uint16_t) * K * N);
  float* C = malloc(sizeof(float) * M * N);
  for (int i = 0; i < M * K; ++i) A[i] = to_bf16(uniform_pm1());
  for (int i = 0; i < K * N; ++i) B[i] = to_bf16(uniform_pm1());
  void* dA = dev_copy(A, sizeof(uint16_t) * M * K);
  void* dB = dev_copy(B, sizeof(uint16_t) * K * N);
  void* dC = NULL;
  CUDA_OK(cudaMalloc(&dC, sizeof(float) * M * N));
  CODA_OK_(coda_gemm(dA, K, 0, dB, N, 0, NULL, NULL, dC, N, 1, M, N, K, NULL));
  CODA_OK_(coda_get_device_error(NULL));
  CUDA_OK(cudaMemcpy(C, dC, sizeof(float) * M * N, cudaMemcpyDeviceToHost));
  double err = 0.0, ref_max = 0.0;
  for (int m = 0; m < M; ++m)
    for (int n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k) acc += from_bf16(A[m * K + k]) * from_bf16(B[k * N + n]);
      err = fmax(err, fabs((double)C[m * N + n] - acc));
      ref_max = fmax(ref_max, fabs(acc));
    }
  if (!(err / ref_max <= 1e-5)) FAIL("gemm: max rel err %.3e", err / ref_max);
  printf("gemm %dx%dx%d fp32 out: max rel err %.3e\n", M, N, K, err / ref_max);
  cudaFree(dA);
  cudaFree(dB);
  cudaFree(dC);
  free(A);
  free(B);
  free(C);
}

static void check_lmhead_ce(void) {
  const int M = 64, d = 64, V = 1000;
  uint16_t* H = malloc(sizeof(uint16_t) * M * d);
  uint16_t* W = malloc(sizeof(uint16_t) * d * V);
  int32_t* t = malloc(sizeof(int32_t) * M);
  float* lse = malloc(sizeof(float) * M);
  float* loss = malloc(sizeof(float) * M);
  for (int i = 0; i < M * d; ++i) H[i] = to_bf16(uniform_pm1());
  for (int i = 0; i < d * V; ++i) W[i] = to_bf16(0.5f * uniform_pm1());
  for (int m = 0; m < M; ++m) t[m] = (int32_t)((m * 7919) % V);
  void* dH = dev_copy(H, sizeof(uint16_t) * M * d);
  void* dW = dev_copy(W, sizeof(uint16_t) * d * V);
  void* dt = dev_copy(t, sizeof(int32_t) * M);
  float *dlse = NULL, *dloss = NULL;
  CUDA_OK(cudaMalloc((void**)&dlse, sizeof(float) * M));
  CUDA_OK(cudaMalloc((void**)&dloss, sizeof(float) * M));
  const size_t wsb = coda_lmhead_ce_workspace_size(M, V);
  void* ws = NULL;
  CUDA_OK(cudaMalloc(&ws, wsb));
  CODA_OK_(coda_lmhead_ce(dH, dW, (const int32_t*)dt, dlse, dloss, ws, wsb, M, V, d, NULL));
  CODA_OK_(coda_get_device_error(NULL));
  CUDA_OK(cudaMemcpy(lse, dlse, sizeof(float) * M, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(loss, dloss, sizeof(float) * M, cudaMemcpyDeviceToHost));
  double err = 0.0, ref_max = 0.0;
  double* l = malloc(sizeof(double) * V);
  for (int m = 0; m < M; ++m) {
    double mx = -INFINITY, s = 0.0;
    for (int v = 0; v < V; ++v) {
      double acc = 0.0;
      for (int k = 0; k < d; ++k) acc += from_bf16(H[m * d + k]) * from_bf16(W[k * V + v]);
      l[v] = acc;
      mx = fmax(mx, acc);
    }
    for (int v = 0; v < V; ++v) s += exp(l[v] - mx);
    const double ref_lse = mx + log(s), ref_loss = ref_lse - l[t[m]];
    err = fmax(err, fmax(fabs(lse[m] - ref_lse), fabs(loss[m] - ref_loss)));
    ref_max = fmax(ref_max, fmax(fabs(ref_lse), fabs(ref_loss)));
  }
  if (!(err / ref_max <= 1e-4)) FAIL("lmhead_ce: max rel err %.3e", err / ref_max);
  printf("lmhead_ce M=%d d=%d V=%d: max rel err %.3e\n", M, d, V, err / ref_max);
  cudaFree(dH);
  cudaFree(dW);
  cudaFree(dt);
  cudaFree(dlse);
  cudaFree(dloss);
  cudaFree(ws);
  free(H);
  free(W);
  free(t);
  free(lse);
  free(loss);
  free(l);
}

int main(void) {
  check_gemm();
  check_lmhead_ce();
  printf("OK\n");
  return 0;
}

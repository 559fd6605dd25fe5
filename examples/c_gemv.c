/* c_gemv.c -- the C ABI from C, no Python: pack an FP32 matrix to NVFP4 on
 * the device, run the GEMV for N columns, read the device error word, and
 * check y on the host against an FP64 sum over the unpacked codes.
 *
 * Build from the repository root once libvgemm.so exists
 * (python -m verify_gemm_gb300.build):
 *
 *   nvcc -x c -O2 examples/c_gemv.c -Iinclude -Lverify_gemm_gb300/_build -lvgemm -lm \
 *        -Xlinker -rpath -Xlinker $PWD/verify_gemm_gb300/_build -o c_gemv && ./c_gemv
 *
 * Exit status 0 when every y is within 4e-3 * sum|w x| + 1e-6 of the sum. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "vgemm.h"

#define CK(call)                                                                    \
  do {                                                                              \
    vg_status s_ = (call);                                                          \
    if (s_ != VG_OK) {                                                              \
      fprintf(stderr, "%s: %s (%s)\n", #call, vg_status_string(s_),                \
              vg_last_cuda_error());                                                \
      return 1;                                                                     \
    }                                                                               \
  } while (0)
#define CU(call)                                                                    \
  do {                                                                              \
    cudaError_t e_ = (call);                                                        \
    if (e_ != cudaSuccess) {                                                        \
      fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));                   \
      return 1;                                                                     \
    }                                                                               \
  } while (0)

/* Seeded normal samples: a 64-bit LCG and the Box-Muller transform. */
static uint64_t rng_state = 12345u;
static double uniform01(void) {
  rng_state = rng_state * 6364136223846793005ull + 1442695040888963407ull;
  return (double)(rng_state >> 11) / 9007199254740992.0;
}
static double normal(void) {
  const double u = uniform01(), v = uniform01();
  return sqrt(-2.0 * log(u + 1e-300)) * cos(6.283185307179586 * v);
}

/* FP32 -> BF16 bits, round to nearest even (finite values), and back. */
static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
static double from_bf16(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* E2M1 magnitudes by the low three bits of a code (bit 3 is the sign), and
 * the value of a non-negative finite E4M3 byte (bias 7, subnormals m * 2^-9). */
static const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
static double e4m3_value(uint8_t b) {
  const int e = (b >> 3) & 15, m = b & 7;
  return e ? ldexp(1.0 + m / 8.0, e - 7) : ldexp((double)m, -9);
}

int main(void) {
  const int64_t M = 1000, K = 2048;   /* 1000 rows: a ragged last tile */
  const int N = 4;
  size_t w_bytes = 0, s_bytes = 0, ws_bytes = 0;
  CK(vg_nvfp4_sizes(M, K, &w_bytes, &s_bytes));
  CK(vg_gemv_workspace_size_n(M, K, VG_FMT_NVFP4, N, &ws_bytes));

  float *hW = malloc(sizeof(float) * M * K);
  uint16_t *hx = malloc(sizeof(uint16_t) * N * K), *hy = malloc(sizeof(uint16_t) * N * M);
  uint8_t *hnib = malloc(M * K / 2), *hsc = malloc(M * K / 16);
  if (!hW || !hx || !hy || !hnib || !hsc) return 1;
  for (int64_t i = 0; i < M * K; ++i) hW[i] = (float)(0.02 * normal());
  for (int64_t i = 0; i < N * K; ++i) hx[i] = to_bf16((float)normal());

  float *dW;
  void *dw, *ds, *dws;
  uint16_t *dx, *dy;
  uint8_t *dnib, *dsc;
  CU(cudaMalloc((void **)&dW, sizeof(float) * M * K));
  CU(cudaMalloc(&dw, w_bytes));
  CU(cudaMalloc(&ds, s_bytes));
  CU(cudaMalloc(&dws, ws_bytes));
  CU(cudaMalloc((void **)&dx, sizeof(uint16_t) * N * K));
  CU(cudaMalloc((void **)&dy, sizeof(uint16_t) * N * M));
  CU(cudaMalloc((void **)&dnib, M * K / 2));
  CU(cudaMalloc((void **)&dsc, M * K / 16));
  CU(cudaMemcpy(dW, hW, sizeof(float) * M * K, cudaMemcpyHostToDevice));
  CU(cudaMemcpy(dx, hx, sizeof(uint16_t) * N * K, cudaMemcpyHostToDevice));
  CU(cudaMemset(dws, 0, ws_bytes));   /* zero-filled once, then reused */

  float gscale = 0.0f;
  CK(vg_nvfp4_pack(dW, M, K, dw, ds, &gscale, NULL));
  CK(vg_gemv_nvfp4(dw, ds, gscale, dx, N, M, K, dy, dws, ws_bytes, NULL));
  int device_error = 0;
  CK(vg_gemv_workspace_check(dws, ws_bytes, &device_error, NULL));
  CK(vg_nvfp4_unpack(dw, ds, M, K, dnib, dsc, NULL));
  CU(cudaMemcpy(hy, dy, sizeof(uint16_t) * N * M, cudaMemcpyDeviceToHost));
  CU(cudaMemcpy(hnib, dnib, M * K / 2, cudaMemcpyDeviceToHost));
  CU(cudaMemcpy(hsc, dsc, M * K / 16, cudaMemcpyDeviceToHost));

  /* y[n][m] against the FP64 sum of x * (e2m1 * block scale * tensor scale)
   * over the canonical codes (low nibble: even k) */
  double worst = 0.0;
  for (int64_t m = 0; m < M; ++m) {
    for (int n = 0; n < N; ++n) {
      double sum = 0.0, abs_sum = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const uint8_t byte = hnib[m * (K / 2) + k / 2];
        const int code = (k & 1) ? byte >> 4 : byte & 15;
        const double w = ((code & 8) ? -1.0 : 1.0) * kE2M1[code & 7] *
                         e4m3_value(hsc[m * (K / 16) + k / 16]) * (double)gscale;
        const double p = w * from_bf16(hx[n * K + k]);
        sum += p;
        abs_sum += fabs(p);
      }
      const double r = fabs(from_bf16(hy[n * M + m]) - sum) / (4e-3 * abs_sum + 1e-6);
      if (r > worst) worst = r;
    }
  }
  printf("NVFP4 %lld x %lld, N = %d: worst error / tolerance %.3f\n", (long long)M,
         (long long)K, N, worst);

  cudaFree(dW);
  cudaFree(dw);
  cudaFree(ds);
  cudaFree(dws);
  cudaFree(dx);
  cudaFree(dy);
  cudaFree(dnib);
  cudaFree(dsc);
  free(hW);
  free(hx);
  free(hy);
  free(hnib);
  free(hsc);
  return worst <= 1.0 ? 0 : 2;
}

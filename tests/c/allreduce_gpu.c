/* A C99 caller on the GPU, with no Python in the process: replicas of small
 * integers (exact in bf16 and in the fp32 sum) are all-reduced by the library;
 * every replica must hold the exact mean afterwards.  Exit status 0 = pass. */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "dpsync.h"

static uint16_t bf16_of_small_int(int v) { /* exact for |v| < 256 */
  float f = (float)v;
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

static float f32_of_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

int main(void) {
  const int32_t P = 8;
  const int64_t sizes[4] = {3, 70000, 4097, 12};
  dp_plan* plan = NULL;
  if (dp_plan_buckets(sizes, NULL, 4, 64 * 1024, P, &plan) != DP_OK) {
    fprintf(stderr, "plan: %s\n", dp_last_error());
    return 1;
  }
  dp_plan_info_t info;
  dp_plan_info(plan, &info);
  const size_t n_rep = (size_t)P * (size_t)info.replica_stride;
  uint16_t* h = (uint16_t*)calloc(n_rep, 2);
  if (!h) return 2;
  /* value of element i of tensor t on rank r: ((7 t + 3 i + 5 r) mod 64) - 32 */
  for (int32_t t = 0; t < 4; ++t) {
    int32_t b;
    int64_t off;
    dp_plan_tensor(plan, t, &b, &off);
    for (int64_t i = 0; i < sizes[t]; ++i)
      for (int32_t r = 0; r < P; ++r)
        h[(size_t)r * info.replica_stride + off + i] =
            bf16_of_small_int((int)((7 * t + 3 * i + 5 * r) % 64) - 32);
  }
  void *d_rep = NULL, *d_ws = NULL;
  if (cudaMalloc(&d_rep, n_rep * 2) != cudaSuccess || cudaMalloc(&d_ws, info.workspace_bytes) != cudaSuccess)
    return 3;
  cudaMemcpy(d_rep, h, n_rep * 2, cudaMemcpyHostToDevice);
  if (dp_plan_upload(plan, d_ws, NULL) != DP_OK || dp_allreduce_mean(plan, d_ws, d_rep, 0, info.n_buckets, NULL) != DP_OK) {
    fprintf(stderr, "allreduce: %s\n", dp_last_error());
    return 4;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return 5;
  cudaMemcpy(h, d_rep, n_rep * 2, cudaMemcpyDeviceToHost);
  long bad = 0;
  for (int32_t t = 0; t < 4; ++t) {
    int32_t b;
    int64_t off;
    dp_plan_tensor(plan, t, &b, &off);
    for (int64_t i = 0; i < sizes[t]; ++i) {
      int sum = 0;
      for (int32_t r = 0; r < P; ++r) sum += (int)((7 * t + 3 * i + 5 * r) % 64) - 32;
      const float want = (float)sum / (float)P; /* a multiple of 1/8: exact in bf16 here */
      for (int32_t r = 0; r < P; ++r)
        if (f32_of_bf16(h[(size_t)r * info.replica_stride + off + i]) != want) ++bad;
    }
  }
  printf("mismatches %ld\n", bad);
  cudaFree(d_rep);
  cudaFree(d_ws);
  free(h);
  dp_plan_free(plan);
  return bad == 0 ? 0 : 6;
}

/* A C99 caller of the fused ZeRO-1/2 step on the GPU, with no Python in the
 * process.  Usage: zero_step_gpu <inputs> <outputs>
 *   inputs:  for each of the STEPS steps the bf16 gradients of every rank in
 *            tensor order (uint16 [P][N]), then the fp32 master weights [N];
 *   outputs: the bf16 parameters of every replica in tensor order
 *            (uint16 [P][N]), fp32 master, m and v [N] after the last step, and
 *            per step the norm (double) and clip coefficient (float).
 * It plans, uploads, runs dp_fused_zero_step with clipping for STEPS steps and
 * reads each step's norm with dp_read_norm.  Exit status 0 = every call
 * succeeded. */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "dpsync.h"

#define P 4
#define NT 5
#define STEPS 2

static const int64_t kSizes[NT] = {3, 70000, 4097, 12, 33000};
static const uint8_t kDecay[NT] = {1, 1, 0, 0, 1};

static int64_t total(void) {
  int64_t n = 0;
  for (int t = 0; t < NT; ++t) n += kSizes[t];
  return n;
}

/* copy n elements of `elem` bytes from tensor order (src) to the flat layout
 * (dst, row of the padded index space), or back when to_flat == 0 */
static void relayout(const dp_plan* plan, void* flat, void* ord, size_t elem, int to_flat) {
  int64_t base = 0;
  for (int32_t t = 0; t < NT; ++t) {
    int32_t b;
    int64_t off;
    dp_plan_tensor(plan, t, &b, &off);
    char* f = (char*)flat + (size_t)off * elem;
    char* o = (char*)ord + (size_t)base * elem;
    if (to_flat)
      memcpy(f, o, (size_t)kSizes[t] * elem);
    else
      memcpy(o, f, (size_t)kSizes[t] * elem);
    base += kSizes[t];
  }
}

int main(int argc, char** argv) {
  if (argc != 3) return 1;
  const int64_t N = total();
  dp_plan* plan = NULL;
  if (dp_plan_buckets(kSizes, kDecay, NT, 64 * 1024, P, &plan) != DP_OK) {
    fprintf(stderr, "plan: %s\n", dp_last_error());
    return 2;
  }
  dp_plan_info_t info;
  dp_plan_info(plan, &info);
  const int64_t L = info.padded_len, stride = info.replica_stride;
  const size_t rep_bytes = (size_t)P * (size_t)stride * 2, st_bytes = (size_t)L * 4;

  /* inputs */
  FILE* fin = fopen(argv[1], "rb");
  if (!fin) return 3;
  uint16_t* g_in = (uint16_t*)malloc((size_t)STEPS * P * N * 2);
  float* master_in = (float*)malloc((size_t)N * 4);
  if (!g_in || !master_in) return 4;
  if (fread(g_in, 2, (size_t)STEPS * P * N, fin) != (size_t)STEPS * P * N ||
      fread(master_in, 4, (size_t)N, fin) != (size_t)N)
    return 5;
  fclose(fin);

  /* device buffers; padding slots stay zero */
  void *d_grads = NULL, *d_params = NULL, *d_ws = NULL;
  float *d_master = NULL, *d_m = NULL, *d_v = NULL;
  if (cudaMalloc(&d_grads, rep_bytes) != cudaSuccess || cudaMalloc(&d_params, rep_bytes) != cudaSuccess ||
      cudaMalloc((void**)&d_master, st_bytes) != cudaSuccess || cudaMalloc((void**)&d_m, st_bytes) != cudaSuccess ||
      cudaMalloc((void**)&d_v, st_bytes) != cudaSuccess || cudaMalloc(&d_ws, (size_t)info.workspace_bytes) != cudaSuccess)
    return 6;
  cudaMemset(d_grads, 0, rep_bytes);
  cudaMemset(d_params, 0, rep_bytes);
  cudaMemset(d_m, 0, st_bytes);
  cudaMemset(d_v, 0, st_bytes);
  uint16_t* h_rep = (uint16_t*)calloc((size_t)P * (size_t)stride, 2);
  float* h_st = (float*)calloc((size_t)L, 4);
  if (!h_rep || !h_st) return 7;
  relayout(plan, h_st, master_in, 4, 1);
  cudaMemcpy(d_master, h_st, st_bytes, cudaMemcpyHostToDevice);
  if (dp_plan_upload(plan, d_ws, NULL) != DP_OK) return 8;

  double norms[STEPS];
  float coefs[STEPS];
  for (int s = 0; s < STEPS; ++s) {
    for (int r = 0; r < P; ++r)
      relayout(plan, h_rep + (size_t)r * stride, g_in + ((size_t)s * P + r) * N, 2, 1);
    cudaMemcpy(d_grads, h_rep, rep_bytes, cudaMemcpyHostToDevice);
    const dp_adamw_cfg cfg = {2e-4, 0.9, 0.95, 1e-8, 0.1, 1.0, s + 1};
    if (dp_fused_zero_step(plan, d_ws, d_grads, d_params, d_master, d_m, d_v, &cfg, NULL, NULL) != DP_OK) {
      fprintf(stderr, "zero step: %s\n", dp_last_error());
      return 9;
    }
    int32_t status = -1;
    if (dp_read_norm(plan, d_ws, &norms[s], &coefs[s], &status, NULL) != DP_OK || status != 0) {
      fprintf(stderr, "read norm: %s (status %d)\n", dp_last_error(), status);
      return 10;
    }
  }

  /* outputs, in tensor order */
  FILE* fout = fopen(argv[2], "wb");
  if (!fout) return 11;
  uint16_t* ord16 = (uint16_t*)malloc((size_t)N * 2);
  float* ord32 = (float*)malloc((size_t)N * 4);
  if (!ord16 || !ord32) return 12;
  cudaMemcpy(h_rep, d_params, rep_bytes, cudaMemcpyDeviceToHost);
  for (int r = 0; r < P; ++r) {
    relayout(plan, h_rep + (size_t)r * stride, ord16, 2, 0);
    fwrite(ord16, 2, (size_t)N, fout);
  }
  float* arrays[3] = {d_master, d_m, d_v};
  for (int a = 0; a < 3; ++a) {
    cudaMemcpy(h_st, arrays[a], st_bytes, cudaMemcpyDeviceToHost);
    relayout(plan, h_st, ord32, 4, 0);
    fwrite(ord32, 4, (size_t)N, fout);
  }
  fwrite(norms, sizeof(double), STEPS, fout);
  fwrite(coefs, sizeof(float), STEPS, fout);
  fclose(fout);
  if (cudaDeviceSynchronize() != cudaSuccess) return 13;
  printf("zero step ok: norms %.6f %.6f\n", norms[0], norms[1]);
  cudaFree(d_grads);
  cudaFree(d_params);
  cudaFree(d_master);
  cudaFree(d_m);
  cudaFree(d_v);
  cudaFree(d_ws);
  free(g_in);
  free(master_in);
  free(h_rep);
  free(h_st);
  free(ord16);
  free(ord32);
  dp_plan_free(plan);
  return 0;
}

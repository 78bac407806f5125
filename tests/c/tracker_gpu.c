/* A C99 caller of the readiness tracker, with no Python in the process.  A
 * producer stream of the highest priority uploads each tensor's gradients in
 * backward order (last tensor first), records an event and marks the tensor
 * ready; the tracker fires every complete bucket's mean all-reduce as
 * short-lived CTAs on a stream of the lowest priority.  Replicas hold small
 * integers, so every mean is exact in bf16: every replica must hold it, the
 * buckets must fire in plan order, one launch each, and a plain
 * dp_allreduce_mean on a stream set to short-lived CTAs must give the same bits.
 * Exit status 0 = pass. */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "dpsync.h"

#define NT 6

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

static int value(int32_t t, int64_t i, int32_t r) { return (int)((7 * t + 3 * i + 5 * r) % 64) - 32; }

int main(void) {
  const int32_t P = 8;
  const int64_t sizes[NT] = {3, 70000, 4097, 12, 33000, 900};
  dp_plan* plan = NULL;
  if (dp_plan_buckets(sizes, NULL, NT, 64 * 1024, P, &plan) != DP_OK) {
    fprintf(stderr, "plan: %s\n", dp_last_error());
    return 1;
  }
  dp_plan_info_t info;
  dp_plan_info(plan, &info);
  const size_t stride = (size_t)info.replica_stride, n_rep = (size_t)P * stride;
  uint16_t* h = (uint16_t*)calloc(n_rep, 2);
  uint16_t* back = (uint16_t*)calloc(n_rep, 2);
  uint16_t* back2 = (uint16_t*)calloc(n_rep, 2);
  if (!h || !back || !back2) return 2;
  int64_t offs[NT];
  for (int32_t t = 0; t < NT; ++t) {
    int32_t b;
    dp_plan_tensor(plan, t, &b, &offs[t]);
    for (int64_t i = 0; i < sizes[t]; ++i)
      for (int32_t r = 0; r < P; ++r) h[(size_t)r * stride + offs[t] + i] = bf16_of_small_int(value(t, i, r));
  }
  void *d_rep = NULL, *d_rep2 = NULL, *d_ws = NULL;
  if (cudaMalloc(&d_rep, n_rep * 2) != cudaSuccess || cudaMalloc(&d_rep2, n_rep * 2) != cudaSuccess ||
      cudaMalloc(&d_ws, info.workspace_bytes) != cudaSuccess)
    return 3;
  cudaMemset(d_rep, 0, n_rep * 2);
  int lowest = 0, highest = 0;
  cudaDeviceGetStreamPriorityRange(&lowest, &highest);
  cudaStream_t comm, producer;
  if (cudaStreamCreateWithPriority(&comm, cudaStreamNonBlocking, lowest) != cudaSuccess ||
      cudaStreamCreateWithPriority(&producer, cudaStreamNonBlocking, highest) != cudaSuccess)
    return 3;
  if (dp_plan_upload(plan, d_ws, NULL) != DP_OK || cudaDeviceSynchronize() != cudaSuccess) return 4;

  dp_tracker* tr = NULL;
  if (dp_tracker_create(plan, DP_TRACK_ALLREDUCE, d_ws, d_rep, NULL, comm, 0, DP_TRACK_SHORT_CTAS, &tr) !=
      DP_OK) {
    fprintf(stderr, "tracker: %s\n", dp_last_error());
    return 4;
  }
  cudaEvent_t ev[NT];
  for (int32_t t = 0; t < NT; ++t) cudaEventCreateWithFlags(&ev[t], cudaEventDisableTiming);
  if (dp_tracker_begin(tr) != DP_OK) return 5;
  for (int32_t t = NT - 1; t >= 0; --t) { /* backward order: last tensor first */
    const size_t o = (size_t)offs[t];
    if (cudaMemcpy2DAsync((uint16_t*)d_rep + o, stride * 2, h + o, stride * 2, (size_t)sizes[t] * 2, (size_t)P,
                          cudaMemcpyHostToDevice, producer) != cudaSuccess ||
        cudaEventRecord(ev[t], producer) != cudaSuccess)
      return 5;
    if (dp_tracker_mark_ready(tr, t, ev[t]) != DP_OK) {
      fprintf(stderr, "mark: %s\n", dp_last_error());
      return 5;
    }
  }
  if (dp_tracker_wait(tr, 10000) != DP_OK) {
    fprintf(stderr, "wait: %s\n", dp_last_error());
    return 6;
  }
  int32_t order[64], n_fired = 0, launches = 0, waits = 0;
  dp_tracker_fired(tr, order, 64, &n_fired);
  dp_tracker_stats(tr, &launches, &waits);
  int bad_order = n_fired != info.n_buckets || launches != info.n_buckets;
  for (int32_t i = 0; i < n_fired && i < 64; ++i) bad_order |= order[i] != i;
  if (cudaStreamSynchronize(comm) != cudaSuccess) return 7;
  cudaMemcpy(back, d_rep, n_rep * 2, cudaMemcpyDeviceToHost);

  /* the same all-reduce as one call on a stream set to short-lived CTAs */
  if (cudaMemcpy(d_rep2, h, n_rep * 2, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) /* a pageable copy may still be in flight */
    return 8;
  if (dp_stream_set_launch(comm, DP_LAUNCH_SHORT_CTAS) != DP_OK ||
      dp_allreduce_mean(plan, d_ws, d_rep2, 0, info.n_buckets, comm) != DP_OK ||
      dp_stream_set_launch(comm, DP_LAUNCH_DEFAULT) != DP_OK || cudaStreamSynchronize(comm) != cudaSuccess)
    return 8;
  cudaMemcpy(back2, d_rep2, n_rep * 2, cudaMemcpyDeviceToHost);

  long bad = 0;
  for (int32_t t = 0; t < NT; ++t)
    for (int64_t i = 0; i < sizes[t]; ++i) {
      int sum = 0;
      for (int32_t r = 0; r < P; ++r) sum += value(t, i, r);
      const float want = (float)sum / (float)P; /* a multiple of 1/8: exact in bf16 here */
      for (int32_t r = 0; r < P; ++r) {
        const size_t k = (size_t)r * stride + (size_t)offs[t] + (size_t)i;
        if (f32_of_bf16(back[k]) != want || back2[k] != back[k]) ++bad;
      }
    }
  printf("buckets %d fired %d launches %d waits %d order %s mismatches %ld\n", (int)info.n_buckets,
         (int)n_fired, (int)launches, (int)waits, bad_order ? "wrong" : "ok", bad);
  for (int32_t t = 0; t < NT; ++t) cudaEventDestroy(ev[t]);
  dp_tracker_free(tr);
  cudaStreamDestroy(comm);
  cudaStreamDestroy(producer);
  cudaFree(d_rep);
  cudaFree(d_rep2);
  cudaFree(d_ws);
  free(h);
  free(back);
  free(back2);
  dp_plan_free(plan);
  return bad == 0 && !bad_order ? 0 : 9;
}

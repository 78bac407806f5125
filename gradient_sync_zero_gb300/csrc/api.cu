// C ABI entry points: argument checks, bucket-range -> tile-range mapping, and
// dispatch to the kernel launchers.  No device memory is allocated here; every
// call only enqueues work on the caller's stream (dp_read_norm also syncs it).
#include <cuda_runtime.h>

#include <cstddef>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>

#include "internal.h"

namespace dps {

int adam_scalars(const char* fn, const dp_adamw_cfg* cfg, AdamScalars* s) {
  if (!cfg) return fail(DP_EINVAL, std::string(fn) + ": NULL cfg");
  if (cfg->step < 1) return fail(DP_EINVAL, std::string(fn) + ": step must be >= 1");
  if (!(cfg->beta1 >= 0.0 && cfg->beta1 < 1.0 && cfg->beta2 >= 0.0 && cfg->beta2 < 1.0))
    return fail(DP_EINVAL, std::string(fn) + ": betas must be in [0, 1)");
  // Scalar factors formed once in double and rounded to fp32 (torch.optim.AdamW
  // forms them as Python floats): decay factor 1 - lr*wd, 1-b1, 1-b2,
  // step size lr / (1 - b1^t) and sqrt(1 - b2^t).
  const double t = static_cast<double>(cfg->step);
  s->wd_factor = static_cast<float>(1.0 - cfg->lr * cfg->weight_decay);
  s->b1 = static_cast<float>(cfg->beta1);
  s->omb1 = static_cast<float>(1.0 - cfg->beta1);
  s->b2 = static_cast<float>(cfg->beta2);
  s->omb2 = static_cast<float>(1.0 - cfg->beta2);
  s->step_size = static_cast<float>(cfg->lr / (1.0 - std::pow(cfg->beta1, t)));
  s->sqrt_bc2 = static_cast<float>(std::sqrt(1.0 - std::pow(cfg->beta2, t)));
  s->eps = static_cast<float>(cfg->eps);
  return DP_OK;
}

namespace {

// Streams set to DP_LAUNCH_SHORT_CTAS, by handle.  The count lets the common
// case (no stream set) skip the lock.
std::mutex g_shape_mu;
std::unordered_map<void*, int32_t> g_shape;
std::atomic<int> g_shape_count{0};

}  // namespace

bool stream_short_ctas(void* stream) {
  if (g_shape_count.load(std::memory_order_acquire) == 0) return false;
  std::lock_guard<std::mutex> lock(g_shape_mu);
  const auto it = g_shape.find(stream);
  return it != g_shape.end() && it->second == DP_LAUNCH_SHORT_CTAS;
}

}  // namespace dps

using namespace dps;

namespace {

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) != 0; }

int cuda_fail(int err, const char* where) {
  return fail(DP_ECUDA, std::string(where) + ": " +
                            cudaGetErrorString(static_cast<cudaError_t>(err)));
}

// Common checks; fills the launch descriptor for buckets [b0, b1).
int prepare(const char* fn, const dp_plan* plan, void* ws, int32_t b0, int32_t b1, void* stream,
            Launch* L) {
  clear_error();
  const Plan* pl = as_plan(plan);
  if (!pl) return fail(DP_EINVAL, std::string(fn) + ": NULL plan");
  if (!ws) return fail(DP_EINVAL, std::string(fn) + ": NULL workspace");
  if (misaligned(ws)) return fail(DP_EALIGN, std::string(fn) + ": workspace not 32-byte aligned");
  const int nb = static_cast<int>(pl->b_off.size());
  if (b0 < 0 || b1 < b0 || b1 > nb)
    return fail(DP_EINVAL, std::string(fn) + ": bucket range [" + std::to_string(b0) + ", " +
                               std::to_string(b1) + ") outside [0, " + std::to_string(nb) + ")");
  L->plan = pl;
  L->ws = static_cast<uint8_t*>(ws);
  L->tile_begin = pl->b_tile0[b0];
  L->tile_end = pl->b_tile0[b1];
  L->stream = stream;
  L->short_ctas = stream_short_ctas(stream);
  return DP_OK;
}

// NULL is accepted only for an empty plan (L == 0), where nothing is accessed.
int check_ptrs(const char* fn, const Plan* pl, std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs) {
    if (!p && pl->L > 0) return fail(DP_EINVAL, std::string(fn) + ": NULL device pointer");
    if (misaligned(p)) return fail(DP_EALIGN, std::string(fn) + ": device pointer not 32-byte aligned");
  }
  return DP_OK;
}

float* stage_of(const Plan* pl, void* ws) {
  DevHeader h;
  std::memcpy(&h, pl->image.data(), sizeof(h));
  return reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + h.off_stage);
}

// The clip coefficient an update multiplies the gradient by: the caller's device
// float (coef_dev), the workspace's last dp_clip_coef result (use_clip_coef), or
// none (NULL: 1).
int coef_source(const char* fn, void* ws, int32_t use_clip_coef, const float* coef_dev,
                const float** out) {
  *out = nullptr;
  if (coef_dev) {
    if (!use_clip_coef)
      return fail(DP_EINVAL, std::string(fn) + ": coef_dev given with use_clip_coef = 0");
    if (reinterpret_cast<uintptr_t>(coef_dev) & 3u)
      return fail(DP_EALIGN, std::string(fn) + ": coef_dev not 4-byte aligned");
    *out = coef_dev;
  } else if (use_clip_coef) {
    *out = reinterpret_cast<const float*>(static_cast<uint8_t*>(ws) + offsetof(DevHeader, coef));
  }
  return DP_OK;
}

int record(void* const* ev, int i, void* stream) {
  if (!ev) return DP_OK;
  const cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(ev[i]),
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "cudaEventRecord");
}

}  // namespace

extern "C" {

int dp_stream_set_launch(void* stream, int32_t shape) {
  clear_error();
  if (shape != DP_LAUNCH_DEFAULT && shape != DP_LAUNCH_SHORT_CTAS)
    return fail(DP_EINVAL, "dp_stream_set_launch: unknown launch shape " + std::to_string(shape));
  std::lock_guard<std::mutex> lock(g_shape_mu);
  try {
    if (shape == DP_LAUNCH_DEFAULT)
      g_shape.erase(stream);
    else
      g_shape[stream] = shape;
  } catch (const std::bad_alloc&) {
    return fail(DP_ENOMEM, "dp_stream_set_launch: out of host memory");
  }
  g_shape_count.store(static_cast<int>(g_shape.size()), std::memory_order_release);
  return DP_OK;
}

int dp_stream_get_launch(void* stream, int32_t* shape) {
  clear_error();
  if (!shape) return fail(DP_EINVAL, "dp_stream_get_launch: NULL shape");
  *shape = stream_short_ctas(stream) ? DP_LAUNCH_SHORT_CTAS : DP_LAUNCH_DEFAULT;
  return DP_OK;
}

int dp_plan_upload(const dp_plan* plan, void* workspace, void* stream) {
  clear_error();
  const Plan* pl = as_plan(plan);
  if (!pl || !workspace) return fail(DP_EINVAL, "dp_plan_upload: NULL argument");
  if (misaligned(workspace)) return fail(DP_EALIGN, "dp_plan_upload: workspace not 32-byte aligned");
  const cudaError_t e = cudaMemcpyAsync(workspace, pl->image.data(), pl->image.size(),
                                        cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "dp_plan_upload");
}

int dp_reduce_scatter_mean(const dp_plan* plan, void* workspace, const void* grads, float* mean,
                           int32_t b0, int32_t b1, int32_t want_sumsq, void* stream) {
  Launch L;
  int rc = prepare("dp_reduce_scatter_mean", plan, workspace, b0, b1, stream, &L);
  if (rc) return rc;
  if ((rc = check_ptrs("dp_reduce_scatter_mean", L.plan, {grads, mean}))) return rc;
  const int e = launch_reduce_scatter(L, grads, mean, want_sumsq != 0);
  return e ? cuda_fail(e, "dp_reduce_scatter_mean") : DP_OK;
}

int dp_clip_coef(const dp_plan* plan, void* workspace, double max_norm, int32_t b0, int32_t b1,
                 void* stream) {
  Launch L;
  const int rc = prepare("dp_clip_coef", plan, workspace, b0, b1, stream, &L);
  if (rc) return rc;
  const int e = launch_norm_finalize(L, max_norm);
  return e ? cuda_fail(e, "dp_clip_coef") : DP_OK;
}

int dp_sharded_adamw_step(const dp_plan* plan, void* workspace, const float* grad, float* master,
                          float* m, float* v, void* params, const dp_adamw_cfg* cfg,
                          int32_t use_clip_coef, const float* coef_dev, int32_t b0, int32_t b1,
                          void* stream) {
  Launch L;
  int rc = prepare("dp_sharded_adamw_step", plan, workspace, b0, b1, stream, &L);
  if (rc) return rc;
  if ((rc = check_ptrs("dp_sharded_adamw_step", L.plan, {grad, master, m, v, params}))) return rc;
  const float* coefp = nullptr;
  if ((rc = coef_source("dp_sharded_adamw_step", workspace, use_clip_coef, coef_dev, &coefp))) return rc;
  AdamScalars s{};
  if (cfg && (rc = adam_scalars("dp_sharded_adamw_step", cfg, &s))) return rc;
  const int e = launch_adamw(L, grad, master, m, v, params, s, coefp, false, !cfg);
  return e ? cuda_fail(e, "dp_sharded_adamw_step") : DP_OK;
}

int dp_all_gather(const dp_plan* plan, void* workspace, void* params, int32_t b0, int32_t b1,
                  void* stream) {
  Launch L;
  int rc = prepare("dp_all_gather", plan, workspace, b0, b1, stream, &L);
  if (rc) return rc;
  if ((rc = check_ptrs("dp_all_gather", L.plan, {params}))) return rc;
  const int e = launch_all_gather(L, params);
  return e ? cuda_fail(e, "dp_all_gather") : DP_OK;
}

int dp_broadcast(const dp_plan* plan, void* workspace, void* params, int32_t src, int32_t b0,
                 int32_t b1, void* stream) {
  Launch L;
  int rc = prepare("dp_broadcast", plan, workspace, b0, b1, stream, &L);
  if (rc) return rc;
  if ((rc = check_ptrs("dp_broadcast", L.plan, {params}))) return rc;
  if (src < 0 || src >= L.plan->P) return fail(DP_EINVAL, "dp_broadcast: src rank out of range");
  const int e = launch_broadcast(L, params, src);
  return e ? cuda_fail(e, "dp_broadcast") : DP_OK;
}

int dp_allreduce_mean(const dp_plan* plan, void* workspace, void* grads, int32_t b0, int32_t b1,
                      void* stream) {
  Launch L;
  int rc = prepare("dp_allreduce_mean", plan, workspace, b0, b1, stream, &L);
  if (rc) return rc;
  if ((rc = check_ptrs("dp_allreduce_mean", L.plan, {grads}))) return rc;
  const int e = launch_allreduce(L, grads);
  return e ? cuda_fail(e, "dp_allreduce_mean") : DP_OK;
}

int dp_adamw_all_gather(const dp_plan* plan, void* workspace, const float* mean, float* master,
                        float* m, float* v, void* params, const dp_adamw_cfg* cfg,
                        int32_t use_clip_coef, const float* coef_dev, void* stream) {
  Launch L;
  const Plan* pl = as_plan(plan);
  int rc = prepare("dp_adamw_all_gather", plan, workspace, 0,
                   pl ? static_cast<int32_t>(pl->b_off.size()) : 0, stream, &L);
  if (rc) return rc;
  if ((rc = check_ptrs("dp_adamw_all_gather", L.plan, {mean, master, m, v, params}))) return rc;
  const float* coefp = nullptr;
  if ((rc = coef_source("dp_adamw_all_gather", workspace, use_clip_coef, coef_dev, &coefp))) return rc;
  AdamScalars s{};
  if (cfg && (rc = adam_scalars("dp_adamw_all_gather", cfg, &s))) return rc;
  const int e = launch_adamw_all_gather(L, mean, params, master, m, v, s, coefp, !cfg);
  return e ? cuda_fail(e, "dp_adamw_all_gather") : DP_OK;
}

int dp_unit_all_gather(const dp_plan* plan, void* workspace, const void* param_shards, int32_t unit,
                       void* unit_buf, int64_t unit_stride, void* stream) {
  Launch L;
  int rc = prepare("dp_unit_all_gather", plan, workspace, unit, unit + 1, stream, &L);
  if (rc) return rc;
  if (unit < 0 || unit >= static_cast<int32_t>(L.plan->b_off.size()))
    return fail(DP_EINVAL, "dp_unit_all_gather: unit out of range");
  if (L.plan->b_len[unit] == 0) return DP_OK;   // an empty unit: nothing to gather
  if ((rc = check_ptrs("dp_unit_all_gather", L.plan, {param_shards, unit_buf}))) return rc;
  if (unit_stride < L.plan->b_len[unit] || unit_stride % 16)
    return fail(DP_EINVAL, "dp_unit_all_gather: unit_stride must be >= the unit length and a multiple of 16");
  const int e = launch_unit_all_gather(L, param_shards, unit_buf, unit_stride,
                                       L.plan->b_off[unit] / kPairElems);
  return e ? cuda_fail(e, "dp_unit_all_gather") : DP_OK;
}

int dp_unit_reduce_scatter(const dp_plan* plan, void* workspace, const void* unit_grads,
                           int64_t unit_stride, int32_t unit, float* mean, int32_t want_sumsq,
                           void* stream) {
  Launch L;
  int rc = prepare("dp_unit_reduce_scatter", plan, workspace, unit, unit + 1, stream, &L);
  if (rc) return rc;
  if (unit < 0 || unit >= static_cast<int32_t>(L.plan->b_off.size()))
    return fail(DP_EINVAL, "dp_unit_reduce_scatter: unit out of range");
  if (L.plan->b_len[unit] == 0) return DP_OK;   // an empty unit: no elements, no partials
  if ((rc = check_ptrs("dp_unit_reduce_scatter", L.plan, {unit_grads, mean}))) return rc;
  if (unit_stride < L.plan->b_len[unit] || unit_stride % 16)
    return fail(DP_EINVAL, "dp_unit_reduce_scatter: unit_stride must be >= the unit length and a multiple of 16");
  const int e = launch_reduce_scatter(L, unit_grads, mean, want_sumsq != 0, unit_stride,
                                      L.plan->b_off[unit] / kPairElems);
  return e ? cuda_fail(e, "dp_unit_reduce_scatter") : DP_OK;
}

int dp_unit_backward(const dp_plan* plan, void* workspace, const void* param_shards,
                     int32_t gather_unit, void* gather_buf, int64_t gather_stride,
                     const void* unit_grads, int64_t grads_stride, int32_t rs_unit, float* mean,
                     int32_t want_sumsq, void* stream) {
  const char* fn = "dp_unit_backward";
  const Plan* pl = as_plan(plan);
  const int32_t nb = pl ? static_cast<int32_t>(pl->b_off.size()) : 0;
  if (pl && (gather_unit < -1 || gather_unit >= nb || rs_unit < -1 || rs_unit >= nb)) {
    clear_error();
    return fail(DP_EINVAL, std::string(fn) + ": unit outside [-1, " + std::to_string(nb) + ")");
  }
  if (pl && gather_unit >= 0 && pl->b_len[gather_unit] == 0) gather_unit = -1;   // empty units:
  if (pl && rs_unit >= 0 && pl->b_len[rs_unit] == 0) rs_unit = -1;               // nothing to do
  if (gather_unit < 0 && rs_unit < 0) {
    Launch L;
    return prepare(fn, plan, workspace, 0, 0, stream, &L);
  }
  if (gather_unit < 0)
    return dp_unit_reduce_scatter(plan, workspace, unit_grads, grads_stride, rs_unit, mean,
                                  want_sumsq, stream);
  if (rs_unit < 0)
    return dp_unit_all_gather(plan, workspace, param_shards, gather_unit, gather_buf, gather_stride,
                              stream);
  Launch La, Lr;
  int rc = prepare(fn, plan, workspace, gather_unit, gather_unit + 1, stream, &La);
  if (rc) return rc;
  if ((rc = prepare(fn, plan, workspace, rs_unit, rs_unit + 1, stream, &Lr))) return rc;
  if ((rc = check_ptrs(fn, pl, {param_shards, gather_buf, unit_grads, mean}))) return rc;
  if (gather_stride < pl->b_len[gather_unit] || gather_stride % 16 || grads_stride < pl->b_len[rs_unit] ||
      grads_stride % 16)
    return fail(DP_EINVAL, std::string(fn) +
                               ": a stride is shorter than its unit or not a multiple of 16");
  // the gather's destination must not overlap what the reduce-scatter reads or writes
  const uintptr_t gb0 = reinterpret_cast<uintptr_t>(gather_buf);
  const uintptr_t gb1 = gb0 + 2 * static_cast<uintptr_t>(pl->P) * static_cast<uintptr_t>(gather_stride);
  const uintptr_t ug0 = reinterpret_cast<uintptr_t>(unit_grads);
  const uintptr_t ug1 = ug0 + 2 * static_cast<uintptr_t>(pl->P) * static_cast<uintptr_t>(grads_stride);
  const uintptr_t mn0 = reinterpret_cast<uintptr_t>(mean);
  const uintptr_t mn1 = mn0 + 4 * static_cast<uintptr_t>(pl->L);
  if ((gb0 < ug1 && ug0 < gb1) || (gb0 < mn1 && mn0 < gb1))
    return fail(DP_EINVAL, std::string(fn) + ": gather_buf overlaps unit_grads or mean");
  const int e = launch_unit_backward(Lr, unit_grads, mean, want_sumsq != 0, grads_stride,
                                     pl->b_off[rs_unit] / kPairElems, La, param_shards, gather_buf,
                                     gather_stride, pl->b_off[gather_unit] / kPairElems);
  return e ? cuda_fail(e, fn) : DP_OK;
}

int dp_shard_adamw_step(const dp_plan* plan, void* workspace, const float* mean, float* master,
                        float* m, float* v, void* param_shards, const dp_adamw_cfg* cfg,
                        int32_t use_clip_coef, const float* coef_dev, void* stream) {
  Launch L;
  const Plan* pl = as_plan(plan);
  int rc = prepare("dp_shard_adamw_step", plan, workspace, 0,
                   pl ? static_cast<int32_t>(pl->b_off.size()) : 0, stream, &L);
  if (rc) return rc;
  if ((rc = check_ptrs("dp_shard_adamw_step", L.plan, {mean, master, m, v, param_shards}))) return rc;
  const float* coefp = nullptr;
  if ((rc = coef_source("dp_shard_adamw_step", workspace, use_clip_coef, coef_dev, &coefp))) return rc;
  AdamScalars s{};
  if (cfg && (rc = adam_scalars("dp_shard_adamw_step", cfg, &s))) return rc;
  const int e = launch_adamw(L, mean, master, m, v, param_shards, s, coefp, true, !cfg);
  return e ? cuda_fail(e, "dp_shard_adamw_step") : DP_OK;
}

int dp_accumulate(const dp_plan* plan, void* workspace, void* acc, const void* micro, int32_t b0,
                  int32_t b1, void* stream) {
  Launch L;
  int rc = prepare("dp_accumulate", plan, workspace, b0, b1, stream, &L);
  if (rc) return rc;
  if ((rc = check_ptrs("dp_accumulate", L.plan, {acc, micro}))) return rc;
  const int e = launch_accumulate(L, acc, micro);
  return e ? cuda_fail(e, "dp_accumulate") : DP_OK;
}

int dp_allreduce_mean_accum(const dp_plan* plan, void* workspace, void* acc, const void* micro,
                            int32_t b0, int32_t b1, void* stream) {
  Launch L;
  int rc = prepare("dp_allreduce_mean_accum", plan, workspace, b0, b1, stream, &L);
  if (rc) return rc;
  if ((rc = check_ptrs("dp_allreduce_mean_accum", L.plan, {acc, micro}))) return rc;
  if (L.plan->R > 1) return fail(DP_EINVAL, "dp_allreduce_mean_accum: flat plans only");
  const int e = launch_allreduce_accum(L, acc, micro);
  return e ? cuda_fail(e, "dp_allreduce_mean_accum") : DP_OK;
}

int dp_reduce_scatter_mean_accum(const dp_plan* plan, void* workspace, const void* acc,
                                 const void* micro, float* mean, int32_t b0, int32_t b1,
                                 int32_t want_sumsq, void* stream) {
  Launch L;
  int rc = prepare("dp_reduce_scatter_mean_accum", plan, workspace, b0, b1, stream, &L);
  if (rc) return rc;
  if ((rc = check_ptrs("dp_reduce_scatter_mean_accum", L.plan, {acc, micro, mean}))) return rc;
  if (L.plan->R > 1) return fail(DP_EINVAL, "dp_reduce_scatter_mean_accum: flat plans only");
  const int e = launch_reduce_scatter_accum(L, acc, micro, mean, want_sumsq != 0);
  return e ? cuda_fail(e, "dp_reduce_scatter_mean_accum") : DP_OK;
}

int dp_allreduce_mean_bf16wire(const dp_plan* plan, void* workspace, void* grads, int32_t b0,
                               int32_t b1, void* stream) {
  Launch L;
  int rc = prepare("dp_allreduce_mean_bf16wire", plan, workspace, b0, b1, stream, &L);
  if (rc) return rc;
  if ((rc = check_ptrs("dp_allreduce_mean_bf16wire", L.plan, {grads}))) return rc;
  if (L.plan->R > 1) return fail(DP_EINVAL, "dp_allreduce_mean_bf16wire: flat plans only");
  const int e = launch_allreduce_bf16wire(L, grads);
  return e ? cuda_fail(e, "dp_allreduce_mean_bf16wire") : DP_OK;
}

int dp_selftest_bounded_wait(int32_t* status_dev, int64_t limit_ns, void* stream) {
  clear_error();
  if (!status_dev) return fail(DP_EINVAL, "dp_selftest_bounded_wait: NULL status");
  if (reinterpret_cast<uintptr_t>(status_dev) & 7u)
    return fail(DP_EALIGN, "dp_selftest_bounded_wait: status must be 8-byte aligned");
  if (limit_ns < 1000 || limit_ns > 10000000000LL)
    return fail(DP_EINVAL, "dp_selftest_bounded_wait: limit_ns outside [1e3, 1e10]");
  const int e = launch_selftest_wait(status_dev, static_cast<uint64_t>(limit_ns), stream);
  return e ? cuda_fail(e, "dp_selftest_bounded_wait") : DP_OK;
}

int64_t dp_bounds_violations(int32_t reset) {
  clear_error();
  const int64_t a = bounds_violations_reduce(reset != 0);
  const int64_t b = bounds_violations_update(reset != 0);
  if (a == -1 && b == -1) return -1;
  if (a < 0 || b < 0) return -2;
  return a + b;
}

int dp_set_adamw_cfg(const dp_plan* plan, void* workspace, const dp_adamw_cfg* cfg, void* stream) {
  clear_error();
  const Plan* pl = as_plan(plan);
  if (!pl || !workspace) return fail(DP_EINVAL, "dp_set_adamw_cfg: NULL plan or workspace");
  if (misaligned(workspace)) return fail(DP_EALIGN, "dp_set_adamw_cfg: workspace not 32-byte aligned");
  struct {
    AdamScalars s;
    uint32_t tag;
  } blob{};
  int rc = adam_scalars("dp_set_adamw_cfg", cfg, &blob.s);
  if (rc) return rc;
  blob.tag = kAdamTag;
  static_assert(offsetof(DevHeader, adam_tag) == offsetof(DevHeader, adam) + sizeof(AdamScalars),
                "scalars and tag are adjacent");
  const cudaError_t e = cudaMemcpyAsync(static_cast<uint8_t*>(workspace) + offsetof(DevHeader, adam),
                                        &blob, sizeof(AdamScalars) + sizeof(uint32_t),
                                        cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DP_OK : cuda_fail(e, "dp_set_adamw_cfg");
}

int dp_workspace_result_offsets(int64_t* offsets) {
  clear_error();
  if (!offsets) return fail(DP_EINVAL, "dp_workspace_result_offsets: NULL offsets");
  offsets[0] = static_cast<int64_t>(offsetof(DevHeader, norm2));
  offsets[1] = static_cast<int64_t>(offsetof(DevHeader, norm));
  offsets[2] = static_cast<int64_t>(offsetof(DevHeader, coef));
  offsets[3] = static_cast<int64_t>(offsetof(DevHeader, status));
  return DP_OK;
}

int dp_fused_zero_step_launches(const dp_adamw_cfg* cfg) {
  return (cfg && cfg->max_norm > 0.0) ? 3 : 1;
}

int dp_fused_zero_step(const dp_plan* plan, void* workspace, const void* grads, void* params,
                       float* master, float* m, float* v, const dp_adamw_cfg* cfg,
                       void* const* stage_events, void* stream) {
  Launch L;
  const Plan* pl = as_plan(plan);
  int rc = prepare("dp_fused_zero_step", plan, workspace, 0,
                   pl ? static_cast<int32_t>(pl->b_off.size()) : 0, stream, &L);
  if (rc) return rc;
  if ((rc = check_ptrs("dp_fused_zero_step", L.plan, {grads, params, master, m, v}))) return rc;
  AdamScalars s;
  if ((rc = adam_scalars("dp_fused_zero_step", cfg, &s))) return rc;
  if ((rc = record(stage_events, 0, stream))) return rc;
  if (!(cfg->max_norm > 0.0)) {
    const int e = launch_zero_fused(L, grads, params, master, m, v, s);
    if (e) return cuda_fail(e, "dp_fused_zero_step");
    return record(stage_events, 1, stream);
  }
  float* stage = stage_of(pl, workspace);
  int e = launch_reduce_scatter(L, grads, stage, true);
  if (e) return cuda_fail(e, "dp_fused_zero_step (reduce-scatter)");
  if ((rc = record(stage_events, 1, stream))) return rc;
  e = launch_norm_finalize(L, cfg->max_norm);
  if (e) return cuda_fail(e, "dp_fused_zero_step (norm)");
  if ((rc = record(stage_events, 2, stream))) return rc;
  const float* ws_coef = reinterpret_cast<const float*>(static_cast<uint8_t*>(workspace) +
                                                        offsetof(DevHeader, coef));
  e = launch_adamw_all_gather(L, stage, params, master, m, v, s, ws_coef);
  if (e) return cuda_fail(e, "dp_fused_zero_step (adamw + all-gather)");
  return record(stage_events, 3, stream);
}

int dp_read_norm(const dp_plan* plan, const void* workspace, double* norm, float* coef,
                 int32_t* status, void* stream) {
  clear_error();
  if (!plan || !workspace) return fail(DP_EINVAL, "dp_read_norm: NULL argument");
  DevHeader h;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess)
    e = cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "dp_read_norm");
  if (norm) *norm = h.norm;
  if (coef) *coef = h.coef;
  if (status) *status = h.status;
  if (h.status & DP_STATUS_PLAN_MISMATCH)
    return fail(DP_EPLAN, "dp_read_norm: a kernel found another plan's image in the workspace");
  if (h.status & DP_STATUS_TIMEOUT)
    return fail(DP_ETIMEOUT, "dp_read_norm: a kernel's bounded wait on its copies gave up");
  if (h.status & DP_STATUS_NONFINITE)
    return fail(DP_ENONFINITE, "dp_read_norm: the global gradient norm was not finite");
  if (h.status & DP_STATUS_NO_SCALARS)
    return fail(DP_EINVAL, "dp_read_norm: an update ran with cfg = NULL before dp_set_adamw_cfg");
  return DP_OK;
}

}  // extern "C"

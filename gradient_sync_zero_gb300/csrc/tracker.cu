// Bucket readiness tracker: streamed per-bucket synchronisation.
// With a micro-batch buffer set (dp_tracker_set_micro), each bucket's launch is the
// last micro-batch of gradient accumulation fused with its sync: every rank's
// bf16(grads + micro) is reduced ("Distributed Training: Data Parallel, Model
// Parallel and FSDP Strategies", "Selecting and Tuning": no_sync on the other
// micro-batches, sync on the final one, bucket by bucket as backward proceeds).
//
// DDP's core mechanism ("4.1 Data parallelism in depth", sec. 4.2): backward
// produces gradients last layer first; a bucket's collective fires as soon as
// every gradient in it is ready, on a separate stream ("Distributed Training:
// Data Parallel, Model Parallel and FSDP Strategies", "Inside DDP"), while the
// earlier layers keep computing.  Buckets fire in plan order, the same order
// every step, as DDP requires of all ranks ("Data Parallelism: DDP, ZeRO and
// FSDP", "DDP, and why it works").  Where DDP hangs on a gradient that never
// becomes ready (find_unused_parameters, sec. 4.2 note), the tracker's wait
// times out and names the missing tensors.
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <condition_variable>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "internal.h"

namespace dps {

struct Tracker {
  const Plan* plan = nullptr;
  int mode = DP_TRACK_ALLREDUCE;
  int flags = 0;
  uint8_t* ws = nullptr;
  void* grads = nullptr;
  const void* micro = nullptr;      // set: the last micro-batch of accumulation (fused add)
  float* mean = nullptr;
  void* stream = nullptr;
  // DP_TRACK_ZERO_STEP: the step's targets and AdamW scalars (dp_tracker_set_zero_step)
  void* params = nullptr;
  float* master = nullptr;
  float* m = nullptr;
  float* v = nullptr;
  AdamScalars adam{};
  bool zero_set = false;
  int max_ctas = 0;
  std::vector<std::vector<int32_t>> bucket_tensors;
  std::mutex mu;
  std::condition_variable cv;
  std::vector<uint8_t> ready;
  std::vector<void*> events;
  std::vector<int32_t> pending;     // per bucket: tensors not yet marked
  int32_t next = 0;                 // next bucket to fire, in plan order
  std::vector<int32_t> fired;
  void* side = nullptr;             // set: every bucket but the last fires here (dp_tracker_set_side_stream)
  int side_ctas = 0;
  cudaEvent_t side_done = nullptr;  // recorded on `side` before the last bucket fires on `stream`
  int32_t launches = 0;             // this step: kernel launches (a launch covers a bucket range)
  int32_t waits = 0;                // this step: cudaStreamWaitEvent calls
  std::vector<void*> wait_list;     // scratch: distinct events of the range being fired
  int error = DP_OK;                // sticky launch error of this step
  std::string error_text;
};

namespace {

void reset(Tracker& tr) {
  const Plan& pl = *tr.plan;
  std::fill(tr.ready.begin(), tr.ready.end(), 0);
  std::fill(tr.events.begin(), tr.events.end(), nullptr);
  for (size_t b = 0; b < tr.bucket_tensors.size(); ++b)
    tr.pending[b] = static_cast<int32_t>(tr.bucket_tensors[b].size());
  tr.next = 0;
  tr.fired.clear();
  tr.launches = 0;
  tr.waits = 0;
  tr.error = DP_OK;
  tr.error_text.clear();
  (void)pl;
}

// Launch buckets [b0, b1) on `stream` as one launch over their tiles, grid
// capped at max_ctas (lock held), after the stream has waited once for each
// distinct event of their tensors.  One launch over consecutive buckets computes
// what per-bucket launches would, tile by tile (the norm partials are per
// sub-tile).  With DP_TRACK_SHORT_CTAS each bucket is its own launch of
// short-lived CTAs (the single-bucket kernels), max_ctas ignored.
int fire_on(Tracker& tr, int32_t b0, int32_t b1, void* stream, int max_ctas);

// With a side stream, buckets before the plan's last fire there; the last bucket
// (ready only when backward ends) fires on the tracker's stream after that stream
// has waited for the side stream's work, so every reduction is ordered before
// the tracker's stream.
int fire(Tracker& tr, int32_t b0, int32_t b1) {
  const int32_t nb = static_cast<int32_t>(tr.pending.size());
  if (!tr.side || (tr.flags & DP_TRACK_DRY_RUN)) return fire_on(tr, b0, b1, tr.stream, tr.max_ctas);
  const int32_t mid = b1 == nb ? nb - 1 : b1;   // [b0, mid) on the side stream
  if (mid > b0) {
    const int rc = fire_on(tr, b0, mid, tr.side, tr.side_ctas);
    if (rc) return rc;
  }
  if (b1 < nb) return DP_OK;
  cudaError_t e = cudaEventRecord(tr.side_done, static_cast<cudaStream_t>(tr.side));
  if (e == cudaSuccess) e = cudaStreamWaitEvent(static_cast<cudaStream_t>(tr.stream), tr.side_done, 0);
  if (e != cudaSuccess) {
    tr.error_text = std::string("dp_tracker: ordering after the side stream: ") + cudaGetErrorString(e);
    return DP_ECUDA;
  }
  return fire_on(tr, nb - 1, nb, tr.stream, tr.max_ctas);
}

int fire_on(Tracker& tr, int32_t b0, int32_t b1, void* stream, int max_ctas) {
  for (int32_t b = b0; b < b1; ++b) tr.fired.push_back(b);
  tr.wait_list.clear();
  for (int32_t b = b0; b < b1; ++b)
    for (int32_t t : tr.bucket_tensors[b]) {
      void* ev = tr.events[t];
      if (ev && std::find(tr.wait_list.begin(), tr.wait_list.end(), ev) == tr.wait_list.end())
        tr.wait_list.push_back(ev);
    }
  const bool short_ctas = (tr.flags & DP_TRACK_SHORT_CTAS) != 0 || stream_short_ctas(stream);
  if (tr.flags & DP_TRACK_DRY_RUN) {   // count what would be issued
    tr.waits += static_cast<int32_t>(tr.wait_list.size());
    tr.launches += short_ctas ? b1 - b0 : 1;
    return DP_OK;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (void* ev : tr.wait_list) {
    const cudaError_t e = cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(ev), 0);
    if (e != cudaSuccess) {
      tr.error_text = std::string("dp_tracker: cudaStreamWaitEvent: ") + cudaGetErrorString(e);
      return DP_ECUDA;
    }
    ++tr.waits;
  }
  if (tr.mode == DP_TRACK_ZERO_STEP && !tr.zero_set) {
    tr.error_text = "dp_tracker: bucket " + std::to_string(b0) +
                    " became ready before dp_tracker_set_zero_step";
    return DP_EINVAL;
  }
  for (int32_t lb = b0; lb < b1;) {
    const int32_t le = short_ctas ? lb + 1 : b1;
    Launch L;
    L.plan = tr.plan;
    L.ws = tr.ws;
    L.tile_begin = tr.plan->b_tile0[lb];
    L.tile_end = tr.plan->b_tile0[le];
    L.stream = stream;
    L.max_ctas = max_ctas;
    L.short_ctas = short_ctas;
    int e;
    if (tr.mode == DP_TRACK_ZERO_STEP)
      e = launch_zero_fused(L, tr.grads, tr.params, tr.master, tr.m, tr.v, tr.adam);
    else if (tr.mode == DP_TRACK_ALLREDUCE)
      e = tr.micro ? launch_allreduce_accum(L, tr.grads, tr.micro) : launch_allreduce(L, tr.grads);
    else
      e = tr.micro ? launch_reduce_scatter_accum(L, tr.grads, tr.micro, tr.mean, true)
                   : launch_reduce_scatter(L, tr.grads, tr.mean, true);
    if (e) {
      tr.error_text = std::string("dp_tracker: bucket launch: ") +
                      cudaGetErrorString(static_cast<cudaError_t>(e));
      return DP_ECUDA;
    }
    ++tr.launches;
    lb = le;
  }
  return DP_OK;
}

// The single event every tensor of bucket b was marked with (NULL included), or
// uniform = false when its tensors carry different events.
void* bucket_event(const Tracker& tr, int32_t b, bool* uniform) {
  const std::vector<int32_t>& ts = tr.bucket_tensors[b];
  void* ev = ts.empty() ? nullptr : tr.events[ts[0]];
  *uniform = true;
  for (int32_t t : ts)
    if (tr.events[t] != ev) {
      *uniform = false;
      break;
    }
  return ev;
}

// Fire the buckets that have become complete, from tr.next on, in plan order.
// Consecutive complete buckets whose tensors were all marked with the same event
// (one layer marked with one event, or no events) become ready at the same moment
// on the GPU and go out as one launch; a bucket whose tensors carry different
// events goes out alone, right after the last of them, so it never waits for a
// later bucket's readiness.
int fire_ready(Tracker& tr) {
  const int32_t nb = static_cast<int32_t>(tr.pending.size());
  while (tr.next < nb && tr.pending[tr.next] == 0) {
    bool uniform = false;
    void* ev = bucket_event(tr, tr.next, &uniform);
    int32_t end = tr.next + 1;
    if (uniform) {
      while (end < nb && tr.pending[end] == 0) {
        bool u2 = false;
        if (bucket_event(tr, end, &u2) != ev || !u2) break;
        ++end;
      }
    }
    const int rc = fire(tr, tr.next, end);
    if (rc) return rc;
    tr.next = end;
  }
  return DP_OK;
}

// Mark n tensors ready — tensor_at(i), written before event_at(i) — and fire what
// became complete (lock held).  Nothing is marked if any tensor is out of range,
// already marked in this step, or listed twice.
template <class T, class E>
int mark_tensors(Tracker& tr, int32_t n, T tensor_at, E event_at, const char* fn, std::string* text,
                 bool* done) {
  const int32_t nt = static_cast<int32_t>(tr.ready.size());
  for (int32_t i = 0; i < n; ++i) {
    const int32_t t = tensor_at(i);
    std::string why;
    if (t < 0 || t >= nt)
      why = " outside [0, " + std::to_string(nt) + ")";
    else if (tr.ready[t] == 2)
      why = " listed twice";
    else if (tr.ready[t])
      why = " already marked in this step";
    if (!why.empty()) {
      *text = std::string(fn) + ": tensor " + std::to_string(t) + why;
      for (int32_t j = 0; j < i; ++j) tr.ready[tensor_at(j)] = 0;   // undo this call's marks
      return DP_EINVAL;
    }
    tr.ready[t] = 2;   // taken by this call (a repeat in the list is refused above)
  }
  for (int32_t i = 0; i < n; ++i) {
    const int32_t t = tensor_at(i);
    tr.ready[t] = 1;
    tr.events[t] = event_at(i);
    --tr.pending[tr.plan->t_bucket[t]];
  }
  int rc = DP_OK;
  if (tr.error == DP_OK) {
    rc = fire_ready(tr);
    if (rc) {
      tr.error = rc;
      *text = tr.error_text;
    }
  }
  *done = tr.next == static_cast<int32_t>(tr.pending.size()) || tr.error != DP_OK;
  return rc;
}

}  // namespace
}  // namespace dps

using namespace dps;

extern "C" {

int dp_tracker_create(const dp_plan* plan, int32_t mode, void* workspace, void* grads, float* mean,
                      void* comm_stream, int32_t max_ctas, int32_t flags, dp_tracker** out) {
  clear_error();
  if (!out) return fail(DP_EINVAL, "dp_tracker_create: out is NULL");
  *out = nullptr;
  const Plan* pl = as_plan(plan);
  if (!pl) return fail(DP_EINVAL, "dp_tracker_create: NULL plan");
  if (mode != DP_TRACK_ALLREDUCE && mode != DP_TRACK_REDUCE_SCATTER && mode != DP_TRACK_ZERO_STEP)
    return fail(DP_EINVAL, "dp_tracker_create: unknown mode");
  if (max_ctas < 0) return fail(DP_EINVAL, "dp_tracker_create: max_ctas must be >= 0");
  if (flags & ~(DP_TRACK_DRY_RUN | DP_TRACK_SHORT_CTAS))
    return fail(DP_EINVAL, "dp_tracker_create: unknown flags " + std::to_string(flags));
  const bool dry = (flags & DP_TRACK_DRY_RUN) != 0;
  if (!dry) {
    if (!workspace || (pl->L > 0 && (!grads || (mode == DP_TRACK_REDUCE_SCATTER && !mean))))
      return fail(DP_EINVAL, "dp_tracker_create: NULL workspace, grads or mean");
    const uintptr_t a = reinterpret_cast<uintptr_t>(workspace) | reinterpret_cast<uintptr_t>(grads) |
                        reinterpret_cast<uintptr_t>(mean);
    if (a & 31u) return fail(DP_EALIGN, "dp_tracker_create: device pointers must be 32-byte aligned");
  }
  Tracker* tr = new (std::nothrow) Tracker();
  if (!tr) return fail(DP_ENOMEM, "dp_tracker_create: out of host memory");
  try {
    tr->plan = pl;
    tr->mode = mode;
    tr->flags = flags;
    tr->ws = static_cast<uint8_t*>(workspace);
    tr->grads = grads;
    tr->mean = mean;
    tr->stream = comm_stream;
    tr->max_ctas = max_ctas;
    const size_t nb = pl->b_off.size(), nt = pl->sizes.size();
    tr->bucket_tensors.assign(nb, {});
    for (size_t t = 0; t < nt; ++t) tr->bucket_tensors[pl->t_bucket[t]].push_back(static_cast<int32_t>(t));
    tr->ready.assign(nt, 0);
    tr->events.assign(nt, nullptr);
    tr->pending.assign(nb, 0);
    reset(*tr);
  } catch (const std::bad_alloc&) {
    delete tr;
    return fail(DP_ENOMEM, "dp_tracker_create: out of host memory");
  }
  *out = reinterpret_cast<dp_tracker*>(tr);
  return DP_OK;
}

int dp_tracker_set_micro(dp_tracker* tracker, const void* micro) {
  clear_error();
  Tracker* tr = reinterpret_cast<Tracker*>(tracker);
  if (!tr) return fail(DP_EINVAL, "dp_tracker_set_micro: NULL tracker");
  if (micro && tr->plan->R > 1) return fail(DP_EINVAL, "dp_tracker_set_micro: flat plans only");
  if (micro && tr->mode == DP_TRACK_ZERO_STEP)
    return fail(DP_EINVAL, "dp_tracker_set_micro: not with DP_TRACK_ZERO_STEP");
  if (reinterpret_cast<uintptr_t>(micro) & 31u)
    return fail(DP_EALIGN, "dp_tracker_set_micro: micro must be 32-byte aligned");
  std::lock_guard<std::mutex> g(tr->mu);
  if (tr->next != 0 && tr->next != static_cast<int32_t>(tr->pending.size()))
    return fail(DP_EINVAL, "dp_tracker_set_micro: a step is in progress (some buckets fired)");
  tr->micro = micro;
  return DP_OK;
}

int dp_tracker_set_zero_step(dp_tracker* tracker, void* params, float* master, float* m, float* v,
                             const dp_adamw_cfg* cfg) {
  clear_error();
  Tracker* tr = reinterpret_cast<Tracker*>(tracker);
  if (!tr) return fail(DP_EINVAL, "dp_tracker_set_zero_step: NULL tracker");
  if (tr->mode != DP_TRACK_ZERO_STEP)
    return fail(DP_EINVAL, "dp_tracker_set_zero_step: the tracker is not in DP_TRACK_ZERO_STEP mode");
  if (tr->micro) return fail(DP_EINVAL, "dp_tracker_set_zero_step: a micro-batch buffer is set");
  if (tr->plan->L > 0 && (!params || !master || !m || !v))
    return fail(DP_EINVAL, "dp_tracker_set_zero_step: NULL device pointer");
  const uintptr_t a = reinterpret_cast<uintptr_t>(params) | reinterpret_cast<uintptr_t>(master) |
                      reinterpret_cast<uintptr_t>(m) | reinterpret_cast<uintptr_t>(v);
  if (a & 31u) return fail(DP_EALIGN, "dp_tracker_set_zero_step: device pointers must be 32-byte aligned");
  AdamScalars s{};
  const int rc = adam_scalars("dp_tracker_set_zero_step", cfg, &s);
  if (rc) return rc;
  if (cfg->max_norm > 0.0)
    return fail(DP_EINVAL, "dp_tracker_set_zero_step: clipping needs the global norm of every "
                           "bucket before any update; use DP_TRACK_REDUCE_SCATTER");
  std::lock_guard<std::mutex> g(tr->mu);
  if (tr->next != 0 && tr->next != static_cast<int32_t>(tr->pending.size()))
    return fail(DP_EINVAL, "dp_tracker_set_zero_step: a step is in progress (some buckets fired)");
  tr->params = params;
  tr->master = master;
  tr->m = m;
  tr->v = v;
  tr->adam = s;
  tr->zero_set = true;
  return DP_OK;
}

int dp_tracker_set_side_stream(dp_tracker* tracker, void* side_stream, int32_t side_ctas) {
  clear_error();
  Tracker* tr = reinterpret_cast<Tracker*>(tracker);
  if (!tr) return fail(DP_EINVAL, "dp_tracker_set_side_stream: NULL tracker");
  if (side_ctas < 0) return fail(DP_EINVAL, "dp_tracker_set_side_stream: side_ctas must be >= 0");
  std::lock_guard<std::mutex> g(tr->mu);
  if (tr->next != 0 && tr->next != static_cast<int32_t>(tr->pending.size()))
    return fail(DP_EINVAL, "dp_tracker_set_side_stream: a step is in progress (some buckets fired)");
  if (side_stream && !tr->side_done && !(tr->flags & DP_TRACK_DRY_RUN)) {
    const cudaError_t e = cudaEventCreateWithFlags(&tr->side_done, cudaEventDisableTiming);
    if (e != cudaSuccess)
      return fail(DP_ECUDA, std::string("dp_tracker_set_side_stream: ") + cudaGetErrorString(e));
  }
  tr->side = side_stream;
  tr->side_ctas = side_ctas;
  return DP_OK;
}

int dp_tracker_begin(dp_tracker* tracker) {
  clear_error();
  Tracker* tr = reinterpret_cast<Tracker*>(tracker);
  if (!tr) return fail(DP_EINVAL, "dp_tracker_begin: NULL tracker");
  std::lock_guard<std::mutex> g(tr->mu);
  reset(*tr);
  return DP_OK;
}

int dp_tracker_mark_ready(dp_tracker* tracker, int32_t tensor, void* ready_event) {
  clear_error();
  Tracker* tr = reinterpret_cast<Tracker*>(tracker);
  if (!tr) return fail(DP_EINVAL, "dp_tracker_mark_ready: NULL tracker");
  std::string text;
  bool done = false;
  std::unique_lock<std::mutex> g(tr->mu);
  const int rc = mark_tensors(
      *tr, 1, [&](int32_t) { return tensor; }, [&](int32_t) { return ready_event; },
      "dp_tracker_mark_ready", &text, &done);
  g.unlock();
  if (done) tr->cv.notify_all();
  return rc ? fail(rc, text) : DP_OK;
}

int dp_tracker_mark_ready_range(dp_tracker* tracker, int32_t t0, int32_t t1, void* ready_event) {
  clear_error();
  Tracker* tr = reinterpret_cast<Tracker*>(tracker);
  if (!tr) return fail(DP_EINVAL, "dp_tracker_mark_ready_range: NULL tracker");
  if (t1 < t0)
    return fail(DP_EINVAL, "dp_tracker_mark_ready_range: empty range [" + std::to_string(t0) +
                               ", " + std::to_string(t1) + ")");
  std::string text;
  bool done = false;
  std::unique_lock<std::mutex> g(tr->mu);
  const int rc = mark_tensors(
      *tr, t1 - t0, [&](int32_t i) { return t0 + i; }, [&](int32_t) { return ready_event; },
      "dp_tracker_mark_ready_range", &text, &done);
  g.unlock();
  if (done) tr->cv.notify_all();
  return rc ? fail(rc, text) : DP_OK;
}

int dp_tracker_mark_ready_batch(dp_tracker* tracker, const int32_t* tensors,
                                void* const* ready_events, int32_t n) {
  clear_error();
  Tracker* tr = reinterpret_cast<Tracker*>(tracker);
  if (!tr) return fail(DP_EINVAL, "dp_tracker_mark_ready_batch: NULL tracker");
  if (n < 0 || (n > 0 && !tensors))
    return fail(DP_EINVAL, "dp_tracker_mark_ready_batch: n < 0 or NULL tensors");
  std::string text;
  bool done = false;
  std::unique_lock<std::mutex> g(tr->mu);
  const int rc = mark_tensors(
      *tr, n, [&](int32_t i) { return tensors[i]; },
      [&](int32_t i) { return ready_events ? ready_events[i] : nullptr; },
      "dp_tracker_mark_ready_batch", &text, &done);
  g.unlock();
  if (done) tr->cv.notify_all();
  return rc ? fail(rc, text) : DP_OK;
}

int dp_tracker_stats(const dp_tracker* tracker, int32_t* launches, int32_t* waits) {
  clear_error();
  Tracker* tr = const_cast<Tracker*>(reinterpret_cast<const Tracker*>(tracker));
  if (!tr) return fail(DP_EINVAL, "dp_tracker_stats: NULL tracker");
  std::lock_guard<std::mutex> g(tr->mu);
  if (launches) *launches = tr->launches;
  if (waits) *waits = tr->waits;
  return DP_OK;
}

int dp_tracker_wait(dp_tracker* tracker, int64_t timeout_ms) {
  clear_error();
  Tracker* tr = reinterpret_cast<Tracker*>(tracker);
  if (!tr) return fail(DP_EINVAL, "dp_tracker_wait: NULL tracker");
  std::unique_lock<std::mutex> g(tr->mu);
  const int32_t nb = static_cast<int32_t>(tr->pending.size());
  const bool ok = tr->cv.wait_for(g, std::chrono::milliseconds(std::max<int64_t>(timeout_ms, 0)),
                                  [&] { return tr->next == nb || tr->error != DP_OK; });
  if (tr->error != DP_OK) return fail(tr->error, tr->error_text);
  if (ok) return DP_OK;
  std::string missing;
  int count = 0;
  for (size_t t = 0; t < tr->ready.size(); ++t) {
    if (tr->ready[t]) continue;
    if (count < 16) missing += (count ? ", " : "") + std::to_string(t);
    ++count;
  }
  return fail(DP_ETIMEOUT, "dp_tracker_wait: " + std::to_string(count) +
                               " tensor(s) never marked ready: " + missing +
                               (count > 16 ? ", ..." : "") + "; bucket " +
                               std::to_string(tr->next) + " of " + std::to_string(nb) +
                               " is the first not launched");
}

int dp_tracker_fired(const dp_tracker* tracker, int32_t* order, int32_t cap, int32_t* n_fired) {
  clear_error();
  Tracker* tr = const_cast<Tracker*>(reinterpret_cast<const Tracker*>(tracker));
  if (!tr || cap < 0 || (cap > 0 && !order)) return fail(DP_EINVAL, "dp_tracker_fired: bad arguments");
  std::lock_guard<std::mutex> g(tr->mu);
  const int32_t n = static_cast<int32_t>(tr->fired.size());
  for (int32_t i = 0; i < std::min(n, cap); ++i) order[i] = tr->fired[i];
  if (n_fired) *n_fired = n;
  return DP_OK;
}

void dp_tracker_free(dp_tracker* tracker) {
  Tracker* tr = reinterpret_cast<Tracker*>(tracker);
  if (tr && tr->side_done) cudaEventDestroy(tr->side_done);
  delete tr;
}

}  // extern "C"

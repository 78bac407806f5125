// Host-side launch helpers shared by the kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include <climits>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <type_traits>
#include <utility>

#include "kernels.cuh"

namespace dps {

inline KCommon make_common(const Launch& L) {
  DevHeader h;
  std::memcpy(&h, L.plan->image.data(), sizeof(h));
  KCommon k;
  k.hdr = reinterpret_cast<DevHeader*>(L.ws);
  k.tiles = reinterpret_cast<const TileDesc*>(L.ws + h.off_tiles);
  k.decay = reinterpret_cast<const uint32_t*>(L.ws + h.off_decay);
  k.sumsq = reinterpret_cast<float*>(L.ws + h.off_sumsq);
  k.fin = reinterpret_cast<float*>(L.ws + h.off_fin);
  k.plan_id = L.plan->id;
  k.stride_bytes = L.plan->stride * 2;
  k.tile_begin = L.tile_begin;
  k.tile_end = L.tile_end;
  k.P = L.plan->P;
  k.R = L.plan->R;
  k.S = L.plan->S;
  k.rep_block0 = 0;
  k.split = 1;
  k.pad_ = 0;
  k.one_v0 = 0;
  k.one_tile0 = 0;
  k.one_nvec = 0;
  k.one_svec = 0;
  k.one_bucket = 0;
  k.pad2_ = 0;
  // a launch inside one bucket carries the bucket (tile descriptors computed)
  if (L.tile_end > L.tile_begin) {
    const TileDesc& a = L.plan->tiles[L.tile_begin];
    const int b = a.bucket;
    if (L.plan->b_tile0[b] <= L.tile_begin && L.tile_end <= L.plan->b_tile0[b + 1] &&
        L.plan->b_len[b] / kVecElems <= INT32_MAX) {
      k.one_v0 = a.bvoff;
      k.one_tile0 = L.plan->b_tile0[b];
      k.one_nvec = static_cast<int32_t>(L.plan->b_len[b] / kVecElems);
      k.one_svec = a.svec;
      k.one_bucket = b;
    }
  }
  return k;
}

inline float* stage_ptr(const Launch& L) {
  DevHeader h;
  std::memcpy(&h, L.plan->image.data(), sizeof(h));
  return reinterpret_cast<float*>(L.ws + h.off_stage);
}

// Opt a kernel in to `bytes` of dynamic shared memory, once per device (so that
// launches inside a CUDA graph capture make no attribute call).
template <class K>
cudaError_t ensure_dyn_smem(K kernel, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
  std::lock_guard<std::mutex> g(mu);
  auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) done[key] = bytes;
  return e;
}

// Resident CTAs per SM for a kernel (occupancy calculator, cached per device),
// optionally capped by DPSYNC_CTAS_PER_SM for tuning sweeps.
template <class K>
int resident_ctas(K kernel, int threads, size_t dyn_smem = 0) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, dyn_smem) !=
      cudaSuccess)
    return 0;
  if (const char* e = std::getenv("DPSYNC_CTAS_PER_SM")) {
    const int cap = std::atoi(e);
    if (cap > 0 && cap < per_sm) per_sm = cap;
  }
  const int n = sms * (per_sm > 0 ? per_sm : 1);
  std::lock_guard<std::mutex> g(mu);
  cache[key] = n;
  return n;
}

// Programmatic dependent launch (on unless DPSYNC_PDL=0): a kernel's CTAs may be
// scheduled while the previous kernel in the stream drains; each kernel waits
// for that kernel's completion (griddepcontrol.wait in plan_ok) before its first
// global access, so stream order and visibility are as for plain launches.
inline bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("DPSYNC_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

// Launch through cudaLaunchKernelEx with the programmatic-serialisation
// attribute; returns the launch's error (and clears the thread's last error).
template <class K, class... A>
int launch_k(K kernel, int grid, int threads, size_t smem, void* stream, A... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  const cudaError_t last = cudaGetLastError();
  return static_cast<int>(e != cudaSuccess ? e : last);
}

// Launch `kernel` over the tiles of L with a persistent grid.
inline int sm_count() {
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> g(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cache[dev] = sms;
  return sms;
}

// Persistent grid over the launch's tiles: at most the resident CTAs, or
// per_sm CTAs per SM when given (some read/write mixes run faster with fewer
// loads in flight than full occupancy keeps).
template <class K, class... A>
int launch_tiles_per_sm(const Launch& L, int per_sm, K kernel, A... args) {
  const int64_t n = L.tile_end - L.tile_begin;
  if (n <= 0) return cudaSuccess;
  int cap = resident_ctas(kernel, kThreads);
  if (cap <= 0) {
    const cudaError_t e = cudaGetLastError();
    return static_cast<int>(e != cudaSuccess ? e : cudaErrorUnknown);
  }
  if (per_sm > 0) {
    const int sms = sm_count();
    if (sms > 0 && cap > sms * per_sm) cap = sms * per_sm;
  }
  int64_t g = n < cap ? n : cap;
  if (L.max_ctas > 0 && g > L.max_ctas) g = L.max_ctas;
  if (L.short_ctas && n <= INT_MAX) g = n;   // one CTA per tile
  return launch_k(kernel, static_cast<int>(g), kThreads, 0, L.stream, args...);
}

template <class K, class... A>
int launch_tiles(const Launch& L, K kernel, A... args) {
  return launch_tiles_per_sm(L, 0, kernel, args...);
}

// As launch_tiles_per_sm for kernels that loop with for_each_block(2): when the
// launch covers at most half as many tiles as CTAs fit, two CTAs share each tile
// (k.split = 2), halving each thread's serial chain of loads for the small
// per-bucket launches of streamed synchronisation.
template <class K, class... A>
int launch_tiles_split(const Launch& L, int per_sm, K kernel, KCommon k, A... args) {
  const int64_t n = L.tile_end - L.tile_begin;
  if (n <= 0) return cudaSuccess;
  int cap = resident_ctas(kernel, kThreads);
  if (cap <= 0) {
    const cudaError_t e = cudaGetLastError();
    return static_cast<int>(e != cudaSuccess ? e : cudaErrorUnknown);
  }
  if (per_sm > 0) {
    const int sms = sm_count();
    if (sms > 0 && cap > sms * per_sm) cap = sms * per_sm;
  }
  if (L.short_ctas && n <= INT_MAX) {   // one CTA per tile
    k.split = 1;
    return launch_k(kernel, static_cast<int>(n), kThreads, 0, L.stream, k, args...);
  }
  if (L.max_ctas > 0 && cap > L.max_ctas) cap = L.max_ctas;
  k.split = 2 * n <= cap ? 2 : 1;
  int64_t g = n * k.split < cap ? n * k.split : cap;
  g -= g % k.split;
  return launch_k(kernel, static_cast<int>(g), kThreads, 0, L.stream, k, args...);
}

// The flat all-reduce and reduce-scatter run `small`: `split` CTAs of `threads`
// threads per tile, each thread one 32-byte block with all of the block's
// replica loads issued at once and the plan checked beside them, and one CTA per
// piece of a tile for the whole launch instead of a persistent loop.  Against a
// persistent grid of `big` on GB300: the whole-plan all-reduce 8% faster at
// P = 8 (0.624 -> 0.572 ms on 124M parameters) and 7% at P = 16, the
// reduce-scatter 3% (3.144 -> 3.050 ms on 1.1e9 parameters at P = 8), and
// per-bucket launches of a few tiles, which latency bounds, gain most.  Each CTA
// lives for about one round of DRAM loads, so beside work of higher priority
// (a GEMM wave of the backward) it hands its SM back within microseconds.  A
// launch capped at L.max_ctas CTAs (SMs left to concurrent work) whose pieces do
// not fit under the cap runs `big` on a persistent grid of at most that many
// CTAs, as launch_tiles_split would, unless L.short_ctas asks for short CTAs.
// `small` reads its tile descriptors from the launch's parameters (inside one
// bucket) and checks the plan beside its first loads; `small_tbl` reads them from
// the workspace's table and checks the plan first.  Two instantiations, so the
// one-bucket kernel carries no early check (measured: 9% faster per-bucket
// reduce-scatter launches of 64 KiB buckets without it).
template <class KB, class KS, class KT, class... A>
int launch_small_or_split(const Launch& L, int per_sm, KB big, KS small, KT small_tbl, int threads,
                          int split, KCommon k, A... args) {
  const int64_t n = L.tile_end - L.tile_begin;
  if (n <= 0) return cudaSuccess;
  if ((L.max_ctas <= 0 || L.short_ctas || n * split <= L.max_ctas) && n * split <= INT_MAX) {
    k.split = split;
    if (k.one_nvec > 0)
      return launch_k(small, static_cast<int>(n * split), threads, 0, L.stream, k, args...);
    return launch_k(small_tbl, static_cast<int>(n * split), threads, 0, L.stream, k, args...);
  }
  return launch_tiles_split(L, per_sm, big, k, args...);
}

// Rank counts with a fully unrolled instantiation; others use the runtime-P one.
template <class F>
int with_P(int P, F&& f) {
  switch (P) {
    case 1: return f(std::integral_constant<int, 1>{});
    case 2: return f(std::integral_constant<int, 2>{});
    case 3: return f(std::integral_constant<int, 3>{});
    case 4: return f(std::integral_constant<int, 4>{});
    case 5: return f(std::integral_constant<int, 5>{});
    case 6: return f(std::integral_constant<int, 6>{});
    case 7: return f(std::integral_constant<int, 7>{});
    case 8: return f(std::integral_constant<int, 8>{});
    case 16: return f(std::integral_constant<int, 16>{});
    default: return f(std::integral_constant<int, 0>{});
  }
}

// Flat ring (0), hybrid mesh with the group size S known at compile time (S,
// for the common shapes of 8 and 16 ranks), or with S read at run time (-1).
template <int P, class F>
int with_mesh(const Plan* pl, F&& f) {
  if (pl->R == 1) return f(std::integral_constant<int, 0>{});
  if constexpr (P == 8) {
    if (pl->S == 2) return f(std::integral_constant<int, 2>{});
    if (pl->S == 4) return f(std::integral_constant<int, 4>{});
  }
  if constexpr (P == 16) {
    if (pl->S == 2) return f(std::integral_constant<int, 2>{});
    if (pl->S == 4) return f(std::integral_constant<int, 4>{});
    if (pl->S == 8) return f(std::integral_constant<int, 8>{});
  }
  return f(std::integral_constant<int, -1>{});
}

}  // namespace dps

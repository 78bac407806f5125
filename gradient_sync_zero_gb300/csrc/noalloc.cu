// dp_clip_coef_noalloc: the reduce-scatter-mean and the global-norm clip
// coefficient for callers that cannot allocate device memory.
//
// Who needs it.  The regular path needs a caller-allocated workspace (the plan's
// device tables plus the per-tile norm partials).  Some callers cannot make
// that allocation: a plugin handed device buffers by a host application whose
// memory pool it must not grow, a caller inside a framework whose caching
// allocator must see every byte (a side cudaMalloc would fragment or
// over-subscribe its pool), or a latency-critical loop where cudaMalloc and
// cudaFree, which may synchronise the device, are not acceptable.  This entry
// point keeps the workspace in a fixed, library-owned device array instead, so
// the caller passes only its inputs and outputs.
//
// The array.  kNoallocScratchBytes (32 MiB) in a file-scope __device__ array;
// every GPU that loads this library's code for it holds those 32 MiB until the
// process exits.  It must hold the plan's device tables (about 160 bytes per
// 8192 parameters: the tile table and the weight-decay bits) and eight 8-byte
// norm partials per 8192-parameter tile, so plans up to about 1.2e9 parameters fit;
// the call refuses larger plans with DP_EINVAL and says why.
//
// Sharing.  Every call, on every stream, uses the same array, and the array
// keeps the last call's contents.  Each call rewrites the tables and clears the
// status word before its kernels run, and its kernels overwrite every partial
// they read.  Two calls whose work overlaps on the GPU (different streams
// without ordering, or different host threads) race on the array and give
// wrong results: serialise them.
//
// Set-up.  The first call on each device looks up the array's device address
// (cudaGetSymbolAddress) with that device current and caches it.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstring>
#include <mutex>
#include <string>

#include "internal.h"

namespace dps {
namespace {

constexpr int64_t kNoallocScratchBytes = int64_t(32) << 20;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint8_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once).
int scratch_for_current_device(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_cast<int>(e);
  if (dev < 0 || dev >= kMaxDevices) return static_cast<int>(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return static_cast<int>(e);
    g_scratch_ptr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return 0;
}

}  // namespace
}  // namespace dps

using namespace dps;

extern "C" int dp_clip_coef_noalloc(const dp_plan* plan, const void* grads, float* mean,
                                    double max_norm, float* coef_out, double* norm_out,
                                    void* stream) {
  clear_error();
  const Plan* pl = as_plan(plan);
  if (!pl) return fail(DP_EINVAL, "dp_clip_coef_noalloc: NULL plan");
  if (!coef_out || !norm_out)
    return fail(DP_EINVAL, "dp_clip_coef_noalloc: NULL coef_out or norm_out");
  if (pl->L > 0 && (!grads || !mean))
    return fail(DP_EINVAL, "dp_clip_coef_noalloc: NULL grads or mean");
  if ((reinterpret_cast<uintptr_t>(grads) | reinterpret_cast<uintptr_t>(mean)) & 31u)
    return fail(DP_EALIGN, "dp_clip_coef_noalloc: grads and mean must be 32-byte aligned");
  if ((reinterpret_cast<uintptr_t>(coef_out) & 3u) || (reinterpret_cast<uintptr_t>(norm_out) & 7u))
    return fail(DP_EALIGN, "dp_clip_coef_noalloc: coef_out / norm_out misaligned");
  // Bytes this plan needs: its device tables and the per-tile partials (the
  // fp32 stage the fused step uses is not touched here).
  DevHeader h;
  std::memcpy(&h, pl->image.data(), sizeof(h));
  const int64_t need = h.off_stage;
  if (need > kNoallocScratchBytes)
    return fail(DP_EINVAL, "dp_clip_coef_noalloc: the plan needs " + std::to_string(need) +
                               " bytes of scratch (tables + " + std::to_string(h.n_tiles) +
                               " tile partials); the static array holds " +
                               std::to_string(kNoallocScratchBytes) +
                               " bytes; use dp_reduce_scatter_mean + dp_clip_coef with a workspace");
  uint8_t* scratch = nullptr;
  int e = scratch_for_current_device(&scratch);
  if (e) return fail(DP_ECUDA, std::string("dp_clip_coef_noalloc: cudaGetSymbolAddress: ") +
                                   cudaGetErrorString(static_cast<cudaError_t>(e)));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The tables, with a fresh header (status cleared, norm results reset).
  cudaError_t ce = cudaMemcpyAsync(scratch, pl->image.data(), pl->image.size(),
                                   cudaMemcpyHostToDevice, s);
  if (ce != cudaSuccess)
    return fail(DP_ECUDA, std::string("dp_clip_coef_noalloc: ") + cudaGetErrorString(ce));
  Launch L;
  L.plan = pl;
  L.ws = scratch;
  L.tile_begin = 0;
  L.tile_end = static_cast<int64_t>(pl->tiles.size());
  L.stream = stream;
  e = launch_reduce_scatter(L, grads, mean, true);
  if (!e) e = launch_norm_finalize(L, max_norm);
  if (e) return fail(DP_ECUDA, std::string("dp_clip_coef_noalloc: ") +
                                   cudaGetErrorString(static_cast<cudaError_t>(e)));
  ce = cudaMemcpyAsync(coef_out, scratch + offsetof(DevHeader, coef), sizeof(float),
                       cudaMemcpyDeviceToDevice, s);
  if (ce == cudaSuccess)
    ce = cudaMemcpyAsync(norm_out, scratch + offsetof(DevHeader, norm), sizeof(double),
                         cudaMemcpyDeviceToDevice, s);
  if (ce != cudaSuccess)
    return fail(DP_ECUDA, std::string("dp_clip_coef_noalloc: ") + cudaGetErrorString(ce));
  return DP_OK;
}

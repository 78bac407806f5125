// Streams confined to a few SMs (green contexts), for the streamed mode's
// reductions beside a backward pass.
//
// On one GPU the "communication" of the synchronisation step is HBM work on the
// same SMs as the backward's GEMMs.  A persistent cuBLAS GEMM holds every
// register and most of the shared memory of each SM it runs on (144 of the 152
// SMs for the shapes measured), so a reduction launched beside it either waits
// for whole GEMM waves or takes SMs a GEMM wave needed.  A green context gives
// the reductions a fixed partition of SMs instead: their CTAs never run
// elsewhere, so a GEMM launched while they run finds its SMs free.  The driver
// API that creates green contexts is reached through the runtime's driver entry
// points, so the library still links no driver library.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "internal.h"

namespace dps {
namespace {

struct GreenApi {
  CUresult (*device_get)(CUdevice*, int) = nullptr;
  CUresult (*get_resource)(CUdevice, CUdevResource*, CUdevResourceType) = nullptr;
  CUresult (*split)(CUdevResource*, unsigned int*, const CUdevResource*, CUdevResource*, unsigned int,
                    unsigned int) = nullptr;
  CUresult (*gen_desc)(CUdevResourceDesc*, CUdevResource*, unsigned int) = nullptr;
  CUresult (*ctx_create)(CUgreenCtx*, CUdevResourceDesc, CUdevice, unsigned int) = nullptr;
  CUresult (*ctx_destroy)(CUgreenCtx) = nullptr;
  CUresult (*stream_create)(CUstream*, CUgreenCtx, unsigned int, int) = nullptr;
  CUresult (*stream_destroy)(CUstream) = nullptr;
  std::string missing;   // empty: every entry point was found
};

template <class F>
void entry(const char* name, F* fn, std::string* missing) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12080, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess && p) {
    *fn = reinterpret_cast<F>(p);
  } else {
    cudaGetLastError();
    *missing += (missing->empty() ? "" : ", ") + std::string(name);
  }
}

const GreenApi& green_api() {
  static GreenApi api;
  static std::once_flag once;
  std::call_once(once, [] {
    entry("cuDeviceGet", &api.device_get, &api.missing);
    entry("cuDeviceGetDevResource", &api.get_resource, &api.missing);
    entry("cuDevSmResourceSplitByCount", &api.split, &api.missing);
    entry("cuDevResourceGenerateDesc", &api.gen_desc, &api.missing);
    entry("cuGreenCtxCreate", &api.ctx_create, &api.missing);
    entry("cuGreenCtxDestroy", &api.ctx_destroy, &api.missing);
    entry("cuGreenCtxStreamCreate", &api.stream_create, &api.missing);
    entry("cuStreamDestroy", &api.stream_destroy, &api.missing);
  });
  return api;
}

int drv_fail(const char* what, CUresult r) {
  return fail(DP_ECUDA, std::string("dp_sm_streams_create: ") + what + " failed (CUresult " +
                            std::to_string(static_cast<int>(r)) + ")");
}

// The streams of one split: a partition of n SMs and, optionally, the rest.
struct SmStreams {
  CUgreenCtx part = nullptr, rest = nullptr;
  CUstream s_part = nullptr, s_rest = nullptr;
};

void destroy_streams(const GreenApi& api, SmStreams* h) {
  if (h->s_part) api.stream_destroy(h->s_part);
  if (h->s_rest) api.stream_destroy(h->s_rest);
  if (h->part) api.ctx_destroy(h->part);
  if (h->rest) api.ctx_destroy(h->rest);
  delete h;
}

}  // namespace
}  // namespace dps

using namespace dps;

extern "C" int dp_sm_streams_create(int32_t n_sms, int32_t priority, void** part_stream,
                                    void** rest_stream, void** handle, int32_t* n_part,
                                    int32_t* n_rest) {
  clear_error();
  if (!part_stream || !handle) return fail(DP_EINVAL, "dp_sm_streams_create: NULL stream or handle");
  *part_stream = nullptr;
  if (rest_stream) *rest_stream = nullptr;
  *handle = nullptr;
  if (n_sms < 1) return fail(DP_EINVAL, "dp_sm_streams_create: n_sms must be >= 1");
  const GreenApi& api = green_api();
  if (!api.missing.empty())
    return fail(DP_ECUDA, "dp_sm_streams_create: driver entry points not available: " + api.missing);
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce == cudaSuccess) ce = cudaFree(nullptr);   // the primary context exists
  if (ce != cudaSuccess)
    return fail(DP_ECUDA, std::string("dp_sm_streams_create: ") + cudaGetErrorString(ce));
  CUdevice cudev;
  CUresult r = api.device_get(&cudev, dev);
  if (r != CUDA_SUCCESS) return drv_fail("cuDeviceGet", r);
  CUdevResource all{};
  if ((r = api.get_resource(cudev, &all, CU_DEV_RESOURCE_TYPE_SM)) != CUDA_SUCCESS)
    return drv_fail("cuDeviceGetDevResource", r);
  if (static_cast<unsigned>(n_sms) >= all.sm.smCount)
    return fail(DP_EINVAL, "dp_sm_streams_create: n_sms " + std::to_string(n_sms) +
                               " leaves no SM outside the partition (the GPU has " +
                               std::to_string(all.sm.smCount) + ")");
  // as many groups of n_sms (rounded up to the granularity) as fit; the first is
  // the partition, the other groups and the remainder form the rest
  unsigned int ng = 0;
  if ((r = api.split(nullptr, &ng, &all, nullptr, 0, static_cast<unsigned>(n_sms))) != CUDA_SUCCESS ||
      ng < 1)
    return drv_fail("cuDevSmResourceSplitByCount (query)", r);
  std::vector<CUdevResource> groups(ng + 1);
  CUdevResource rem{};
  if ((r = api.split(groups.data(), &ng, &all, &rem, 0, static_cast<unsigned>(n_sms))) != CUDA_SUCCESS ||
      ng < 1)
    return drv_fail("cuDevSmResourceSplitByCount", r);
  SmStreams* h = new (std::nothrow) SmStreams();
  if (!h) return fail(DP_ENOMEM, "dp_sm_streams_create: out of host memory");
  CUdevResourceDesc desc = nullptr;
  if ((r = api.gen_desc(&desc, &groups[0], 1)) != CUDA_SUCCESS ||
      (r = api.ctx_create(&h->part, desc, cudev, CU_GREEN_CTX_DEFAULT_STREAM)) != CUDA_SUCCESS ||
      (r = api.stream_create(&h->s_part, h->part, CU_STREAM_NON_BLOCKING, priority)) != CUDA_SUCCESS) {
    destroy_streams(api, h);
    return drv_fail("creating the partition", r);
  }
  int32_t rest_sms = 0;
  if (rest_stream) {
    std::vector<CUdevResource> rest(groups.begin() + 1, groups.begin() + ng);
    if (rem.sm.smCount > 0) rest.push_back(rem);
    for (const CUdevResource& x : rest) rest_sms += static_cast<int32_t>(x.sm.smCount);
    if (rest.empty() ||
        (r = api.gen_desc(&desc, rest.data(), static_cast<unsigned>(rest.size()))) != CUDA_SUCCESS ||
        (r = api.ctx_create(&h->rest, desc, cudev, CU_GREEN_CTX_DEFAULT_STREAM)) != CUDA_SUCCESS ||
        (r = api.stream_create(&h->s_rest, h->rest, CU_STREAM_NON_BLOCKING, 0)) != CUDA_SUCCESS) {
      destroy_streams(api, h);
      return drv_fail("creating the rest", r);
    }
    *rest_stream = h->s_rest;
  }
  *part_stream = h->s_part;
  *handle = h;
  if (n_part) *n_part = static_cast<int32_t>(groups[0].sm.smCount);
  if (n_rest) *n_rest = rest_sms;
  return DP_OK;
}

extern "C" int dp_sm_streams_destroy(void* handle) {
  clear_error();
  if (!handle) return DP_OK;
  const GreenApi& api = green_api();
  if (!api.missing.empty()) return fail(DP_ECUDA, "dp_sm_streams_destroy: driver entry points not available");
  destroy_streams(api, static_cast<SmStreams*>(handle));
  return DP_OK;
}

// Reduce-scatter-mean, fused mean all-reduce, and the global-norm finalisation.
//
// Roofline (HBM-bound): reduce-scatter reads 2P bytes and writes 4 bytes per
// element; the all-reduce reads 2P and writes 2P ("4.1 Data parallelism in
// depth", sec. 5.2: each ring phase moves (N-1)/N of the data; here every
// replica is read or written exactly once).
#include <cmath>

#include "launch.cuh"

namespace dps {

// CTAs per SM for the in-place kernels whose reads and writes are both P blocks
// per element: fewer loads in flight than full occupancy run the 1:1 (all-reduce)
// and 2:1 (accumulation) mixes faster on this HBM.  Measured on the 1.1B case,
// P = 8: all-reduce 5.50 -> 5.42 ms at 2 per SM (3 resident), bf16-wire ring
// 5.57 -> 5.32, accumulate 7.83 -> 7.58 and the fused last micro-batch
// 7.94 -> 7.58 at 3 per SM (6 and 4 resident).
constexpr int kAllreducePerSm = 2;
constexpr int kAccumPerSm = 3;

// Reduce-scatter + 1/P: shard c of each bucket receives the fp32 mean rank c
// owns; optionally one partial of sum(mean^2) per tile for the clip norm (the
// walk, the float-float partials and the split rule are rs_tiles in kernels.cuh).
// ACC: the last micro-batch of gradient accumulation fused in — replica r's
// value is bf16(g_r + micro_r), formed in registers (flat plans).
// SMALL (eight 64-thread CTAs per tile, one block per thread): a block's
// replicas are all loaded at once; inside one bucket (descriptors from the
// launch's parameters) the plan id is checked beside the first loads and gates
// the stores, over several buckets (descriptors from the workspace's table) it
// is checked before the table is read.
// NT: threads per CTA (kSmallThreads for small launches without norm partials).
// TBL: a SMALL launch over several buckets (descriptors from the workspace's table:
// the plan is checked before the table is read).
template <int P, int MS, bool ACC, bool SMALL = false, int NT = kThreads, bool TBL = false>
__global__ void __launch_bounds__(NT) k_reduce_scatter(KCommon k, const uint8_t* g, float* mean,
                                                       int sumsq, const uint8_t* micro) {
  uint64_t id = k.plan_id;
  if constexpr (SMALL) {
    id = plan_id_deferred(k);
    if constexpr (TBL) {
      if (!plan_matches(k, id)) return;
    }
  } else {
    if (!plan_ok(k)) return;
  }
  __shared__ FF warp_part[2 * kWarps];
  rs_tiles<P, MS, ACC, SMALL, NT>(k, g, mean, sumsq, micro, id, blockIdx.x, gridDim.x, warp_part);
  if (SMALL) plan_matches(k, id);
}

// Fused mean all-reduce in place: sum in ring order, 1/P, bf16, written back to
// every replica (the all-gather of the reduced shards).
// SMALL: as for k_reduce_scatter.
// TBL: as for k_reduce_scatter.
template <int P, int MS, bool SMALL = false, bool TBL = false>
__global__ void __launch_bounds__(SMALL ? kSmallThreads : kThreads) k_allreduce(KCommon k, uint8_t* g) {
  uint64_t id = k.plan_id;
  if constexpr (SMALL) {
    id = plan_id_deferred(k);
    if constexpr (TBL) {
      if (!plan_matches(k, id)) return;
    }
  } else {
    if (!plan_ok(k)) return;
  }
  for_each_block2<true, SMALL ? kSmallThreads : kThreads>(k, [&](const TileDesc& d, int64_t b, int c) {
    float acc[16];
    block_mean16<P, MS, SMALL ? 16 : 8>(k, g, b, d, c, acc);
    if (!SMALL || id == k.plan_id) store_replicas<P>(g, k.stride_bytes, 32 * b, pack16_rne(acc), k.P);
  });
  if (SMALL) plan_matches(k, id);
}

// The start of the accumulation kernels: SMALL (eight 64-thread CTAs per tile, one
// block per thread) checks the plan as the small all-reduce does (TBL: before the
// workspace's tile table is read), the persistent form before anything.  Returns
// false when the kernel stops; *id is the plan id that gates a SMALL kernel's stores.
template <bool SMALL, bool TBL>
__device__ __forceinline__ bool accum_start(const KCommon& k, uint64_t* id) {
  *id = k.plan_id;
  if constexpr (SMALL) {
    *id = plan_id_deferred(k);
    if constexpr (TBL) return plan_matches(k, *id);
    return true;
  } else {
    return plan_ok(k);
  }
}

// acc[r] = bf16(acc[r] + micro[r]) for every replica.
template <bool SMALL = false, bool TBL = false>
__global__ void __launch_bounds__(SMALL ? kSmallThreads : kThreads)
    k_accumulate(KCommon k, uint8_t* acc, const uint8_t* micro) {
  uint64_t id;
  if (!accum_start<SMALL, TBL>(k, &id)) return;
  for_each_block2<true, SMALL ? kSmallThreads : kThreads>(k, [&](const TileDesc&, int64_t b, int) {
#pragma unroll 4
    for (int r = 0; r < k.P; ++r) {
      const Blk x = ld_blk(acc + r * k.stride_bytes + 32 * b);
      const Blk y = ld_blk(micro + r * k.stride_bytes + 32 * b);
      float a[16], c[16];
      unpack16(x, a);
      unpack16(y, c);
#pragma unroll
      for (int e = 0; e < 16; ++e) a[e] = __fadd_rn(a[e], c[e]);
      if (SMALL && id != k.plan_id) continue;
      st_blk(acc + r * k.stride_bytes + 32 * b, pack16_rne(a));
    }
  });
  if (SMALL) plan_matches(k, id);
}

// Last micro-batch: accumulate and mean all-reduce in one pass, result in acc.
template <int P, bool SMALL = false, bool TBL = false>
__global__ void __launch_bounds__(SMALL ? kSmallThreads : kThreads)
    k_allreduce_accum(KCommon k, uint8_t* acc, const uint8_t* micro) {
  uint64_t id;
  if (!accum_start<SMALL, TBL>(k, &id)) return;
  for_each_block2<SMALL, SMALL ? kSmallThreads : kThreads>(k, [&](const TileDesc&, int64_t b, int c) {
    float mean[16];
    ring_mean16_accum<P>(acc, micro, k.stride_bytes, 32 * b, c, k.P, mean);
    if (!SMALL || id == k.plan_id) store_replicas<P>(acc, k.stride_bytes, 32 * b, pack16_rne(mean), k.P);
  });
  if (SMALL) plan_matches(k, id);
}

// Mean all-reduce with bf16 partial sums on the ring.
template <int P, bool SMALL = false, bool TBL = false>
__global__ void __launch_bounds__(SMALL ? kSmallThreads : kThreads)
    k_allreduce_bf16wire(KCommon k, uint8_t* g) {
  uint64_t id;
  if (!accum_start<SMALL, TBL>(k, &id)) return;
  for_each_block2<SMALL, SMALL ? kSmallThreads : kThreads>(k, [&](const TileDesc&, int64_t b, int c) {
    float mean[16];
    ring_mean16_bf16wire<P>(g, k.stride_bytes, 32 * b, c, k.P, mean);
    if (!SMALL || id == k.plan_id) store_replicas<P>(g, k.stride_bytes, 32 * b, pack16_rne(mean), k.P);
  });
  if (SMALL) plan_matches(k, id);
}

// The global norm over tiles [tile_begin, tile_end): their sub-tile partials
// merged in float-float in a fixed order, then the norm and the clip coefficient
// min(1, max_norm / (norm + 1e-6)) in double ("Distributed Training: Data
// Parallel, Model Parallel and FSDP Strategies", "Inside DDP": clip_grad_norm_
// after the averaged gradients).  The grid's size depends only on the number of
// partials n (ceil(n / kFinPerCta), at most kFinMaxCtas): CTA i merges its
// contiguous share, thread t every 256th partial of it in order, then the warps'
// butterflies and the warps in order; the CTA that finishes last (a counter in
// the workspace header, no waiting) merges the CTAs' sums in CTA order and
// writes the results.  So the norm depends only on the partials, whatever
// launches produced them.
constexpr int kFinThreads = 256;

__device__ __forceinline__ FF ld_ff(const float* p) {
  const float2 q = __ldcg(reinterpret_cast<const float2*>(p));
  return FF{q.x, q.y};
}

__global__ void __launch_bounds__(kFinThreads) k_norm_finalize(KCommon k, double max_norm) {
  if (!plan_ok(k)) return;
  __shared__ FF warp_part[kFinThreads / 32];
  __shared__ int is_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t p0 = kSubTiles * k.tile_begin, n = kSubTiles * (k.tile_end - k.tile_begin);
  const int64_t share = (n + gridDim.x - 1) / gridDim.x;
  const int64_t c0 = p0 + blockIdx.x * share;
  const int64_t c1 = c0 + share < p0 + n ? c0 + share : p0 + n;
  FF acc{0.0f, 0.0f};
  int64_t i = c0 + threadIdx.x;
  for (; i + 3 * kFinThreads < c1; i += 4 * kFinThreads) {
    FF q[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) q[u] = ld_ff(k.sumsq + 2 * (i + u * kFinThreads));
#pragma unroll
    for (int u = 0; u < 4; ++u) acc = ff_merge(acc, q[u]);
  }
  for (; i < c1; i += kFinThreads) acc = ff_merge(acc, ld_ff(k.sumsq + 2 * i));
  acc = warp_ff_sum(acc);
  if (lane == 0) warp_part[warp] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    FF c = warp_part[0];
    for (int w = 1; w < kFinThreads / 32; ++w) c = ff_merge(c, warp_part[w]);
    *reinterpret_cast<float2*>(k.fin + 2 * blockIdx.x) = make_float2(c.hi, c.lo);
    __threadfence();
    is_last = atomicAdd(&k.hdr->fin_count, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!is_last || warp != 0) return;
  __threadfence();
  FF a{0.0f, 0.0f};
  for (int64_t c = lane; c < gridDim.x; c += 32) a = ff_merge(a, ld_ff(k.fin + 2 * c));
  a = warp_ff_sum(a);
  if (lane == 0) {
    const double n2 = static_cast<double>(a.hi) + static_cast<double>(a.lo);
    const double norm = sqrt(n2);
    float coef = 1.0f;
    if (!isfinite(norm)) {
      atomicOr(&k.hdr->status, DP_STATUS_NONFINITE);
      if (max_norm > 0.0) coef = __int_as_float(0x7fc00000);
    } else if (max_norm > 0.0) {
      coef = __double2float_rn(fmin(1.0, max_norm / (norm + 1e-6)));
    }
    k.hdr->norm2 = n2;
    k.hdr->norm = norm;
    k.hdr->coef = coef;
    k.hdr->fin_count = 0;   // ready for the next norm pass on this workspace
  }
}

int launch_reduce_scatter(const Launch& L, const void* grads, float* mean, bool sumsq,
                          int64_t rep_stride, int64_t rep_block0) {
  KCommon k = make_common(L);
  if (rep_stride > 0) k.stride_bytes = 2 * rep_stride;   // replicas in a unit buffer
  k.rep_block0 = rep_block0;
  return with_P(L.plan->P, [&](auto pc) {
    constexpr int P = decltype(pc)::value;
    return with_mesh<P>(L.plan, [&](auto mc) {
      constexpr int M = decltype(mc)::value;
      // mesh plans keep the persistent grid: measured on GB300 the small kernel was
      // 5% slower on a 2 x 4 mesh (3.29 against 3.13 ms on 1.1e9 parameters) and
      // 2% faster on 4 x 2
      if constexpr (M != 0) {
        if (sumsq)
          return launch_tiles(L, k_reduce_scatter<P, M, false>, k, static_cast<const uint8_t*>(grads),
                              mean, 1, static_cast<const uint8_t*>(nullptr));
        return launch_tiles_split(L, 0, k_reduce_scatter<P, M, false>, k,
                                  static_cast<const uint8_t*>(grads), mean, 0,
                                  static_cast<const uint8_t*>(nullptr));
      }
      // flat plans: the SMALL kernel (launch_small_or_split); each small CTA forms
      // its sub-tile's norm partial as a whole-tile CTA would
      return launch_small_or_split(L, 0, k_reduce_scatter<P, M, false>,
                                   k_reduce_scatter<P, M, false, true, kSmallThreads>,
                                   k_reduce_scatter<P, M, false, true, kSmallThreads, true>,
                                   kSmallThreads, kSmallSplit, k,
                                   static_cast<const uint8_t*>(grads), mean, sumsq ? 1 : 0,
                                   static_cast<const uint8_t*>(nullptr));
    });
  });
}

int launch_reduce_scatter_accum(const Launch& L, const void* acc, const void* micro, float* mean,
                                bool sumsq) {
  const KCommon k = make_common(L);
  return with_P(L.plan->P, [&](auto pc) {
    constexpr int P = decltype(pc)::value;
    return launch_tiles(L, k_reduce_scatter<P, 0, true>, k, static_cast<const uint8_t*>(acc), mean,
                        sumsq ? 1 : 0, static_cast<const uint8_t*>(micro));
  });
}

int launch_allreduce(const Launch& L, void* grads) {
  const KCommon k = make_common(L);
  return with_P(L.plan->P, [&](auto pc) {
    constexpr int P = decltype(pc)::value;
    return with_mesh<P>(L.plan, [&](auto mc) {
      constexpr int M = decltype(mc)::value;
      // the SMALL kernel (launch_small_or_split)
      return launch_small_or_split(L, kAllreducePerSm, k_allreduce<P, M>, k_allreduce<P, M, true>,
                                   k_allreduce<P, M, true, true>,
                                   kSmallThreads, kSmallSplit, k, static_cast<uint8_t*>(grads));
    });
  });
}

int64_t bounds_violations_reduce(bool reset) {
#ifdef DPSYNC_CHECKED
  unsigned long long n = 0;
  if (cudaMemcpyFromSymbol(&n, g_bounds_violations, sizeof n) != cudaSuccess) return -2;
  if (reset) {
    const unsigned long long z = 0;
    if (cudaMemcpyToSymbol(g_bounds_violations, &z, sizeof z) != cudaSuccess) return -2;
  }
  return static_cast<int64_t>(n);
#else
  (void)reset;
  return -1;
#endif
}

int launch_accumulate(const Launch& L, void* acc, const void* micro) {
  return launch_small_or_split(L, kAccumPerSm, k_accumulate<>, k_accumulate<true>,
                               k_accumulate<true, true>, kSmallThreads, kSmallSplit, make_common(L),
                               static_cast<uint8_t*>(acc), static_cast<const uint8_t*>(micro));
}

int launch_allreduce_accum(const Launch& L, void* acc, const void* micro) {
  const KCommon k = make_common(L);
  return with_P(L.plan->P, [&](auto pc) {
    constexpr int P = decltype(pc)::value;
    return launch_small_or_split(L, kAccumPerSm, k_allreduce_accum<P>, k_allreduce_accum<P, true>,
                                 k_allreduce_accum<P, true, true>, kSmallThreads, kSmallSplit, k,
                                 static_cast<uint8_t*>(acc), static_cast<const uint8_t*>(micro));
  });
}

int launch_allreduce_bf16wire(const Launch& L, void* grads) {
  const KCommon k = make_common(L);
  return with_P(L.plan->P, [&](auto pc) {
    constexpr int P = decltype(pc)::value;
    return launch_small_or_split(L, kAllreducePerSm, k_allreduce_bf16wire<P>,
                                 k_allreduce_bf16wire<P, true>, k_allreduce_bf16wire<P, true, true>,
                                 kSmallThreads, kSmallSplit, k, static_cast<uint8_t*>(grads));
  });
}

int launch_norm_finalize(const Launch& L, double max_norm) {
  const KCommon k = make_common(L);
  const int64_t n = kSubTiles * (L.tile_end - L.tile_begin);
  int64_t g = (n + kFinPerCta - 1) / kFinPerCta;
  if (g < 1) g = 1;
  if (g > kFinMaxCtas) g = kFinMaxCtas;
  return launch_k(k_norm_finalize, static_cast<int>(g), kFinThreads, 0, L.stream, k, max_norm);
}

}  // namespace dps

// Sharded AdamW, all-gather / broadcast write-back, and the fused ZeRO-1/2 step.
//
// ZeRO-1 and ZeRO-2 keep DDP's reduce-scatter, let each rank update only the
// shard it owns, and all-gather the new parameters ("Data Parallelism: DDP, ZeRO
// and FSDP", "The three stages").  On one GPU the P replicas are P HBM
// buffers, so the fused kernel performs the three phases per 32-byte block:
// read P gradient blocks and the owner's fp32 state once, write the state and
// P parameter blocks once.
//
// Roofline (HBM-bound), bytes per element: fused step 2P + 12 read, 12 + 2P
// written; AdamW alone 16 read, 12 + 2 written; all-gather 2 read, 2(P-1)
// written; AdamW fused with the all-gather (second pass of the clipped step)
// 16 read, 12 + 2P written.
#include "launch.cuh"

namespace dps {

// Sharded AdamW on an fp32 gradient [L]; the owner's replica gets bf16(theta).
// dev_s: take the step's scalars from the workspace header (dp_set_adamw_cfg), so a
// captured graph of the step replays with the scalars of the current step.
__device__ __forceinline__ bool header_scalars(const KCommon& k, AdamScalars& s) {
  if (k.hdr->adam_tag != kAdamTag) {
    if (threadIdx.x == 0) atomicOr(&k.hdr->status, DP_STATUS_NO_SCALARS);
    return false;
  }
  s = k.hdr->adam;
  return true;
}

// coefp: the clip coefficient (device fp32: the workspace's, or the caller's own),
// read once the previous kernel has finished; NULL = no clipping.
__device__ __forceinline__ void adamw_body(const KCommon& k, const float* grad, float* master,
                                           float* m, float* v, uint8_t* params,
                                           const AdamScalars& s, const float* coefp) {
  const float coef = coefp ? *coefp : 1.0f;
  for_each_block(k, [&](int64_t, int64_t b, int c) {
    float g[16], th[16], mm[16], vv[16];
    ld_f16(grad, b, g);
    ld_f16(master, b, th);
    ld_f16(m, b, mm);
    ld_f16(v, b, vv);
    const uint32_t dec = decay_bits2(k.decay, b);
    if (coefp) {
#pragma unroll
      for (int e = 0; e < 16; ++e) g[e] = __fmul_rn(g[e], coef);
    }
    adamw16(g, th, mm, vv, dec, s);
    st_f16(master, b, th);
    st_f16(m, b, mm);
    st_f16(v, b, vv);
    const Blk val = pack16_rne(th);
    // the owner of shard c in every group (rank c on a flat ring)
    for (int g = 0; g < k.R; ++g) st_blk(params + (g * k.S + c) * k.stride_bytes + 32 * b, val);
  });
}

// DEV_S: the scalars come from the workspace header (a separate instantiation, so
// the per-call path keeps them in the kernel's parameter space).
template <bool DEV_S>
__global__ void __launch_bounds__(kThreads)
    k_adamw(KCommon k, const float* grad, float* master, float* m, float* v, uint8_t* params,
            AdamScalars s, const float* coefp) {
  if (!plan_ok(k)) return;
  if constexpr (DEV_S) {
    AdamScalars sd;
    if (!header_scalars(k, sd)) return;
    adamw_body(k, grad, master, m, v, params, sd, coefp);
  } else {
    adamw_body(k, grad, master, m, v, params, s, coefp);
  }
}

// ---- replica write-back with bulk copies: all-gather, broadcast, unit all-gather ----
// (Kept for comparison, selected with DPSYNC_REP_BULK: the default is the small-CTA
// write-back, k_replicate_small, 10% faster on GB300.)
// Each tile (<= 8192 elements, inside one bucket) is one job: one thread streams
// the tile's source segments into a shared-memory stage (bulk loads counted on an
// mbarrier) and writes the stage to every destination row with bulk stores.
// Written with per-thread 32-byte accesses on a persistent grid, one load feeds
// P-1 stores and the LSU queue limited the kernel (lg_throttle 23 stalls per issue
// at P = 8); a bulk store moves a whole segment per instruction.  A 6-deep ring of 16 KB stages
// (96 KB, 2 CTAs per SM): against 2-4 stages it changes the all-gather by <0.5%
// and makes each short ZeRO-3 unit gather 5% faster.  Every wait is bounded
// (DP_STATUS_TIMEOUT, the CTA still drains its copies).
//   all-gather: the owner's row of each shard -> every row r with r mod S != owner
//   broadcast:  row src -> every other row
//   unit:       the flat bf16 shard array -> all P rows of a unit buffer
enum RepMode : int { kRepAllGather = 0, kRepBroadcast = 1, kRepUnit = 2 };
constexpr int kRepStages = 6;
constexpr uint32_t kRepStageBytes = static_cast<uint32_t>(kTileElems) * 2;   // 16 KB
constexpr size_t kRepSmem = kRepStages * static_cast<size_t>(kRepStageBytes) +
                            kRepStages * sizeof(uint64_t);

struct RepArgs {
  const uint8_t* src;     // replicas (all-gather, broadcast) or the flat shards (unit)
  uint8_t* dst;           // replicas or the unit buffer
  int64_t dst_stride;     // bytes between destination rows
  int64_t dst_vec0;       // unit: the unit's first 16-byte vector (destination column 0)
  int64_t dst_vec_limit;  // unit: 16-byte vectors per destination row
  int mode;
  int src_rank;           // broadcast
};

// The replicate walk for CTA `cta` of `ncta`, run by one thread with an ST-deep
// ring of 16 KB stages at `smem` (ST * kRepStageBytes + ST barriers).
template <int ST>
__device__ __forceinline__ void replicate_tiles(const KCommon& k, const RepArgs& a, int64_t cta,
                                                int64_t ncta, uint8_t* smem) {
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + ST * kRepStageBytes);
  for (int q = 0; q < ST; ++q) mbar_init(&bar[q]);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const int64_t first = k.tile_begin + cta, step = ncta;
  const int64_t mine = first < k.tile_end ? (k.tile_end - first + step - 1) / step : 0;

  // f(x, e, c) for each run [x, e) of 16-byte vectors of the tile with one source row
  auto segments = [&](const TileDesc& d, auto&& f) {
    const int64_t end = d.v0 + d.nvec;
    if (a.mode != kRepAllGather) {
      f(d.v0, end, a.src_rank);
      return;
    }
    for (int64_t x = d.v0; x < end;) {
      const int c = owner_of(d, x);
      int64_t e = d.bvoff + static_cast<int64_t>(c + 1) * d.svec;
      if (e > end) e = end;
      f(x, e, c);
      x = e;
    }
  };
  auto issue_load = [&](int64_t i) {
    if (i >= mine) return;
    const int64_t tile = first + i * step;
    const TileDesc d = load_tile(k, tile);
    uint64_t* q = &bar[i % ST];
    if (!tile_ok(k, tile, d)) {
      mbar_arrive_expect_tx(q, 0u);   // checked build: the stage completes empty
      return;
    }
    uint8_t* stage = smem + (i % ST) * kRepStageBytes;
    mbar_arrive_expect_tx(q, 16u * static_cast<uint32_t>(d.nvec));
    segments(d, [&](int64_t x, int64_t e, int c) {
      const uint8_t* src = a.mode == kRepUnit ? a.src + 16 * x : a.src + c * k.stride_bytes + 16 * x;
      bulk_load(stage + 16 * (x - d.v0), src, 16u * static_cast<uint32_t>(e - x), q);
    });
  };
  auto issue_stores = [&](int64_t i) {
    const int64_t tile = first + i * step;
    const TileDesc d = load_tile(k, tile);
    if (!tile_ok(k, tile, d)) return;
    const uint8_t* stage = smem + (i % ST) * kRepStageBytes;
    segments(d, [&](int64_t x, int64_t e, int c) {
      const uint32_t bytes = 16u * static_cast<uint32_t>(e - x);
      const uint8_t* sm = stage + 16 * (x - d.v0);
      for (int r = 0; r < k.P; ++r) {
        if (a.mode == kRepAllGather && r % k.S == c) continue;
        if (a.mode == kRepBroadcast && r == a.src_rank) continue;
        const int64_t col = a.mode == kRepUnit ? x - a.dst_vec0 : x;
        if (a.mode == kRepUnit && !DP_IN_BOUNDS(col >= 0 && col + (e - x) <= a.dst_vec_limit)) continue;
        bulk_store(a.dst + r * a.dst_stride + 16 * col, sm, bytes);
      }
    });
  };

  for (int q = 0; q < ST - 1; ++q) issue_load(q);
  bool timed_out = false;
  int64_t i = 0;
  for (; i < mine; ++i) {
    if (!mbar_wait_bounded(&bar[i % ST], static_cast<uint32_t>((i / ST) & 1))) {
      timed_out = true;
      break;
    }
    issue_stores(i);
    bulk_commit();
    bulk_wait_read<1>();                // tile i-1's stores have left its stage ...
    issue_load(i + ST - 1);             // ... which now receives the tile ST-1 ahead
  }
  if (timed_out) {
    atomicOr(&k.hdr->status, DP_STATUS_TIMEOUT);
    for (int64_t q = i; q < i + ST - 1 && q < mine; ++q)   // loads in flight (bounded)
      mbar_wait_bounded(&bar[q % ST], static_cast<uint32_t>((q / ST) & 1));
  }
  bulk_wait_all();
}

__global__ void __launch_bounds__(32) k_replicate(KCommon k, RepArgs a) {
  if (!plan_ok(k)) return;
  if (threadIdx.x != 0) return;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  replicate_tiles<kRepStages>(k, a, blockIdx.x, gridDim.x, smem_raw);
}

// The same write-back as eight 64-thread CTAs per tile, one 32-byte block per
// thread: one load, then a store to every destination row.  Short CTAs that
// each own one block keep the stores spread over the whole GPU, where a
// persistent grid of such threads queued on the LSU (above).  The plan is checked
// before the tile table is read.
// id: the plan id this launch read, compared before the stores (inside one bucket the
// walk reads descriptors from the launch's parameters, so the check can wait until
// the loads are out; over several buckets the caller checks it before the walk).
__device__ __forceinline__ void replicate_small(const KCommon& k, const RepArgs& a, int64_t cta,
                                                int64_t ncta, uint64_t id) {
  for_each_block2_of<true, kSmallThreads>(k, cta, ncta, [&](const TileDesc&, int64_t b, int c) {
    const int64_t x = 2 * b;   // the block's first 16-byte vector
    if (a.mode == kRepUnit) {
      const int64_t col = x - a.dst_vec0;
      if (!DP_IN_BOUNDS(col >= 0 && col + 2 <= a.dst_vec_limit)) return;
      const Blk val = ld_blk(a.src + 16 * x);
      if (id != k.plan_id) return;
#pragma unroll 1
      for (int r = 0; r < k.P; ++r) st_blk(a.dst + r * a.dst_stride + 16 * col, val);
      return;
    }
    const int src_row = a.mode == kRepAllGather ? c : a.src_rank;
    const Blk val = ld_blk(a.src + src_row * k.stride_bytes + 16 * x);
    if (id != k.plan_id) return;
#pragma unroll 1
    for (int r = 0; r < k.P; ++r) {
      if (a.mode == kRepAllGather && r % k.S == c) continue;
      if (a.mode == kRepBroadcast && r == a.src_rank) continue;
      st_blk(a.dst + r * a.dst_stride + 16 * x, val);
    }
  });
}

// TBL: descriptors from the workspace's table (a launch over several buckets).
template <bool TBL>
__global__ void __launch_bounds__(kSmallThreads) k_replicate_small(KCommon k, RepArgs a) {
  const uint64_t id = plan_id_deferred(k);
  if constexpr (TBL) {
    if (!plan_matches(k, id)) return;
  }
  replicate_small(k, a, blockIdx.x, gridDim.x, id);
  if constexpr (!TBL) plan_matches(k, id);
}

bool rep_bulk() {
  static const bool bulk = std::getenv("DPSYNC_REP_BULK") != nullptr;
  return bulk;
}

// ZeRO-3 backward, two units in one launch: the gather of one unit's parameters
// (the next unit's, FSDP's prefetch) and the reduce-scatter of another unit's
// gradients ("Data Parallelism: DDP, ZeRO and FSDP", "How FSDP actually runs":
// the next unit is gathered while the current one's gradients are reduced).  The
// two touch disjoint memory, so the grid splits: CTAs [0, n_rs) run the
// reduce-scatter's tile walk (256 threads each), the rest the replicate walk
// (one thread, a 3-deep ring of 16 KB stages, which leaves room for three CTAs
// per SM).  One launch instead of two removes a launch ramp and tail per unit,
// and mixes the reduce-scatter's read-heavy traffic with the gather's
// write-heavy traffic.
constexpr int kUnitBwdStages = 3;
constexpr size_t kUnitBwdSmem = kUnitBwdStages * static_cast<size_t>(kRepStageBytes) +
                                kUnitBwdStages * sizeof(uint64_t);

template <int P, int MS>
__global__ void __launch_bounds__(kThreads)
    k_unit_backward(KCommon krs, const uint8_t* g, float* mean, int sumsq, KCommon kag, RepArgs a,
                    int n_rs) {
  if (!plan_ok(krs)) return;
  if (static_cast<int>(blockIdx.x) < n_rs) {
    __shared__ FF warp_part[2 * kWarps];
    rs_tiles<P, MS, false, false>(krs, g, mean, sumsq, nullptr, krs.plan_id, blockIdx.x, n_rs,
                                  warp_part);
  } else if (threadIdx.x == 0) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    replicate_tiles<kUnitBwdStages>(kag, a, blockIdx.x - n_rs, gridDim.x - n_rs, smem_raw);
  }
}

// The same two jobs as eight 64-thread CTAs per tile each: CTAs [0, n_rs) take
// the reduce-scatter's pieces, the rest the gather's.  Both units are single
// buckets (descriptors from the launch's parameters), so both check the plan
// beside their first loads and gate their stores on it.
template <int P, int MS>
__global__ void __launch_bounds__(kSmallThreads)
    k_unit_backward_small(KCommon krs, const uint8_t* g, float* mean, int sumsq, KCommon kag,
                          RepArgs a, int n_rs) {
  const uint64_t id = plan_id_deferred(krs);
  if (static_cast<int>(blockIdx.x) < n_rs) {
    __shared__ FF warp_part[2 * (kSmallThreads / 32)];
    rs_tiles<P, MS, false, true, kSmallThreads>(krs, g, mean, sumsq, nullptr, id, blockIdx.x, n_rs,
                                               warp_part);
    plan_matches(krs, id);
  } else {
    replicate_small(kag, a, blockIdx.x - n_rs, gridDim.x - n_rs, id);
    plan_matches(kag, id);
  }
}

int launch_replicate(const Launch& L, const RepArgs& a) {
  if (L.tile_end <= L.tile_begin) return cudaSuccess;
  if (!rep_bulk() && (L.max_ctas <= 0 || L.short_ctas) &&
      (L.tile_end - L.tile_begin) * kSmallSplit <= INT_MAX) {
    KCommon k = make_common(L);
    k.split = kSmallSplit;
    const int grid = static_cast<int>((L.tile_end - L.tile_begin) * kSmallSplit);
    if (k.one_nvec > 0) return launch_k(k_replicate_small<false>, grid, kSmallThreads, 0, L.stream, k, a);
    return launch_k(k_replicate_small<true>, grid, kSmallThreads, 0, L.stream, k, a);
  }
  cudaError_t e = ensure_dyn_smem(k_replicate, kRepSmem);
  if (e != cudaSuccess) return static_cast<int>(e);
  const int64_t cap = resident_ctas(k_replicate, 32, kRepSmem);
  if (cap <= 0) {
    e = cudaGetLastError();
    return static_cast<int>(e != cudaSuccess ? e : cudaErrorUnknown);
  }
  const int64_t n = L.tile_end - L.tile_begin;
  int64_t g = n < cap ? n : cap;
  if (L.max_ctas > 0 && g > L.max_ctas) g = L.max_ctas;
  if (L.short_ctas && n <= INT_MAX) g = n;   // one CTA per tile
  return launch_k(k_replicate, static_cast<int>(g), 32, kRepSmem, L.stream, make_common(L), a);
}

// The whole ZeRO-1/2 step without clipping, one pass.  The replica blocks are
// loaded and folded first, then the fp32 state is loaded, which bounds the live
// registers to one of the two groups.  SMALL: eight 64-thread CTAs per tile, one
// block per thread with all of its replica loads at once, the plan checked as in
// the small all-reduce (beside the first loads inside one bucket, before the tile
// table is read over several), every store gated on it.
template <int P, int MS, bool SMALL = false, bool TBL = false>
__global__ void __launch_bounds__(SMALL ? kSmallThreads : kThreads)
    k_zero_fused(KCommon k, const uint8_t* grads, uint8_t* params, float* master, float* m,
                 float* v, AdamScalars s) {
  uint64_t id = k.plan_id;
  if constexpr (SMALL) {
    id = plan_id_deferred(k);
    if constexpr (TBL) {   // descriptors from the workspace: check before reading them
      if (!plan_matches(k, id)) return;
    }
  } else {
    if (!plan_ok(k)) return;
  }
  for_each_block2<true, SMALL ? kSmallThreads : kThreads>(k, [&](const TileDesc& d, int64_t b, int c) {
    float g[16];
    block_mean16<P, MS, SMALL ? 16 : 8>(k, grads, b, d, c, g);
    if (SMALL && id != k.plan_id) return;
    float th[16], mm[16], vv[16];
    ld_f16(master, b, th);
    ld_f16(m, b, mm);
    ld_f16(v, b, vv);
    const uint32_t dec = decay_bits2(k.decay, b);
    adamw16(g, th, mm, vv, dec, s);
    st_f16(master, b, th);
    st_f16(m, b, mm);
    st_f16(v, b, vv);
    store_replicas<P>(params, k.stride_bytes, 32 * b, pack16_rne(th), k.P);
  });
  if (SMALL) plan_matches(k, id);
}

// ---- second pass of the clipped step, staged through shared memory by bulk copies ----
// (Kept for comparison, selected with DPSYNC_AG_BULK: the default is the small-CTA
// pass below, 10% faster on GB300.)  The pass needs no shard owner (every replica
// gets the same parameters), so it walks [0, L) in chunks of kTmaChunk elements.  One elected thread streams the
// four fp32 inputs of a chunk (mean, master, m, v) into a shared-memory ring
// with cp.async.bulk (completion counted on an mbarrier), the CTA updates
// the chunk in place, and the elected thread streams master, m, v and the bf16
// parameters back out with bulk stores, the parameters once per replica.  Large
// contiguous bulk transfers run the 36%-read / 64%-write mix of this pass closer
// to the HBM limit than per-thread 32-byte accesses from a persistent grid did
// (short-lived CTAs with one block per thread do better still).  Every wait is bounded: a
// timeout sets DP_STATUS_TIMEOUT, and the CTA still drains its own copies.
//
// Chunk and ring depth: 2048 elements and 2 stages (36 KB per stage, 3 CTAs per
// SM), one chunk loading while the previous one is updated and stored.  Measured
// on the 1.1B case against 1024 x {2, 3, 4} stages, 2048 x 3 and 3072 / 4096 x 2:
// 3.3% faster than 1024 x 3 (the deeper rings keep more reads in flight and run
// the read/write mix worse); per-thread 32-byte accesses on a persistent grid were
// slower still.
template <int CH>
struct TmaStageT {
  float in[4][CH];           // mean, master, m, v
  uint32_t out[CH / 2];      // bf16 parameters, two per word
};
template <int CH, int ST>
constexpr size_t tma_smem() { return ST * sizeof(TmaStageT<CH>) + ST * sizeof(uint64_t); }
constexpr int kTmaChunk = 2048;
constexpr int kTmaStages = 2;

template <int CH, int ST>
__device__ __forceinline__ void adamw_ag_body(const KCommon& k, const float* mean, uint8_t* params,
                                              float* master, float* m, float* v,
                                              const AdamScalars& s, int64_t L,
                                              const float* coefp, int rows, int64_t row_bytes) {
  using Stage = TmaStageT<CH>;
  constexpr int kPer = CH / kThreads;   // elements per thread per chunk (multiple of 4)
  static_assert(kPer % 4 == 0 && ST >= 2, "float4 lanes; at least double buffering");
  if (!DP_IN_BOUNDS(L >= 0 && L <= kVecElems * k.hdr->n_vec)) return;
  const int64_t nchunks = (L + CH - 1) / CH;
  if (static_cast<int64_t>(blockIdx.x) >= nchunks) return;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Stage* buf = reinterpret_cast<Stage*>(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw + ST * sizeof(Stage));
  const float coef = coefp ? *coefp : 1.0f;   // x 1 is exact: no clipping
  if (threadIdx.x == 0) {
    for (int q = 0; q < ST; ++q) mbar_init(&bar[q]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int64_t first = blockIdx.x, step = gridDim.x;
  auto issue_load = [&](int64_t i) {  // elected thread: chunk i of this CTA into stage i % ST
    const int64_t c = first + i * step;
    if (c >= nchunks) return;
    const int64_t e0 = c * CH;
    const uint32_t n = static_cast<uint32_t>(L - e0 < CH ? L - e0 : CH);
    Stage& b = buf[i % ST];
    uint64_t* q = &bar[i % ST];
    mbar_arrive_expect_tx(q, 16u * n);
    bulk_load(b.in[0], mean + e0, 4u * n, q);
    bulk_load(b.in[1], master + e0, 4u * n, q);
    bulk_load(b.in[2], m + e0, 4u * n, q);
    bulk_load(b.in[3], v + e0, 4u * n, q);
  };
  if (threadIdx.x == 0)
    for (int q = 0; q < ST - 1; ++q) issue_load(q);
  bool timed_out = false;
  int64_t i = 0;
  for (; first + i * step < nchunks; ++i) {
    const int sidx = static_cast<int>(i % ST);
    const bool ok = mbar_wait_bounded(&bar[sidx], static_cast<uint32_t>((i / ST) & 1));
    if (__syncthreads_or(!ok)) {
      timed_out = true;
      break;
    }
    const int64_t e0 = (first + i * step) * CH;
    const int n = static_cast<int>(L - e0 < CH ? L - e0 : CH);
    Stage& b = buf[sidx];
#pragma unroll
    for (int q = 0; q < kPer / 4; ++q) {
      const int j = 4 * threadIdx.x + q * 4 * kThreads;
      if (j >= n) break;
      float4 g = *reinterpret_cast<const float4*>(&b.in[0][j]);
      float4 th = *reinterpret_cast<const float4*>(&b.in[1][j]);
      float4 mm = *reinterpret_cast<const float4*>(&b.in[2][j]);
      float4 vv = *reinterpret_cast<const float4*>(&b.in[3][j]);
      const int64_t vec = (e0 + j) >> 3;  // the 16-byte gradient vector of these 4 elements
      const bool dec = (__ldg(k.decay + (vec >> 5)) >> (vec & 31)) & 1u;
      adamw1(__fmul_rn(g.x, coef), th.x, mm.x, vv.x, dec, s);
      adamw1(__fmul_rn(g.y, coef), th.y, mm.y, vv.y, dec, s);
      adamw1(__fmul_rn(g.z, coef), th.z, mm.z, vv.z, dec, s);
      adamw1(__fmul_rn(g.w, coef), th.w, mm.w, vv.w, dec, s);
      *reinterpret_cast<float4*>(&b.in[1][j]) = th;
      *reinterpret_cast<float4*>(&b.in[2][j]) = mm;
      *reinterpret_cast<float4*>(&b.in[3][j]) = vv;
      *reinterpret_cast<uint2*>(&b.out[j / 2]) = make_uint2(pack2_rne(th.x, th.y),
                                                             pack2_rne(th.z, th.w));
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      bulk_store(master + e0, b.in[1], 4u * n);
      bulk_store(m + e0, b.in[2], 4u * n);
      bulk_store(v + e0, b.in[3], 4u * n);
      for (int r = 0; r < rows; ++r) bulk_store(params + r * row_bytes + 2 * e0, b.out, 2u * n);
      bulk_commit();
      bulk_wait_read<1>();    // the previous chunk's stores have left its stage ...
      issue_load(i + ST - 1); // ... which now receives the chunk ST-1 ahead
    }
  }
  if (threadIdx.x == 0) {
    if (timed_out) {
      atomicOr(&k.hdr->status, DP_STATUS_TIMEOUT);
      for (int64_t q = i; q < i + ST - 1; ++q)  // loads still in flight: drain them (bounded)
        if (first + q * step < nchunks)
          mbar_wait_bounded(&bar[q % ST], static_cast<uint32_t>((q / ST) & 1));
    }
    bulk_wait_all();
  }
}

// The same pass as eight 64-thread CTAs per tile, one 16-element block per thread
// with all of its loads issued at once (plain 256-bit loads and stores, no
// staging): g = mean x coef, AdamW on master/m/v, bf16(theta) into each of
// `rows` rows.  The pass covers every bucket, so the plan is checked before the
// tile table is read.
// OWNER: the staged step's AdamW instead, bf16(theta) into the owner's row of
// each group only (the all-gather follows as its own pass).
template <bool DEV_S, bool OWNER = false>
__global__ void __launch_bounds__(kSmallThreads)
    k_adamw_all_gather_small(KCommon k, const float* mean, uint8_t* params, float* master,
                             float* m, float* v, AdamScalars s, const float* coefp, int rows,
                             int64_t row_bytes) {
  if (!plan_matches(k, plan_id_deferred(k))) return;
  if constexpr (DEV_S) {
    if (!header_scalars(k, s)) return;
  }
  const float coef = coefp ? *coefp : 1.0f;   // x 1 is exact: no clipping
  for_each_block2<true, kSmallThreads>(k, [&](const TileDesc&, int64_t b, int c) {
    float g[16], th[16], mm[16], vv[16];
    ld_f16(mean, b, g);
    ld_f16(master, b, th);
    ld_f16(m, b, mm);
    ld_f16(v, b, vv);
    const uint32_t dec = decay_bits2(k.decay, b);
#pragma unroll
    for (int e = 0; e < 16; ++e) g[e] = __fmul_rn(g[e], coef);
    adamw16(g, th, mm, vv, dec, s);
    st_f16(master, b, th);
    st_f16(m, b, mm);
    st_f16(v, b, vv);
    const Blk val = pack16_rne(th);
    if constexpr (OWNER) {
#pragma unroll 1
      for (int g2 = 0; g2 < k.R; ++g2) st_blk(params + (g2 * k.S + c) * k.stride_bytes + 32 * b, val);
    } else {
#pragma unroll 1
      for (int r = 0; r < rows; ++r) st_blk(params + r * row_bytes + 32 * b, val);
    }
  });
}

// DEV_S: the scalars come from the workspace header (see k_adamw).
template <bool DEV_S, int CH = kTmaChunk, int ST = kTmaStages>
__global__ void __launch_bounds__(kThreads)
    k_adamw_all_gather(KCommon k, const float* mean, uint8_t* params, float* master, float* m,
                       float* v, AdamScalars s, int64_t L, const float* coefp, int rows,
                       int64_t row_bytes) {
  if (!plan_ok(k)) return;
  if constexpr (DEV_S) {
    AdamScalars sd;
    if (!header_scalars(k, sd)) return;
    adamw_ag_body<CH, ST>(k, mean, params, master, m, v, sd, L, coefp, rows, row_bytes);
  } else {
    adamw_ag_body<CH, ST>(k, mean, params, master, m, v, s, L, coefp, rows, row_bytes);
  }
}

// Failure-path check of the bounded wait: one thread arms an mbarrier for 16
// bytes that no copy will ever deliver, waits with the bulk-copy kernels' bounded
// wait, and reports the timeout.  Nothing is in flight when it returns.
__global__ void k_selftest_wait(int32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  mbar_arrive_expect_tx(&bar, 16u);
  const uint64_t t0 = global_ns();
  const bool ok = mbar_wait_bounded(&bar, 0u, limit_ns);
  status[0] = ok ? 0 : DP_STATUS_TIMEOUT;
  status[1] = static_cast<int32_t>((global_ns() - t0) / 1000000ull);  // ms waited
}

int launch_selftest_wait(int32_t* status, uint64_t limit_ns, void* stream) {
  k_selftest_wait<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_ns);
  return static_cast<int>(cudaGetLastError());
}

int64_t bounds_violations_update(bool reset) {
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

int launch_unit_all_gather(const Launch& L, const void* shards, void* out, int64_t out_stride,
                           int64_t block0) {
  RepArgs a{static_cast<const uint8_t*>(shards), static_cast<uint8_t*>(out), 2 * out_stride,
            2 * block0, out_stride / kVecElems, kRepUnit, 0};
  return launch_replicate(L, a);
}

int launch_unit_backward(const Launch& Lrs, const void* grads, float* mean, bool sumsq,
                         int64_t rep_stride, int64_t rep_block0, const Launch& Lag,
                         const void* shards, void* out, int64_t out_stride, int64_t block0) {
  KCommon krs = make_common(Lrs);
  krs.stride_bytes = 2 * rep_stride;
  krs.rep_block0 = rep_block0;
  krs.split = 1;
  const KCommon kag = make_common(Lag);
  const RepArgs a{static_cast<const uint8_t*>(shards), static_cast<uint8_t*>(out), 2 * out_stride,
                  2 * block0, out_stride / kVecElems, kRepUnit, 0};
  const int64_t n_rs_tiles = Lrs.tile_end - Lrs.tile_begin;
  const int64_t n_ag_tiles = Lag.tile_end - Lag.tile_begin;
  return with_P(Lrs.plan->P, [&](auto pc) {
    constexpr int P = decltype(pc)::value;
    return with_mesh<P>(Lrs.plan, [&](auto mc) {
      constexpr int M = decltype(mc)::value;
      auto kern = k_unit_backward<P, M>;
      cudaError_t e = ensure_dyn_smem(kern, kUnitBwdSmem);
      if (e != cudaSuccess) return static_cast<int>(e);
      const int64_t cap = resident_ctas(kern, kThreads, kUnitBwdSmem);
      const int sms = sm_count();
      if (cap < 2 || sms <= 0) {
        e = cudaGetLastError();
        return static_cast<int>(e != cudaSuccess ? e : cudaErrorUnknown);
      }
      // one gathering CTA per SM (its one thread keeps a tile's copies in flight),
      // the rest of the resident grid reduce-scatters; DPSYNC_UNIT_AG_CTAS
      // overrides the gathering CTAs' count for tuning sweeps
      static const int64_t ag_env = [] {
        const char* e = std::getenv("DPSYNC_UNIT_AG_CTAS");
        return e ? static_cast<int64_t>(std::atoll(e)) : int64_t(0);
      }();
      int64_t n_ag = ag_env > 0 ? ag_env : sms;
      if (n_ag > n_ag_tiles) n_ag = n_ag_tiles;
      if (n_ag > cap / 2) n_ag = cap / 2;
      int64_t n_rs = cap - n_ag;
      if (n_rs > n_rs_tiles) n_rs = n_rs_tiles;
      if (Lrs.short_ctas && n_rs_tiles + n_ag_tiles <= INT_MAX) {   // one CTA per tile
        n_rs = n_rs_tiles;
        n_ag = n_ag_tiles;
      }
      if (!rep_bulk() && (n_rs_tiles + n_ag_tiles) * kSmallSplit <= INT_MAX) {
        KCommon krs8 = krs, kag8 = kag;
        krs8.split = kag8.split = kSmallSplit;
        const int64_t rs8 = n_rs_tiles * kSmallSplit, ag8 = n_ag_tiles * kSmallSplit;
        if (rs8 + ag8 == 0) return static_cast<int>(cudaSuccess);
        return launch_k(k_unit_backward_small<P, M>, static_cast<int>(rs8 + ag8), kSmallThreads, 0,
                        Lrs.stream, krs8, static_cast<const uint8_t*>(grads), mean, sumsq ? 1 : 0,
                        kag8, a, static_cast<int>(rs8));
      }
      if (n_rs + n_ag == 0) return static_cast<int>(cudaSuccess);   // two empty units
      return launch_k(kern, static_cast<int>(n_rs + n_ag), kThreads, kUnitBwdSmem, Lrs.stream, krs,
                      static_cast<const uint8_t*>(grads), mean, sumsq ? 1 : 0, kag, a,
                      static_cast<int>(n_rs));
    });
  });
}

int launch_all_gather(const Launch& L, void* params) {
  RepArgs a{static_cast<const uint8_t*>(params), static_cast<uint8_t*>(params), 2 * L.plan->stride,
            0, 0, kRepAllGather, 0};
  return launch_replicate(L, a);
}

int launch_broadcast(const Launch& L, void* params, int src) {
  RepArgs a{static_cast<const uint8_t*>(params), static_cast<uint8_t*>(params), 2 * L.plan->stride,
            0, 0, kRepBroadcast, src};
  return launch_replicate(L, a);
}

int launch_zero_fused(const Launch& L, const void* grads, void* params, float* master, float* m,
                      float* v, const AdamScalars& s) {
  const KCommon k = make_common(L);
  return with_P(L.plan->P, [&](auto pc) {
    constexpr int P = decltype(pc)::value;
    return with_mesh<P>(L.plan, [&](auto mc) {
      constexpr int M = decltype(mc)::value;
      // the SMALL kernel (launch_small_or_split)
      return launch_small_or_split(L, 0, k_zero_fused<P, M>, k_zero_fused<P, M, true>,
                                   k_zero_fused<P, M, true, true>,
                                   kSmallThreads, kSmallSplit, k,
                                   static_cast<const uint8_t*>(grads),
                                   static_cast<uint8_t*>(params), master, m, v, s);
    });
  });
}

// rows = P, row_bytes = the replica stride: every replica gets the parameters
// (the all-gather); rows = 1, row_bytes = 0: one flat bf16 array [L] (the ZeRO-3
// shard update).
template <bool DEV_S, int CH, int ST>
int launch_ag(const Launch& L, const KCommon& k, const float* stage, void* params,
              float* master, float* m, float* v, const AdamScalars& s, const float* coefp,
              int rows, int64_t row_bytes) {
  const int64_t Lp = L.plan->L;
  auto kern = k_adamw_all_gather<DEV_S, CH, ST>;
  constexpr size_t smem = tma_smem<CH, ST>();
  cudaError_t e = ensure_dyn_smem(kern, smem);
  if (e != cudaSuccess) return static_cast<int>(e);
  const int64_t cap = resident_ctas(kern, kThreads, smem);
  if (cap <= 0) {
    e = cudaGetLastError();
    return static_cast<int>(e != cudaSuccess ? e : cudaErrorUnknown);
  }
  const int64_t nchunks = (Lp + CH - 1) / CH;
  int64_t g = nchunks < cap ? nchunks : cap;
  if (L.max_ctas > 0 && g > L.max_ctas) g = L.max_ctas;
  return launch_k(kern, static_cast<int>(g), kThreads, smem, L.stream, k, stage,
                  static_cast<uint8_t*>(params), master, m, v, s, Lp, coefp, rows, row_bytes);
}

// The small-CTA pass over the whole plan (k_adamw_all_gather_small).
template <bool DEV_S>
int launch_ag_small(const Launch& L, KCommon k, const float* stage, void* params, float* master,
                    float* m, float* v, const AdamScalars& s, const float* coefp, int rows,
                    int64_t row_bytes) {
  const int64_t n = L.tile_end - L.tile_begin;
  if (n <= 0) return cudaSuccess;
  if (n * kSmallSplit > INT_MAX) return cudaErrorInvalidValue;
  k.split = kSmallSplit;
  return launch_k(k_adamw_all_gather_small<DEV_S>, static_cast<int>(n * kSmallSplit), kSmallThreads,
                  0, L.stream, k, stage, static_cast<uint8_t*>(params), master, m, v, s, coefp,
                  rows, row_bytes);
}

bool ag_bulk() {
  static const bool bulk = std::getenv("DPSYNC_AG_BULK") != nullptr;
  return bulk;
}

int launch_adamw(const Launch& L, const float* grad, float* master, float* m, float* v,
                 void* params, const AdamScalars& s, const float* coefp, bool flat_params,
                 bool dev_scalars) {
  // The ZeRO-3 shard update covers the whole plan and writes one flat bf16 array:
  // the bulk-copy pass with a single output row streams it (no owner rows needed).
  if (flat_params) {
    if (L.tile_begin != 0 || L.tile_end != static_cast<int64_t>(L.plan->tiles.size()))
      return cudaErrorInvalidValue;   // only whole-plan flat updates exist
    if (L.plan->L == 0) return cudaSuccess;
    const KCommon k = make_common(L);
    if (!ag_bulk())
      return dev_scalars ? launch_ag_small<true>(L, k, grad, params, master, m, v, s, coefp, 1, 0)
                         : launch_ag_small<false>(L, k, grad, params, master, m, v, s, coefp, 1, 0);
    return dev_scalars ? launch_ag<true, kTmaChunk, kTmaStages>(L, k, grad, params, master, m, v,
                                                                s, coefp, 1, 0)
                       : launch_ag<false, kTmaChunk, kTmaStages>(L, k, grad, params, master, m,
                                                                 v, s, coefp, 1, 0);
  }
  const int64_t n = L.tile_end - L.tile_begin;
  if (!ag_bulk() && (L.max_ctas <= 0 || L.short_ctas) && n * kSmallSplit <= INT_MAX) {
    if (n <= 0) return cudaSuccess;
    KCommon k = make_common(L);
    k.split = kSmallSplit;
    return launch_k(dev_scalars ? k_adamw_all_gather_small<true, true>
                                : k_adamw_all_gather_small<false, true>,
                    static_cast<int>(n * kSmallSplit), kSmallThreads, 0, L.stream, k, grad,
                    static_cast<uint8_t*>(params), master, m, v, s, coefp, 0, int64_t(0));
  }
  return launch_tiles_split(L, 0, dev_scalars ? k_adamw<true> : k_adamw<false>, make_common(L), grad,
                            master, m, v, static_cast<uint8_t*>(params), s, coefp);
}

int launch_adamw_all_gather(const Launch& L, const float* stage, void* params, float* master,
                            float* m, float* v, const AdamScalars& s, const float* coefp,
                            bool dev_scalars) {
  const KCommon k = make_common(L);
  if (L.plan->L == 0) return cudaSuccess;
  const int rows = L.plan->P;
  const int64_t rb = k.stride_bytes;
  if (!ag_bulk())
    return dev_scalars ? launch_ag_small<true>(L, k, stage, params, master, m, v, s, coefp, rows, rb)
                       : launch_ag_small<false>(L, k, stage, params, master, m, v, s, coefp, rows, rb);
  return dev_scalars ? launch_ag<true, kTmaChunk, kTmaStages>(L, k, stage, params, master, m, v, s,
                                                              coefp, rows, rb)
                     : launch_ag<false, kTmaChunk, kTmaStages>(L, k, stage, params, master, m, v,
                                                               s, coefp, rows, rb);
}

}  // namespace dps

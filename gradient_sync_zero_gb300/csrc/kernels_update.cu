// Sharded AdamW, all-gather / broadcast write-back, and the fused ZeRO-1/2 step.
//
// "ZeRO-1 and ZeRO-2 simply stop after the reduce-scatter, update the shard each
// rank owns, and all-gather the updated parameters" ("Data Parallelism: DDP,
// ZeRO and FSDP", "The three stages").  On one GPU the P replicas are P HBM
// buffers, so the fused kernel performs the three phases per 16-byte vector:
// read P gradient vectors and the owner's fp32 state once, write the state and
// P parameter vectors once.
//
// Roofline (HBM-bound), bytes per element: fused step 2P + 12 read, 12 + 2P
// written; AdamW alone 16 read, 12 + 2 written; all-gather 2 read, 2(P-1) written.
#include "launch.cuh"

namespace dps {

// Sharded AdamW on an fp32 gradient [L]; the owner's replica gets bf16(theta).
__global__ void __launch_bounds__(kThreads)
    k_adamw(KCommon k, const float4* __restrict__ grad, float4* __restrict__ master,
            float4* __restrict__ m, float4* __restrict__ v, uint4* __restrict__ params,
            AdamScalars s, int use_coef) {
  if (!plan_ok(k)) return;
  const float coef = use_coef ? k.hdr->coef : 1.0f;
  for (int64_t tile = k.tile_begin + blockIdx.x; tile < k.tile_end; tile += gridDim.x) {
    const TileDesc d = load_tile(k, tile);
#pragma unroll 1
    for (int j = threadIdx.x; j < d.nvec; j += kThreads) {
      const int64_t x = d.v0 + j;
      const int c = owner_of(d, x);
      float g[8], th[8], mm[8], vv[8];
      load8(grad, x, g);
      load8(master, x, th);
      load8(m, x, mm);
      load8(v, x, vv);
      const bool dec = decay_bit(k.decay, x);
      if (use_coef) {
#pragma unroll
        for (int e = 0; e < 8; ++e) g[e] = __fmul_rn(g[e], coef);
      }
      adamw8(g, th, mm, vv, dec, s);
      store8(master, x, th);
      store8(m, x, mm);
      store8(v, x, vv);
      st_stream(params + c * k.stride_vec + x, pack8_rne(th));
    }
  }
}

// In-place all-gather: the owner's slice of each shard goes to every other replica.
__global__ void __launch_bounds__(kThreads) k_all_gather(KCommon k, uint4* params) {
  if (!plan_ok(k)) return;
  for (int64_t tile = k.tile_begin + blockIdx.x; tile < k.tile_end; tile += gridDim.x) {
    const TileDesc d = load_tile(k, tile);
#pragma unroll 1
    for (int j = threadIdx.x; j < d.nvec; j += kThreads) {
      const int64_t x = d.v0 + j;
      const int c = owner_of(d, x);
      const uint4 val = ld_stream(params + c * k.stride_vec + x);
      for (int r = 0; r < k.P; ++r)
        if (r != c) st_stream(params + r * k.stride_vec + x, val);
    }
  }
}

// Replica `src` to every other replica.
__global__ void __launch_bounds__(kThreads) k_broadcast(KCommon k, uint4* params, int src) {
  if (!plan_ok(k)) return;
  for (int64_t tile = k.tile_begin + blockIdx.x; tile < k.tile_end; tile += gridDim.x) {
    const TileDesc d = load_tile(k, tile);
#pragma unroll 1
    for (int j = threadIdx.x; j < d.nvec; j += kThreads) {
      const int64_t x = d.v0 + j;
      const uint4 val = ld_stream(params + src * k.stride_vec + x);
      for (int r = 0; r < k.P; ++r)
        if (r != src) st_stream(params + r * k.stride_vec + x, val);
    }
  }
}

template <int P>
__device__ __forceinline__ void store_replicas(uint4* params, int64_t stride_vec, int64_t x,
                                               const uint4& val, int p_runtime) {
  if constexpr (P > 0) {
#pragma unroll
    for (int r = 0; r < P; ++r) st_stream(params + r * stride_vec + x, val);
  } else {
    for (int r = 0; r < p_runtime; ++r) st_stream(params + r * stride_vec + x, val);
  }
}

// The whole ZeRO-1/2 step without clipping, one pass.
template <int P>
__global__ void __launch_bounds__(kThreads)
    k_zero_fused(KCommon k, const uint4* __restrict__ grads, uint4* __restrict__ params,
                 float4* __restrict__ master, float4* __restrict__ m, float4* __restrict__ v,
                 AdamScalars s) {
  if (!plan_ok(k)) return;
  for (int64_t tile = k.tile_begin + blockIdx.x; tile < k.tile_end; tile += gridDim.x) {
    const TileDesc d = load_tile(k, tile);
#pragma unroll 1
    for (int j = threadIdx.x; j < d.nvec; j += kThreads) {
      const int64_t x = d.v0 + j;
      const int c = owner_of(d, x);
      float g[8];
      float th[8], mm[8], vv[8];
      if constexpr (P > 0) {
        uint4 rep[P];
#pragma unroll
        for (int r = 0; r < P; ++r) rep[r] = ld_stream(grads + r * k.stride_vec + x);
        load8(master, x, th);
        load8(m, x, mm);
        load8(v, x, vv);
        ring_sum<P>(c, rep, g);
      } else {
        load8(master, x, th);
        load8(m, x, mm);
        load8(v, x, vv);
        ring_sum_runtime(k.P, c, grads, k.stride_vec, x, g);
      }
      scale_mean<P>(g, k.P);
      const bool dec = decay_bit(k.decay, x);
      adamw8(g, th, mm, vv, dec, s);
      store8(master, x, th);
      store8(m, x, mm);
      store8(v, x, vv);
      store_replicas<P>(params, k.stride_vec, x, pack8_rne(th), k.P);
    }
  }
}

// Second pass of the clipped step: AdamW on mean*coef fused with the all-gather.
template <int P>
__global__ void __launch_bounds__(kThreads)
    k_adamw_all_gather(KCommon k, const float4* __restrict__ stage, uint4* __restrict__ params,
                       float4* __restrict__ master, float4* __restrict__ m,
                       float4* __restrict__ v, AdamScalars s) {
  if (!plan_ok(k)) return;
  const float coef = k.hdr->coef;
  for (int64_t tile = k.tile_begin + blockIdx.x; tile < k.tile_end; tile += gridDim.x) {
    const TileDesc d = load_tile(k, tile);
#pragma unroll 1
    for (int j = threadIdx.x; j < d.nvec; j += kThreads) {
      const int64_t x = d.v0 + j;
      float g[8], th[8], mm[8], vv[8];
      load8(stage, x, g);
      load8(master, x, th);
      load8(m, x, mm);
      load8(v, x, vv);
      const bool dec = decay_bit(k.decay, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) g[e] = __fmul_rn(g[e], coef);
      adamw8(g, th, mm, vv, dec, s);
      store8(master, x, th);
      store8(m, x, mm);
      store8(v, x, vv);
      store_replicas<P>(params, k.stride_vec, x, pack8_rne(th), k.P);
    }
  }
}

int launch_adamw(const Launch& L, const float* grad, float* master, float* m, float* v,
                 void* params, const AdamScalars& s, bool use_coef) {
  const KCommon k = make_common(L);
  return launch_tiles(L, k_adamw, k, reinterpret_cast<const float4*>(grad),
                      reinterpret_cast<float4*>(master), reinterpret_cast<float4*>(m),
                      reinterpret_cast<float4*>(v), static_cast<uint4*>(params), s,
                      use_coef ? 1 : 0);
}

int launch_all_gather(const Launch& L, void* params) {
  return launch_tiles(L, k_all_gather, make_common(L), static_cast<uint4*>(params));
}

int launch_broadcast(const Launch& L, void* params, int src) {
  return launch_tiles(L, k_broadcast, make_common(L), static_cast<uint4*>(params), src);
}

int launch_zero_fused(const Launch& L, const void* grads, void* params, float* master, float* m,
                      float* v, const AdamScalars& s) {
  const KCommon k = make_common(L);
  return with_P(L.plan->P, [&](auto pc) {
    constexpr int P = decltype(pc)::value;
    return launch_tiles(L, k_zero_fused<P>, k, static_cast<const uint4*>(grads),
                        static_cast<uint4*>(params), reinterpret_cast<float4*>(master),
                        reinterpret_cast<float4*>(m), reinterpret_cast<float4*>(v), s);
  });
}

int launch_adamw_all_gather(const Launch& L, const float* stage, void* params, float* master,
                            float* m, float* v, const AdamScalars& s) {
  const KCommon k = make_common(L);
  return with_P(L.plan->P, [&](auto pc) {
    constexpr int P = decltype(pc)::value;
    return launch_tiles(L, k_adamw_all_gather<P>, k, reinterpret_cast<const float4*>(stage),
                        static_cast<uint4*>(params), reinterpret_cast<float4*>(master),
                        reinterpret_cast<float4*>(m), reinterpret_cast<float4*>(v), s);
  });
}

}  // namespace dps

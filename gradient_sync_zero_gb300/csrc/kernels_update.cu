// Sharded AdamW, all-gather / broadcast write-back, and the fused ZeRO-1/2 step.
//
// "ZeRO-1 and ZeRO-2 simply stop after the reduce-scatter, update the shard each
// rank owns, and all-gather the updated parameters" ("Data Parallelism: DDP,
// ZeRO and FSDP", "The three stages").  On one GPU the P replicas are P HBM
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
__global__ void __launch_bounds__(kThreads)
    k_adamw(KCommon k, const float* grad, float* master, float* m, float* v, uint8_t* params,
            AdamScalars s, int use_coef) {
  if (!plan_ok(k)) return;
  const float coef = use_coef ? k.hdr->coef : 1.0f;
  for_each_block(k, [&](int64_t, int64_t b, int c) {
    float g[16], th[16], mm[16], vv[16];
    ld_f16(grad, b, g);
    ld_f16(master, b, th);
    ld_f16(m, b, mm);
    ld_f16(v, b, vv);
    const uint32_t dec = decay_bits2(k.decay, b);
    if (use_coef) {
#pragma unroll
      for (int e = 0; e < 16; ++e) g[e] = __fmul_rn(g[e], coef);
    }
    adamw16(g, th, mm, vv, dec, s);
    st_f16(master, b, th);
    st_f16(m, b, mm);
    st_f16(v, b, vv);
    st_blk(params + c * k.stride_bytes + 32 * b, pack16_rne(th));
  });
}

// In-place all-gather: the owner's slice of each shard goes to every other replica.
__global__ void __launch_bounds__(kThreads) k_all_gather(KCommon k, uint8_t* params) {
  if (!plan_ok(k)) return;
  for_each_block(k, [&](int64_t, int64_t b, int c) {
    const Blk val = ld_blk(params + c * k.stride_bytes + 32 * b);
    for (int r = 0; r < k.P; ++r)
      if (r != c) st_blk(params + r * k.stride_bytes + 32 * b, val);
  });
}

// Replica `src` to every other replica.
__global__ void __launch_bounds__(kThreads) k_broadcast(KCommon k, uint8_t* params, int src) {
  if (!plan_ok(k)) return;
  for_each_block(k, [&](int64_t, int64_t b, int) {
    const Blk val = ld_blk(params + src * k.stride_bytes + 32 * b);
    for (int r = 0; r < k.P; ++r)
      if (r != src) st_blk(params + r * k.stride_bytes + 32 * b, val);
  });
}

// The whole ZeRO-1/2 step without clipping, one pass.  The replica blocks are
// loaded and folded first, then the fp32 state is loaded, which bounds the live
// registers to one of the two groups.
template <int P>
__global__ void __launch_bounds__(kThreads)
    k_zero_fused(KCommon k, const uint8_t* grads, uint8_t* params, float* master, float* m,
                 float* v, AdamScalars s) {
  if (!plan_ok(k)) return;
  for_each_block(k, [&](int64_t, int64_t b, int c) {
    float g[16];
    ring_mean16<P>(grads, k.stride_bytes, 32 * b, c, k.P, g);
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
}

// Second pass of the clipped step: AdamW on mean*coef fused with the all-gather.
template <int P>
__global__ void __launch_bounds__(kThreads)
    k_adamw_all_gather(KCommon k, const float* stage, uint8_t* params, float* master, float* m,
                       float* v, AdamScalars s) {
  if (!plan_ok(k)) return;
  const float coef = k.hdr->coef;
  for_each_block(k, [&](int64_t, int64_t b, int) {
    float g[16], th[16], mm[16], vv[16];
    ld_f16(stage, b, g);
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
    store_replicas<P>(params, k.stride_bytes, 32 * b, pack16_rne(th), k.P);
  });
}

int launch_adamw(const Launch& L, const float* grad, float* master, float* m, float* v,
                 void* params, const AdamScalars& s, bool use_coef) {
  return launch_tiles(L, k_adamw, make_common(L), grad, master, m, v,
                      static_cast<uint8_t*>(params), s, use_coef ? 1 : 0);
}

int launch_all_gather(const Launch& L, void* params) {
  return launch_tiles(L, k_all_gather, make_common(L), static_cast<uint8_t*>(params));
}

int launch_broadcast(const Launch& L, void* params, int src) {
  return launch_tiles(L, k_broadcast, make_common(L), static_cast<uint8_t*>(params), src);
}

int launch_zero_fused(const Launch& L, const void* grads, void* params, float* master, float* m,
                      float* v, const AdamScalars& s) {
  const KCommon k = make_common(L);
  return with_P(L.plan->P, [&](auto pc) {
    constexpr int P = decltype(pc)::value;
    return launch_tiles(L, k_zero_fused<P>, k, static_cast<const uint8_t*>(grads),
                        static_cast<uint8_t*>(params), master, m, v, s);
  });
}

int launch_adamw_all_gather(const Launch& L, const float* stage, void* params, float* master,
                            float* m, float* v, const AdamScalars& s) {
  const KCommon k = make_common(L);
  return with_P(L.plan->P, [&](auto pc) {
    constexpr int P = decltype(pc)::value;
    return launch_tiles(L, k_adamw_all_gather<P>, k, stage, static_cast<uint8_t*>(params),
                        master, m, v, s);
  });
}

}  // namespace dps

// Device-side building blocks for the synchronisation kernels (sm_103a).
//
// Work decomposition.  The flat padded index space is cut into 16-byte vectors
// (8 bf16 gradient elements); the plan groups them into tiles of <= 1024
// vectors that never cross a bucket.  A persistent grid (a multiple of the SM
// count) walks the tiles of the requested bucket range round-robin; each of a
// CTA's 256 threads takes every 256th vector of the tile, so every replica
// stream is read and written as whole 512-byte warp transactions.
//
// Every kernel is HBM-bound (<= ~0.4 flop per byte): there is no contraction,
// so no tensor cores; the design goal is to keep enough 16-byte loads in flight
// and touch every byte exactly once.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace dps {

struct KCommon {
  DevHeader* hdr;
  const TileDesc* __restrict__ tiles;
  const uint32_t* __restrict__ decay;
  float* sumsq;          // per tile: sum of squares of the mean as float-float (hi, lo)
  uint64_t plan_id;
  int64_t stride_vec;    // replica stride in 16-byte vectors
  int64_t tile_begin;
  int64_t tile_end;
  int32_t P;             // rank count (used by the runtime-P instantiation)
};

// ---- memory access: streaming (evict-first) 16-byte loads and stores ----
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) { __stcs(p, v); }
__device__ __forceinline__ void st_stream(float4* p, const float4& v) { __stcs(p, v); }

// ---- bf16 <-> fp32 (bf16 -> fp32 is exact; fp32 -> bf16 rounds to nearest even) ----
__device__ __forceinline__ void unpack8(const uint4& q, float (&f)[8]) {
  f[0] = __uint_as_float(q.x << 16);
  f[1] = __uint_as_float(q.x & 0xffff0000u);
  f[2] = __uint_as_float(q.y << 16);
  f[3] = __uint_as_float(q.y & 0xffff0000u);
  f[4] = __uint_as_float(q.z << 16);
  f[5] = __uint_as_float(q.z & 0xffff0000u);
  f[6] = __uint_as_float(q.w << 16);
  f[7] = __uint_as_float(q.w & 0xffff0000u);
}

__device__ __forceinline__ uint32_t pack2_rne(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}

__device__ __forceinline__ uint4 pack8_rne(const float (&f)[8]) {
  return make_uint4(pack2_rne(f[0], f[1]), pack2_rne(f[2], f[3]), pack2_rne(f[4], f[5]),
                    pack2_rne(f[6], f[7]));
}

// ---- ring-ordered reduction ----
// The owner c of a shard receives its sum in the ring's order: rank c+1's
// value first, then c+2, ..., ending with rank c (indices mod P) — the order in
// which "every rank sends one chunk clockwise ... the received chunk is added
// into a local partial sum" ("Data Parallelism: From Parameter Server to Ring All-Reduce",
// sec. 5).  fp32 adds, no reassociation.
template <int P, int C>
__device__ __forceinline__ void ring_sum_fixed(const uint4 (&x)[P], float (&acc)[8]) {
  unpack8(x[(C + 1) % P], acc);
#pragma unroll
  for (int k = 2; k <= P; ++k) {
    float t[8];
    unpack8(x[(C + k) % P], t);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], t[e]);
  }
}

template <int P, int C = 0>
__device__ __forceinline__ void ring_sum(int c, const uint4 (&x)[P], float (&acc)[8]) {
  if constexpr (C + 1 < P) {
    if (c == C) {
      ring_sum_fixed<P, C>(x, acc);
      return;
    }
    ring_sum<P, C + 1>(c, x, acc);
  } else {
    ring_sum_fixed<P, C>(x, acc);
  }
}

// Runtime-P version (P not instantiated): loads inside the loop.
__device__ __forceinline__ void ring_sum_runtime(int P, int c, const uint4* g, int64_t stride_vec,
                                                 int64_t v, float (&acc)[8]) {
  int r = (c + 1) % P;
  unpack8(ld_stream(g + r * stride_vec + v), acc);
  for (int k = 2; k <= P; ++k) {
    r = (c + k) % P;
    float t[8];
    unpack8(ld_stream(g + r * stride_vec + v), t);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], t[e]);
  }
}

// G = sum_i G_i / N ("Data Parallelism: From Parameter Server to Ring All-Reduce", sec. 1): IEEE
// division, which a multiply by 1/P reproduces exactly when P is a power of two.
template <int P>
__device__ __forceinline__ void scale_mean(float (&acc)[8], int p_runtime) {
  if constexpr (P > 0 && (P & (P - 1)) == 0) {
    constexpr float inv = 1.0f / P;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = __fmul_rn(acc[e], inv);
  } else {
    const float fp = static_cast<float>(P > 0 ? P : p_runtime);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = __fdiv_rn(acc[e], fp);
  }
}

// ---- AdamW, torch.optim.AdamW's algorithm ("Distributed Training: Data Parallel,
// Model Parallel and FSDP Strategies", "Inside DDP"), fp32, each op rounded ----
__device__ __forceinline__ void adamw8(const float (&g)[8], float (&th)[8], float (&m)[8],
                                       float (&v)[8], bool decay, const AdamScalars& s) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float t = th[e];
    if (decay) t = __fmul_rn(t, s.wd_factor);
    m[e] = __fadd_rn(__fmul_rn(s.b1, m[e]), __fmul_rn(s.omb1, g[e]));
    v[e] = __fadd_rn(__fmul_rn(s.b2, v[e]), __fmul_rn(s.omb2, __fmul_rn(g[e], g[e])));
    const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v[e]), s.sqrt_bc2), s.eps);
    th[e] = __fsub_rn(t, __fmul_rn(s.step_size, __fdiv_rn(m[e], denom)));
  }
}

__device__ __forceinline__ void load8(const float4* p, int64_t v, float (&f)[8]) {
  const float4 a = ld_stream(p + 2 * v), b = ld_stream(p + 2 * v + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ void store8(float4* p, int64_t v, const float (&f)[8]) {
  st_stream(p + 2 * v, make_float4(f[0], f[1], f[2], f[3]));
  st_stream(p + 2 * v + 1, make_float4(f[4], f[5], f[6], f[7]));
}

__device__ __forceinline__ bool decay_bit(const uint32_t* __restrict__ bits, int64_t v) {
  return (__ldg(bits + (v >> 5)) >> (v & 31)) & 1u;
}

// ---- float-float accumulation (value = hi + lo) for the gradient norm ----
struct FF {
  float hi, lo;
};

// Knuth's TwoSum: s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// acc += x*x, with x*x split exactly as p + q by an FMA (TwoProduct).
__device__ __forceinline__ void ff_add_square(FF& acc, float x) {
  const float p = __fmul_rn(x, x);
  const float q = __fmaf_rn(x, x, -p);
  float s, e;
  two_sum(acc.hi, p, s, e);
  acc.hi = s;
  acc.lo = __fadd_rn(acc.lo, __fadd_rn(e, q));
}

__device__ __forceinline__ FF ff_merge(FF a, FF b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  FF r;
  r.hi = __fadd_rn(s, e);
  r.lo = __fsub_rn(e, __fsub_rn(r.hi, s));
  return r;
}

// Butterfly merge over the 32 lanes; every lane ends with the same value.
__device__ __forceinline__ FF warp_ff_sum(FF a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    FF b;
    b.hi = __shfl_xor_sync(0xffffffffu, a.hi, o);
    b.lo = __shfl_xor_sync(0xffffffffu, a.lo, o);
    a = ff_merge(a, b);
  }
  return a;
}

// Merge the CTA's per-thread partials in a fixed order and store hi, lo at out.
__device__ __forceinline__ void block_ff_store(FF a, FF* warp_part, float* out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  a = warp_ff_sum(a);
  if (lane == 0) warp_part[warp] = a;
  __syncthreads();
  if (warp == 0) {
    FF b = lane < kWarps ? warp_part[lane] : FF{0.0f, 0.0f};
    b = warp_ff_sum(b);
    if (lane == 0) *reinterpret_cast<float2*>(out) = make_float2(b.hi, b.lo);
  }
  __syncthreads();
}

// Plan check: a workspace holding another plan's image is refused.
__device__ __forceinline__ bool plan_ok(const KCommon& k) {
  if (k.hdr->plan_id == k.plan_id) return true;
  if (threadIdx.x == 0) atomicOr(&k.hdr->status, DP_STATUS_PLAN_MISMATCH);
  return false;
}

__device__ __forceinline__ TileDesc load_tile(const KCommon& k, int64_t tile) {
  const int4* p = reinterpret_cast<const int4*>(k.tiles + tile);
  const int4 a = __ldg(p), b = __ldg(p + 1);
  TileDesc d;
  d.v0 = (static_cast<int64_t>(static_cast<uint32_t>(a.y)) << 32) | static_cast<uint32_t>(a.x);
  d.bvoff = (static_cast<int64_t>(static_cast<uint32_t>(a.w)) << 32) | static_cast<uint32_t>(a.z);
  d.nvec = b.x;
  d.svec = b.y;
  d.bucket = b.z;
  d.pad_ = 0;
  return d;
}

// Owner (shard index) of vector v in its bucket.
__device__ __forceinline__ int owner_of(const TileDesc& d, int64_t v) {
  return static_cast<int>(static_cast<uint32_t>(v - d.bvoff) / static_cast<uint32_t>(d.svec));
}

}  // namespace dps

// Device-side building blocks for the synchronisation kernels (sm_103a).
//
// Work decomposition.  The flat padded index space is cut into 32-byte blocks
// of 16 bf16 gradient elements ("pairs" of 16-byte vectors); buckets are padded
// to 16P elements, so a block never straddles two shards.  The plan groups the
// blocks into tiles of <= 512 blocks that never cross a bucket.  A persistent
// grid (SM count x resident CTAs) walks the tiles round-robin; each of a CTA's
// 256 threads takes every 256th block, so every replica stream is read and
// written in 1 KB warp transactions of 256-bit accesses (half the memory
// instructions of 16-byte accesses, which keeps the load/store queues from
// throttling issue).
//
// Every kernel is HBM-bound (<= ~0.6 flop per byte): there is no contraction,
// so no tensor cores; the aim is enough bytes in flight and every byte touched
// exactly once.  All global accesses are streaming (.cs: evict-first), since no
// byte is reused within a step.
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
  float* sumsq;          // per sub-tile: sum of squares of the mean as float-float (hi, lo)
  float* fin;            // the norm pass's per-CTA float-float sums
  uint64_t plan_id;
  int64_t stride_bytes;  // replica stride in bytes
  int64_t tile_begin;
  int64_t tile_end;
  int32_t P;             // rank count (used by the runtime-P instantiation)
  int32_t R;             // mesh: replicate groups (1 = flat ring)
  int32_t S;             // mesh: shard ranks per group (P = R * S)
  int64_t rep_block0;    // replica buffers start at this 32-byte block (unit buffers)
  int32_t split;         // CTAs per tile (1; 2 or kSmallSplit for launches with few tiles)
  int32_t pad_;
  // A launch inside one bucket carries that bucket in its parameters, so its
  // tile descriptors are computed, not loaded (one dependent load fewer per
  // small per-bucket launch).  one_nvec = 0: descriptors come from the table.
  int64_t one_v0;        // the bucket's first 16-byte vector
  int64_t one_tile0;     // the bucket's first tile
  int32_t one_nvec;      // the bucket's length in vectors
  int32_t one_svec;      // its shard length in vectors
  int32_t one_bucket;
  int32_t pad2_;
};

// ---- optional index checks (built with -DDPSYNC_CHECKED) ----
// The checked build tests every tile descriptor, block index, owner and replica
// index against the plan before the access it guards.  A failed check is counted
// in this translation unit's device counter and the access is skipped or sent to
// replica 0 — never a trap.  In the normal build the checks compile away.
#ifdef DPSYNC_CHECKED
static __device__ unsigned long long g_bounds_violations;
__device__ __forceinline__ bool bounds_ok(bool ok) {
  if (!ok) atomicAdd(&g_bounds_violations, 1ull);
  return ok;
}
#define DP_IN_BOUNDS(cond) (::dps::bounds_ok(cond))
#else
#define DP_IN_BOUNDS(cond) (true)
#endif

// ---- 256-bit streaming accesses (sm_100-family ld/st .v8.b32) ----
// Every global access is volatile asm, so the compiler keeps them in program
// order (loads of a block are issued before its stores, never re-issued).
struct Blk {  // 16 bf16 = 32 bytes
  uint32_t w[8];
};

__device__ __forceinline__ Blk ld_blk(const uint8_t* p) {
  Blk r;
  asm volatile("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]),
                 "=r"(r.w[5]), "=r"(r.w[6]), "=r"(r.w[7])
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_blk(uint8_t* p, const Blk& v) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]),
               "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]),
               "r"(v.w[7])
               : "memory");
}

// 8 fp32 (32 bytes)
__device__ __forceinline__ void ld_f8(const float* p, float* f) {
  asm volatile("ld.global.cs.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3]), "=f"(f[4]), "=f"(f[5]),
                 "=f"(f[6]), "=f"(f[7])
               : "l"(p));
}

__device__ __forceinline__ void st_f8(float* p, const float* f) {
  asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(f[0]),
               "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7])
               : "memory");
}

// 16 fp32 of block b of an fp32 [L] array (elements 16b .. 16b+15)
__device__ __forceinline__ void ld_f16(const float* base, int64_t b, float (&f)[16]) {
  ld_f8(base + 16 * b, f);
  ld_f8(base + 16 * b + 8, f + 8);
}

__device__ __forceinline__ void st_f16(float* base, int64_t b, const float (&f)[16]) {
  st_f8(base + 16 * b, f);
  st_f8(base + 16 * b + 8, f + 8);
}

// ---- bf16 <-> fp32 (bf16 -> fp32 is exact; fp32 -> bf16 rounds to nearest even) ----
__device__ __forceinline__ void unpack16(const Blk& q, float (&f)[16]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = __uint_as_float(q.w[i] << 16);
    f[2 * i + 1] = __uint_as_float(q.w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint32_t pack2_rne(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}

__device__ __forceinline__ Blk pack16_rne(const float (&f)[16]) {
  Blk b;
#pragma unroll
  for (int i = 0; i < 8; ++i) b.w[i] = pack2_rne(f[2 * i], f[2 * i + 1]);
  return b;
}

// ---- ring-ordered reduction + mean ----
// The owner c of a shard receives its sum in the ring's order: rank c+1's value
// first, then c+2, ..., ending with rank c (indices mod P) — the order a ring
// builds it in, each rank passing a chunk to its neighbour, which adds it to its
// own running sum ("Data Parallelism: From Parameter Server to Ring All-Reduce",
// sec. 5).  The replicas are loaded directly in that order (the
// owner is known from the block index), up to 8 blocks in flight per thread,
// and folded with fp32 adds in the same order.  Then G = sum / N (sec. 1) as an
// IEEE division, which a multiply by 1/P reproduces exactly for P = 2^k.
// KC: replica blocks in flight per thread (8, or 16 for the latency-bound small
// launches, where one round of loads instead of two is worth the registers).
template <int P, int KC = 8>
__device__ __forceinline__ void ring_fold_chunk(const uint8_t* g, int64_t stride_bytes,
                                                int64_t byte_off, int np, int r_first, int k0,
                                                float (&acc)[16]) {
  constexpr int K = (P > 0 && P < KC) ? P : KC;
  Blk x[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    if (P == 0 && k0 + k >= np) break;
    int r = r_first + k0 + k;
    if (r >= np) r -= np;
    if (!DP_IN_BOUNDS(r >= 0 && r < np)) r = 0;
    x[k] = ld_blk(g + r * stride_bytes + byte_off);
  }
#pragma unroll
  for (int k = 0; k < K; ++k) {
    if (P == 0 && k0 + k >= np) break;
    if (k0 + k == 0) {
      unpack16(x[k], acc);
    } else {
      float t[16];
      unpack16(x[k], t);
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] = __fadd_rn(acc[e], t[e]);
    }
  }
}

template <int P, int KC = 8>
__device__ __forceinline__ void ring_mean16(const uint8_t* g, int64_t stride_bytes,
                                            int64_t byte_off, int c, int p_rt,
                                            float (&acc)[16]) {
  constexpr int K = (P > 0 && P < KC) ? P : KC;
  const int np = P > 0 ? P : p_rt;
  const int r_first = (c + 1 == np) ? 0 : c + 1;
  if constexpr (P > 0) {
#pragma unroll
    for (int k0 = 0; k0 < P; k0 += K)
      ring_fold_chunk<P, KC>(g, stride_bytes, byte_off, np, r_first, k0, acc);
  } else {
#pragma unroll 1
    for (int k0 = 0; k0 < np; k0 += K)
      ring_fold_chunk<P, KC>(g, stride_bytes, byte_off, np, r_first, k0, acc);
  }
  if constexpr (P > 0 && (P & (P - 1)) == 0) {
    constexpr float inv = 1.0f / P;
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = __fmul_rn(acc[e], inv);
  } else {
    const float fp = static_cast<float>(np);
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = __fdiv_rn(acc[e], fp);
  }
}

// Hybrid R x S mesh: the sum of element i of shard s in sub-chunk j is
//   sum over groups g = j+1, ..., j (mod R) of
//     [sum over members s' = s+1, ..., s (mod S) of grad(g*S + s')[i]]
// — a ring reduce-scatter inside each group, then a ring all-reduce of the shard
// across groups ("4.1 Data parallelism in depth", sec. 6.3 HYBRID_SHARD).  The P
// blocks are loaded in that order (8 in flight per thread) and folded left to
// right, the inner sum restarting at each group boundary.
template <int P>
__device__ __forceinline__ void mesh_mean16(const uint8_t* g, int64_t stride_bytes,
                                            int64_t byte_off, int s, int j, int R, int S,
                                            int p_rt, float (&acc)[16]) {
  const int np = P > 0 ? P : p_rt;
  float inner[16];
  int gi = 0, si = 0;
  int grp = (j + 1 == R) ? 0 : j + 1;    // current group in fold order
  int mem = (s + 1 == S) ? 0 : s + 1;    // current member in fold order
#pragma unroll 1
  for (int k0 = 0; k0 < np; k0 += 8) {
    Blk x[8];
    int gg = grp, mm = mem, sii = si;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k0 + k >= np) break;
      int rr = gg * S + mm;
      if (!DP_IN_BOUNDS(rr >= 0 && rr < np)) rr = 0;
      x[k] = ld_blk(g + rr * stride_bytes + byte_off);
      if (++sii == S) {
        sii = 0;
        gg = (gg + 1 == R) ? 0 : gg + 1;
      }
      mm = (mm + 1 == S) ? 0 : mm + 1;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k0 + k >= np) break;
      float t[16];
      unpack16(x[k], t);
      if (si == 0) {
#pragma unroll
        for (int e = 0; e < 16; ++e) inner[e] = t[e];
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) inner[e] = __fadd_rn(inner[e], t[e]);
      }
      if (++si == S) {
        si = 0;
        if (gi == 0) {
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[e] = inner[e];
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[e] = __fadd_rn(acc[e], inner[e]);
        }
        ++gi;
      }
    }
    grp = gg;
    mem = mm;
  }
  const float fp = static_cast<float>(np);
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = __fdiv_rn(acc[e], fp);
}

// The same fold with P and the group size S known at compile time (P a multiple
// of 8 and of S): the rank order is fixed by (s, j) alone, so the loop unrolls
// like the flat ring's, 8 blocks in flight, whole groups per batch.
template <int P, int S>
__device__ __forceinline__ void mesh_mean16_ct(const uint8_t* g, int64_t stride_bytes,
                                               int64_t byte_off, int s, int j, float (&acc)[16]) {
  static_assert(P % 8 == 0 && 8 % S == 0 && P % S == 0, "whole groups per batch of 8");
  constexpr int R = P / S;
  float inner[16];
#pragma unroll
  for (int k0 = 0; k0 < P; k0 += 8) {
    Blk x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int q = k0 + k;                       // position in the fold order
      int grp = j + 1 + q / S;                    // < 2R
      grp -= (grp >= R) ? R : 0;
      int mem = s + 1 + q % S;                    // < 2S
      mem -= (mem >= S) ? S : 0;
      int rr = grp * S + mem;
      if (!DP_IN_BOUNDS(rr >= 0 && rr < P)) rr = 0;
      x[k] = ld_blk(g + rr * stride_bytes + byte_off);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int q = k0 + k;
      float t[16];
      unpack16(x[k], t);
      if (q % S == 0) {
#pragma unroll
        for (int e = 0; e < 16; ++e) inner[e] = t[e];
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) inner[e] = __fadd_rn(inner[e], t[e]);
      }
      if (q % S == S - 1) {
        if (q / S == 0) {
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[e] = inner[e];
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[e] = __fadd_rn(acc[e], inner[e]);
        }
      }
    }
  }
  constexpr float inv = 1.0f / P;                 // P is a power of two: exact
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = __fmul_rn(acc[e], inv);
}

// The mean of block b for its owner: MS = 0 flat ring, MS > 0 hybrid mesh with
// group size MS fixed at compile time, MS < 0 hybrid mesh with the shape read
// at run time.  s = shard index in the bucket (the owner rank on a flat ring).
template <int P, int MS, int KC = 8>
__device__ __forceinline__ void block_mean16(const KCommon& k, const uint8_t* g, int64_t b,
                                             const TileDesc& d, int s, float (&acc)[16]) {
  if constexpr (MS == 0) {
    ring_mean16<P, KC>(g, k.stride_bytes, 32 * (b - k.rep_block0), s, k.P, acc);
  } else {
    const uint32_t within = static_cast<uint32_t>(2 * b - d.bvoff) % static_cast<uint32_t>(d.svec);
    const int j = static_cast<int>(within / (static_cast<uint32_t>(d.svec) / k.R));
    if constexpr (MS > 0) {
      mesh_mean16_ct<P, MS>(g, k.stride_bytes, 32 * (b - k.rep_block0), s, j, acc);
    } else {
      mesh_mean16<P>(g, k.stride_bytes, 32 * (b - k.rep_block0), s, j, k.R, k.S, k.P, acc);
    }
  }
}

__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// Accumulation fused with the reduction: replica r's value is bf16(acc_r + micro_r)
// (what dp_accumulate would have stored), folded in ring order as in ring_mean16.
template <int P>
__device__ __forceinline__ void ring_mean16_accum(const uint8_t* acc, const uint8_t* micro,
                                                  int64_t stride_bytes, int64_t byte_off, int c,
                                                  int p_rt, float (&out)[16]) {
  constexpr int K = (P > 0 && P < 4) ? P : 4;
  const int np = P > 0 ? P : p_rt;
  const int r_first = (c + 1 == np) ? 0 : c + 1;
#pragma unroll
  for (int k0 = 0; k0 < (P > 0 ? P : kMaxP); k0 += K) {
    if (k0 >= np) break;
    Blk x[K], y[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      if (k0 + k >= np) break;
      int r = r_first + k0 + k;
      if (r >= np) r -= np;
      if (!DP_IN_BOUNDS(r >= 0 && r < np)) r = 0;
      x[k] = ld_blk(acc + r * stride_bytes + byte_off);
      y[k] = ld_blk(micro + r * stride_bytes + byte_off);
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
      if (k0 + k >= np) break;
      float a[16], b[16];
      unpack16(x[k], a);
      unpack16(y[k], b);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float t = bf16_round(__fadd_rn(a[e], b[e]));
        out[e] = (k0 + k == 0) ? t : __fadd_rn(out[e], t);
      }
    }
  }
  const float fp = static_cast<float>(np);
#pragma unroll
  for (int e = 0; e < 16; ++e) out[e] = __fdiv_rn(out[e], fp);
}

// The ring with bf16 partial sums: each hop rounds its fp32 add to bf16.
template <int P>
__device__ __forceinline__ void ring_mean16_bf16wire(const uint8_t* g, int64_t stride_bytes,
                                                     int64_t byte_off, int c, int p_rt,
                                                     float (&out)[16]) {
  constexpr int K = (P > 0 && P < 8) ? P : 8;
  const int np = P > 0 ? P : p_rt;
  const int r_first = (c + 1 == np) ? 0 : c + 1;
#pragma unroll
  for (int k0 = 0; k0 < (P > 0 ? P : kMaxP); k0 += K) {
    if (k0 >= np) break;
    Blk x[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      if (k0 + k >= np) break;
      int r = r_first + k0 + k;
      if (r >= np) r -= np;
      if (!DP_IN_BOUNDS(r >= 0 && r < np)) r = 0;
      x[k] = ld_blk(g + r * stride_bytes + byte_off);
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
      if (k0 + k >= np) break;
      float t[16];
      unpack16(x[k], t);
#pragma unroll
      for (int e = 0; e < 16; ++e) out[e] = (k0 + k == 0) ? t[e] : bf16_round(__fadd_rn(out[e], t[e]));
    }
  }
  const float fp = static_cast<float>(np);
#pragma unroll
  for (int e = 0; e < 16; ++e) out[e] = __fdiv_rn(out[e], fp);
}

// Store one block into every replica.
template <int P>
__device__ __forceinline__ void store_replicas(uint8_t* base, int64_t stride_bytes,
                                               int64_t byte_off, const Blk& val, int p_rt) {
  if constexpr (P > 0) {
#pragma unroll
    for (int r = 0; r < P; ++r) st_blk(base + r * stride_bytes + byte_off, val);
  } else {
#pragma unroll 1
    for (int r = 0; r < p_rt; ++r) st_blk(base + r * stride_bytes + byte_off, val);
  }
}

// ---- AdamW, torch.optim.AdamW's algorithm ("Distributed Training: Data Parallel,
// Model Parallel and FSDP Strategies", "Inside DDP"), fp32, each op rounded ----
__device__ __forceinline__ void adamw1(float g, float& th, float& m, float& v, bool decay,
                                       const AdamScalars& s) {
  float t = th;
  if (decay) t = __fmul_rn(t, s.wd_factor);
  m = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
  v = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
  const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), s.sqrt_bc2), s.eps);
  th = __fsub_rn(t, __fmul_rn(s.step_size, __fdiv_rn(m, denom)));
}

// 16 elements: the first 8 belong to 16-byte vector 2b, the last 8 to 2b+1,
// each with its own decay bit.
__device__ __forceinline__ void adamw16(const float (&g)[16], float (&th)[16], float (&m)[16],
                                        float (&v)[16], uint32_t dec2, const AdamScalars& s) {
#pragma unroll
  for (int e = 0; e < 16; ++e) adamw1(g[e], th[e], m[e], v[e], (dec2 >> (e >> 3)) & 1u, s);
}

// Decay bits of the two 16-byte vectors of block b (vector 2b is even, so both
// bits sit in the same 32-bit word).
__device__ __forceinline__ uint32_t decay_bits2(const uint32_t* __restrict__ bits, int64_t b) {
  const int64_t v = 2 * b;
  return (__ldg(bits + (v >> 5)) >> (v & 31)) & 3u;
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

// Norm partials of one tile: one float-float value per sub-tile of
// kSubTileBlocks consecutive 32-byte blocks, formed the same way whatever the
// launch's shape: each lane's squares of its block, a butterfly over the warp's
// 32 lanes (32 consecutive blocks), then the two warps of the sub-tile merged,
// lower blocks first.  ss[p] is the thread's sum for its p-th block of the tile
// (blocks j0 + p * jstep, j0 = this CTA's first block in the tile plus
// threadIdx.x); out receives the tile's kSubTiles (hi, lo) pairs, every slot
// this CTA covers written (zero for blocks past the tile's end).
template <int NT>
__device__ __forceinline__ void subtile_ff_store(const FF (&ss)[2], int cta_j0, int jstep,
                                                 FF* warp_part, float* out) {
  constexpr int W = NT / 32;
  constexpr int kTileBlocks = kTileVec / 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int npass = (kTileBlocks + jstep - 1) / jstep;   // 2 (256 threads, one CTA) or 1
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    if (p < npass) {
      const FF a = warp_ff_sum(ss[p]);
      if (lane == 0) warp_part[p * W + warp] = a;
    }
  }
  __syncthreads();
  constexpr int pairs = W / 2;                           // sub-tiles per pass
  if (static_cast<int>(threadIdx.x) < npass * pairs) {
    const int p = threadIdx.x / pairs, q = threadIdx.x % pairs;
    const FF m = ff_merge(warp_part[p * W + 2 * q], warp_part[p * W + 2 * q + 1]);
    const int sub = (cta_j0 + p * jstep) / kSubTileBlocks + q;
    if (DP_IN_BOUNDS(sub >= 0 && sub < kSubTiles))
      *reinterpret_cast<float2*>(out + 2 * sub) = make_float2(m.hi, m.lo);
  }
  __syncthreads();
}

// ---- bulk asynchronous copies (cp.async.bulk) and mbarriers ----
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: polls until the phase completes or limit_ns of the global timer
// have passed (1 s unless told otherwise); false on timeout.  2^32 polls end it
// as well, should the timer not advance.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1; i != 0; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && global_ns() - t0 > limit_ns) return false;
  }
  return false;
}

// global -> shared, completion counted on `bar` (bytes and addresses 16-byte multiples)
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// shared -> global, tracked by the issuing thread's bulk groups
__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_addr(smem_src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to bulk copies.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Plan check: a workspace holding another plan's image is refused.
//
// Every library kernel starts here.  The kernels are launched as programmatic
// dependents of the previous kernel in their stream, so the launch is prepared
// while that kernel runs and its CTAs are dispatched as that kernel's CTAs exit
// (no early trigger: a persistent grid is never placed on SMs still busy with
// its predecessor).  The wait below returns once the predecessor has finished
// and its writes are visible (at once for an ordinary launch), and only then is
// global memory touched.
__device__ __forceinline__ bool plan_ok(const KCommon& k) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (k.hdr->plan_id == k.plan_id) return true;
  if (threadIdx.x == 0) atomicOr(&k.hdr->status, DP_STATUS_PLAN_MISMATCH);
  return false;
}

// Start of a SMALL kernel: after the dependency wait, the plan id is loaded, but
// not waited for.  A launch inside one bucket (k.one_nvec > 0) takes its tile
// descriptors from its parameters, so its first replica loads go out beside the
// id and plan_matches() gates the stores: with another plan's image in the
// workspace it still reads only the caller's buffers of this plan.  A launch over
// several buckets reads descriptors from the workspace's table and so checks the
// id first.
// (Letting the next launch be scheduled early from here, griddepcontrol
// .launch_dependents at entry, was measured: per-bucket launches of 64 KiB
// buckets unchanged, of 1 MiB buckets 17% slower; not kept.)
__device__ __forceinline__ uint64_t plan_id_deferred(const KCommon& k) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  uint64_t id;
  asm volatile("ld.global.u64 %0, [%1];" : "=l"(id) : "l"(&k.hdr->plan_id) : "memory");
  return id;
}

__device__ __forceinline__ bool plan_matches(const KCommon& k, uint64_t id) {
  if (id == k.plan_id) return true;
  if (threadIdx.x == 0) atomicOr(&k.hdr->status, DP_STATUS_PLAN_MISMATCH);
  return false;
}

__device__ __forceinline__ TileDesc load_tile(const KCommon& k, int64_t tile) {
  if (k.one_nvec > 0) {   // one bucket: tiles of kTileVec vectors from its start
    const int64_t i = tile - k.one_tile0;
    const int64_t rest = static_cast<int64_t>(k.one_nvec) - i * kTileVec;
    TileDesc d;
    d.v0 = k.one_v0 + i * kTileVec;
    d.bvoff = k.one_v0;
    d.nvec = static_cast<int32_t>(rest < kTileVec ? rest : kTileVec);
    d.svec = k.one_svec;
    d.bucket = k.one_bucket;
    d.pad_ = 0;
    return d;
  }
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

// Checked build: the descriptor lies inside the plan (even start and count,
// within [0, n_vec), a shard of at least one block).  The same for every thread
// of the CTA, so a skipped tile is skipped by all of them.
__device__ __forceinline__ bool tile_ok(const KCommon& k, int64_t tile, const TileDesc& d) {
  return DP_IN_BOUNDS(tile >= 0 && tile < k.hdr->n_tiles && d.v0 >= 0 && (d.v0 & 1) == 0 &&
                      d.nvec >= 0 && (d.nvec & 1) == 0 && d.v0 + d.nvec <= k.hdr->n_vec &&
                      d.svec >= 2 && d.bvoff >= 0 && d.bvoff <= d.v0);
}

// Owner (shard index) of 16-byte vector v in its bucket.
__device__ __forceinline__ int owner_of(const TileDesc& d, int64_t v) {
  return static_cast<int>(static_cast<uint32_t>(v - d.bvoff) / static_cast<uint32_t>(d.svec));
}

// Loop over the 32-byte blocks of the CTA's tiles: f(tile, block index b,
// owner c).  Tiles start at even 16-byte vectors and hold an even count.  With
// k.split = s > 1 (launches over few tiles) s CTAs share each tile, taking
// turns at runs of NT blocks (NT = threads per CTA), so every thread of a small
// launch moves one block.
template <bool SPLIT = true, int NT = kThreads, class F>
__device__ __forceinline__ void for_each_block(const KCommon& k, F&& f) {
  // the common case (split 1) keeps constant strides; splits are for small launches
  // (SPLIT = false: a kernel always launched unsplit compiles the first walk only)
  auto walk = [&](int64_t t0, int64_t tstride, int j0, int jstep) {
    for (int64_t tile = t0; tile < k.tile_end; tile += tstride) {
      const TileDesc d = load_tile(k, tile);
      if (!tile_ok(k, tile, d)) continue;
      const int nblk = d.nvec >> 1;
      const int64_t b0 = d.v0 >> 1;
#pragma unroll 1
      for (int j = j0; j < nblk; j += jstep) {
        const int64_t b = b0 + j;
        const int c = owner_of(d, 2 * b);
        if (!DP_IN_BOUNDS(c >= 0 && c < k.S)) continue;
        f(tile, b, c);
      }
    }
  };
  if (!SPLIT || k.split == 1) {
    walk(k.tile_begin + blockIdx.x, gridDim.x, threadIdx.x, NT);
  } else {
    const int64_t cta_tile = blockIdx.x / k.split;
    walk(k.tile_begin + cta_tile, gridDim.x / k.split,
         static_cast<int>(blockIdx.x - k.split * cta_tile) * NT + threadIdx.x, k.split * NT);
  }
}

// Same loop, giving the body the tile descriptor: f(desc, block b, owner c);
// CTA `cta` of `ncta` (a kernel may give the walk to part of its grid).
template <bool SPLIT = true, int NT = kThreads, class F>
__device__ __forceinline__ void for_each_block2_of(const KCommon& k, int64_t cta, int64_t ncta,
                                                   F&& f) {
  auto walk = [&](int64_t t0, int64_t tstride, int j0, int jstep) {
    for (int64_t tile = t0; tile < k.tile_end; tile += tstride) {
      const TileDesc d = load_tile(k, tile);
      if (!tile_ok(k, tile, d)) continue;
      const int nblk = d.nvec >> 1;
      const int64_t b0 = d.v0 >> 1;
#pragma unroll 1
      for (int j = j0; j < nblk; j += jstep) {
        const int64_t b = b0 + j;
        const int c = owner_of(d, 2 * b);
        if (!DP_IN_BOUNDS(c >= 0 && c < k.S)) continue;
        f(d, b, c);
      }
    }
  };
  if (!SPLIT || k.split == 1) {
    walk(k.tile_begin + cta, ncta, threadIdx.x, NT);
  } else {
    const int64_t cta_tile = cta / k.split;
    walk(k.tile_begin + cta_tile, ncta / k.split,
         static_cast<int>(cta - k.split * cta_tile) * NT + threadIdx.x, k.split * NT);
  }
}

template <bool SPLIT = true, int NT = kThreads, class F>
__device__ __forceinline__ void for_each_block2(const KCommon& k, F&& f) {
  // the common case (split 1) keeps constant strides; splits are for small launches
  auto walk = [&](int64_t t0, int64_t tstride, int j0, int jstep) {
    for (int64_t tile = t0; tile < k.tile_end; tile += tstride) {
      const TileDesc d = load_tile(k, tile);
      if (!tile_ok(k, tile, d)) continue;
      const int nblk = d.nvec >> 1;
      const int64_t b0 = d.v0 >> 1;
#pragma unroll 1
      for (int j = j0; j < nblk; j += jstep) {
        const int64_t b = b0 + j;
        const int c = owner_of(d, 2 * b);
        if (!DP_IN_BOUNDS(c >= 0 && c < k.S)) continue;
        f(d, b, c);
      }
    }
  };
  if (!SPLIT || k.split == 1) {
    walk(k.tile_begin + blockIdx.x, gridDim.x, threadIdx.x, NT);
  } else {
    const int64_t cta_tile = blockIdx.x / k.split;
    walk(k.tile_begin + cta_tile, gridDim.x / k.split,
         static_cast<int>(blockIdx.x - k.split * cta_tile) * NT + threadIdx.x, k.split * NT);
  }
}

// The reduce-scatter's tile walk for CTA `cta` of `ncta` (a kernel may give the
// role to part of its grid): shard c of each block's bucket gets the fp32 mean
// rank c owns; with sumsq, kSubTiles float-float partials of sum(mean^2) per
// tile (subtile_ff_store).  The partials are accumulated in float-float
// arithmetic (value = hi + lo): each square is split exactly into p + q with the
// FMA-based TwoProduct and added with Knuth's TwoSum (Ogita, Rump & Oishi,
// "Accurate sum and dot product", SIAM J. Sci. Comput. 26(6), 2005).  The norm
// is then good to ~1e-15 relative, so its fp32 clip coefficient rounds like one
// computed from the exact sum.  The partials are formed per sub-tile in a fixed
// order, so the norm does not depend on the grid, the CTA shape (NT threads,
// k.split CTAs per tile: 256 x 1 or 64 x kSmallSplit with sumsq) or on how the
// bucket range is split into launches.  ACC: the last micro-batch of gradient
// accumulation fused in (flat plans, always unsplit); SMALL: stores gated on
// the plan id `id` loaded beside the first loads.  warp_part: 2 * NT / 32 FF of
// shared memory.
template <int P, int MS, bool ACC, bool SMALL, int NT = kThreads>
__device__ __forceinline__ void rs_tiles(const KCommon& k, const uint8_t* g, float* mean, int sumsq,
                                         const uint8_t* micro, uint64_t id, int64_t cta,
                                         int64_t ncta, FF* warp_part) {
  auto walk = [&](int64_t t0, int64_t tstride, int j0, int jstep) {
    for (int64_t tile = t0; tile < k.tile_end; tile += tstride) {
      const TileDesc d = load_tile(k, tile);
      if (!tile_ok(k, tile, d)) continue;
      const int nblk = d.nvec >> 1;
      const int64_t b0 = d.v0 >> 1;
      FF ss[2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};
      int pass = 0;
#pragma unroll 1
      for (int j = j0; j < nblk; j += jstep, ++pass) {
        const int64_t b = b0 + j;
        const int c = owner_of(d, 2 * b);
        if (!DP_IN_BOUNDS(c >= 0 && c < k.S)) continue;
        float acc[16];
        if constexpr (ACC) {
          ring_mean16_accum<P>(g, micro, k.stride_bytes, 32 * b, c, k.P, acc);
        } else {
          block_mean16<P, MS, SMALL ? 16 : 8>(k, g, b, d, c, acc);
        }
        if (SMALL && id != k.plan_id) continue;
        st_f16(mean, b, acc);
        if (sumsq) {
          FF& sp = ss[pass & 1];
#pragma unroll
          for (int e = 0; e < 16; ++e) ff_add_square(sp, acc[e]);
        }
      }
      if (sumsq && (!SMALL || id == k.plan_id))
        subtile_ff_store<NT>(ss, j0 - static_cast<int>(threadIdx.x), jstep, warp_part,
                             k.sumsq + 2 * kSubTiles * tile);
    }
  };
  if (ACC || k.split == 1) {
    walk(k.tile_begin + cta, ncta, threadIdx.x, NT);
  } else {
    const int64_t cta_tile = cta / k.split;
    walk(k.tile_begin + cta_tile, ncta / k.split,
         static_cast<int>(cta - k.split * cta_tile) * NT + threadIdx.x, k.split * NT);
  }
}

}  // namespace dps

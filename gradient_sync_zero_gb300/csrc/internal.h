// Internal declarations shared by the library's translation units (host
// planner, C-ABI, kernel launchers).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "dpsync.h"

namespace dps {

constexpr int kThreads = 256;                 // threads per CTA
// The small-CTA launch shape (the default for the step's kernels): CTAs of
// kSmallThreads threads, kSmallSplit per tile, one CTA per piece of a tile for the
// whole launch, so one thread moves one 32-byte block with all of its loads in
// flight and the launch's loads and stores spread over the whole GPU.
constexpr int kSmallThreads = 64;
constexpr int kSmallSplit = 8;
// Norm partials: one float-float pair per sub-tile of kSubTileBlocks 32-byte
// blocks (1024 elements), kSubTiles per tile, so that CTAs of kSmallThreads
// threads can form them exactly as a whole-tile CTA does.
constexpr int kSubTileBlocks = 64;
constexpr int kSubTiles = 8;
// The norm pass: each CTA merges up to kFinPerCta consecutive partials, at most
// kFinMaxCtas CTAs (the count depends only on the number of partials).
constexpr int kFinPerCta = 8192;
constexpr int kFinMaxCtas = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kVecElems = 8;                  // bf16 elements per 16-byte vector
constexpr int kPairElems = 16;                // bf16 elements per 32-byte (256-bit) access
constexpr int kTileVec = 1024;                // vectors per tile (8192 elements)
constexpr int kTileElems = kTileVec * kVecElems;
static_assert(kSubTiles * kSubTileBlocks * 2 == kTileVec, "sub-tiles cover a tile");
static_assert(kSmallSplit * kSmallThreads * 2 == kTileVec, "a small CTA's threads cover a sub-tile pair");
constexpr int kMaxP = 64;
constexpr uint64_t kMagic = 0x31304e5953435044ull;  // "DPCSYN01"

// One work tile: a run of <= kTileVec vectors inside one bucket.
struct TileDesc {
  int64_t v0;      // first vector (flat vector index)
  int64_t bvoff;   // first vector of the tile's bucket
  int32_t nvec;    // vectors in the tile
  int32_t svec;    // shard length of the bucket (len / S), in vectors (>= 2)
  int32_t bucket;
  int32_t pad_;
};
static_assert(sizeof(TileDesc) == 32, "TileDesc is one 32-byte sector");

// AdamW's per-step scalars, formed on the host (in double, rounded once).
struct AdamScalars {
  float wd_factor, b1, omb1, b2, omb2, step_size, sqrt_bc2, eps;
};
constexpr uint32_t kAdamTag = 0x574d4441u;   // "ADMW": the header holds scalars

// Header at the start of the workspace (device).  The first part is uploaded
// with the plan; the results part is written by kernels.
struct DevHeader {
  uint64_t magic;
  uint64_t plan_id;
  int64_t n_vec;
  int64_t n_tiles;
  int32_t n_buckets;
  int32_t P;
  int32_t R, S;
  int64_t off_tiles;      // byte offsets of the arrays inside the workspace
  int64_t off_btile;      // int64 [n_buckets+1]: first tile of each bucket
  int64_t off_decay;      // uint32 [ceil(n_vec/32)]
  int64_t off_sumsq;      // float2 [n_tiles * kSubTiles]: per-sub-tile sum of mean^2, hi + lo (scratch)
  int64_t off_stage;      // float [L] (scratch)
  int64_t off_fin;        // float2 [kFinMaxCtas]: the norm pass's per-CTA sums (scratch)
  int64_t reserved_[2];
  // ---- written by kernels ----
  double norm2;
  double norm;
  float coef;
  int32_t status;
  AdamScalars adam;       // set by dp_set_adamw_cfg, read by the update kernels when
  uint32_t adam_tag;      // called without a cfg (graph-captured steps); kAdamTag
  int32_t pad3_;
  uint32_t fin_count;     // norm pass: CTAs done (the last one resets it to 0)
  uint32_t pad4_;
  int64_t reserved2_;
};
static_assert(sizeof(DevHeader) % 64 == 0, "header keeps the arrays aligned");
// the results part's layout is public (include/dpsync.h, DP_WS_*_OFFSET)
static_assert(offsetof(DevHeader, norm2) == DP_WS_NORM2_OFFSET, "public offset of norm2");
static_assert(offsetof(DevHeader, norm) == DP_WS_NORM_OFFSET, "public offset of norm");
static_assert(offsetof(DevHeader, coef) == DP_WS_COEF_OFFSET, "public offset of coef");
static_assert(offsetof(DevHeader, status) == DP_WS_STATUS_OFFSET, "public offset of status");

struct Plan {
  int32_t P = 0;
  int32_t R = 1, S = 0;   // mesh: R groups x S shard ranks (P = R * S)
  int64_t bucket_bytes = 0;
  int64_t n_params = 0;
  int64_t L = 0;
  int64_t stride = 0;
  uint64_t id = 0;
  std::vector<int64_t> sizes;
  std::vector<uint8_t> decay;
  std::vector<int64_t> t_off;
  std::vector<int32_t> t_bucket;
  std::vector<int64_t> b_off, b_len;
  std::vector<int64_t> b_tile0;     // [n_buckets+1]
  std::vector<TileDesc> tiles;
  std::vector<uint32_t> decay_bits; // bit per 16-byte vector
  // workspace layout
  int64_t table_bytes = 0;
  int64_t workspace_bytes = 0;
  std::vector<uint8_t> image;       // host copy of the device image (table_bytes)
};

// AdamW's per-step scalars from a cfg (checked; DP_EINVAL with a message naming fn).
int adam_scalars(const char* fn, const dp_adamw_cfg* cfg, AdamScalars* s);

// Thread-local last-error text (dp_last_error); fail() records and returns code.
int fail(int code, const std::string& msg);
void clear_error();
const char* last_error_text();
const Plan* as_plan(const dp_plan* p);

// ---- kernel launchers (kernels_*.cu) ----
struct Launch {
  const Plan* plan;
  uint8_t* ws;          // workspace base (device)
  int64_t tile_begin;   // [tile_begin, tile_end)
  int64_t tile_end;
  void* stream;
  int max_ctas = 0;     // > 0: cap on the grid (leave SMs to concurrent work)
  bool short_ctas = false;   // one short-lived CTA per tile (piece) instead of a
                             // persistent grid; max_ctas is then ignored
};

// The launch shape set for `stream` by dp_stream_set_launch (host registry).
bool stream_short_ctas(void* stream);

// Each returns a cudaError_t value (0 = success).
int launch_reduce_scatter(const Launch& L, const void* grads, float* mean, bool sumsq,
                          int64_t rep_stride = 0, int64_t rep_block0 = 0);
int launch_unit_all_gather(const Launch& L, const void* shards, void* out, int64_t out_stride,
                           int64_t block0);
// One launch: the reduce-scatter of Lrs's unit (replicas at rep_stride, first
// block rep_block0) and the gather of Lag's unit into out (both non-empty).
int launch_unit_backward(const Launch& Lrs, const void* grads, float* mean, bool sumsq,
                         int64_t rep_stride, int64_t rep_block0, const Launch& Lag,
                         const void* shards, void* out, int64_t out_stride, int64_t block0);
int launch_allreduce(const Launch& L, void* grads);
int launch_accumulate(const Launch& L, void* acc, const void* micro);
int launch_selftest_wait(int32_t* status, uint64_t limit_ns, void* stream);
// Checked build: failed index checks counted by each kernel translation unit
// (-1 in the normal build, -2 if the counter cannot be read).
int64_t bounds_violations_reduce(bool reset);
int64_t bounds_violations_update(bool reset);
int launch_allreduce_accum(const Launch& L, void* acc, const void* micro);
int launch_reduce_scatter_accum(const Launch& L, const void* acc, const void* micro, float* mean,
                                bool sumsq);
int launch_allreduce_bf16wire(const Launch& L, void* grads);
int launch_norm_finalize(const Launch& L, double max_norm);
// coefp: device fp32 clip coefficient multiplying the gradient (NULL = 1).
int launch_adamw(const Launch& L, const float* grad, float* master, float* m, float* v,
                 void* params, const AdamScalars& s, const float* coefp, bool flat_params = false,
                 bool dev_scalars = false);
int launch_all_gather(const Launch& L, void* params);
int launch_broadcast(const Launch& L, void* params, int src);
int launch_zero_fused(const Launch& L, const void* grads, void* params, float* master, float* m,
                      float* v, const AdamScalars& s);
int launch_adamw_all_gather(const Launch& L, const float* stage, void* params, float* master,
                            float* m, float* v, const AdamScalars& s, const float* coefp,
                            bool dev_scalars = false);

}  // namespace dps

// Host bucket planner and the device plan image.
//
// Bucket rule ("4.1 Data parallelism in depth", sec. 4.2: gradients are packed
// into ~25 MB buckets in reverse compute order, one collective per bucket;
// bucket_cap_mb is the knob): tensors are taken from the last to the first,
// each in a 16-byte aligned slot; a bucket that already holds data is closed
// when the next slot would push it past the cap; tensors are never split; a
// closed bucket is padded to a multiple of 16P so that its P shards (sec. 5.1:
// each rank's buffer is cut into one chunk per rank) are whole 32-byte blocks of 16 bf16 — the
// unit of one 256-bit access, which therefore never straddles two owners.
//
// The device image lets one launch walk any bucket range: a table of work
// tiles (<= 1024 vectors, never crossing a bucket), each bucket's first tile,
// and one weight-decay bit per 16-byte vector.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdio>
#include <cstring>
#include <new>
#include <random>

#include "internal.h"

namespace dps {

namespace {
thread_local std::string g_last_error;

int64_t round_up(int64_t x, int64_t q) { return (x + q - 1) / q * q; }

uint64_t fresh_plan_id() {
  static std::atomic<uint64_t> counter{0};
  std::random_device rd;
  uint64_t x = (static_cast<uint64_t>(rd()) << 32) ^ rd();
  x ^= static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count());
  x ^= (++counter) * 0x9E3779B97F4A7C15ull;
  return x | 1;  // never 0
}
}  // namespace

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}
void clear_error() { g_last_error.clear(); }
const char* last_error_text() { return g_last_error.c_str(); }

const Plan* as_plan(const dp_plan* p) { return reinterpret_cast<const Plan*>(p); }

namespace {

// Assign tensors to buckets.  Returns false on bad input.
bool assign_buckets(Plan& pl) {
  const int n = static_cast<int>(pl.sizes.size());
  const int64_t cap_elems = pl.bucket_bytes / 2;
  const int64_t align = static_cast<int64_t>(kPairElems) * pl.P;
  pl.t_off.assign(n, 0);
  pl.t_bucket.assign(n, -1);
  pl.b_off.clear();
  pl.b_len.clear();
  int64_t bucket_start = 0;  // flat offset of the open bucket
  int64_t fill = 0;          // elements used in the open bucket
  int32_t nb = 0;            // buckets opened so far
  for (int t = n - 1; t >= 0; --t) {
    const int64_t need = round_up(pl.sizes[t], kVecElems);
    const bool have_open = nb > static_cast<int32_t>(pl.b_off.size());
    if (have_open && fill > 0 && fill + need > cap_elems) {
      pl.b_off.push_back(bucket_start);
      pl.b_len.push_back(round_up(fill, align));
      bucket_start += pl.b_len.back();
      fill = 0;
    }
    if (nb == static_cast<int32_t>(pl.b_off.size())) ++nb;  // open a new bucket
    pl.t_bucket[t] = nb - 1;
    pl.t_off[t] = bucket_start + fill;
    fill += need;
  }
  if (nb > static_cast<int32_t>(pl.b_off.size())) {
    pl.b_off.push_back(bucket_start);
    pl.b_len.push_back(round_up(fill, align));
    bucket_start += pl.b_len.back();
  }
  pl.L = bucket_start;
  return true;
}

void build_tiles(Plan& pl) {
  const int nb = static_cast<int>(pl.b_off.size());
  pl.tiles.clear();
  pl.b_tile0.assign(nb + 1, 0);
  for (int b = 0; b < nb; ++b) {
    pl.b_tile0[b] = static_cast<int64_t>(pl.tiles.size());
    const int64_t bv = pl.b_off[b] / kVecElems;
    const int64_t nv = pl.b_len[b] / kVecElems;
    const int32_t sv = static_cast<int32_t>(nv / pl.S);
    for (int64_t v = 0; v < nv; v += kTileVec) {
      TileDesc d{};
      d.v0 = bv + v;
      d.bvoff = bv;
      d.nvec = static_cast<int32_t>(std::min<int64_t>(kTileVec, nv - v));
      d.svec = sv;
      d.bucket = b;
      pl.tiles.push_back(d);
    }
  }
  pl.b_tile0[nb] = static_cast<int64_t>(pl.tiles.size());
}

void build_decay_bits(Plan& pl) {
  const int64_t n_vec = pl.L / kVecElems;
  pl.decay_bits.assign((n_vec + 31) / 32, 0u);
  for (size_t t = 0; t < pl.sizes.size(); ++t) {
    if (!pl.decay[t] || pl.sizes[t] == 0) continue;
    const int64_t v0 = pl.t_off[t] / kVecElems;
    const int64_t v1 = (pl.t_off[t] + pl.sizes[t] + kVecElems - 1) / kVecElems;
    for (int64_t v = v0; v < v1; ++v) pl.decay_bits[v >> 5] |= 1u << (v & 31);
  }
}

void build_image(Plan& pl) {
  DevHeader h{};
  h.magic = kMagic;
  h.plan_id = pl.id;
  h.n_vec = pl.L / kVecElems;
  h.n_tiles = static_cast<int64_t>(pl.tiles.size());
  h.n_buckets = static_cast<int32_t>(pl.b_off.size());
  h.P = pl.P;
  h.R = pl.R;
  h.S = pl.S;
  int64_t off = round_up(sizeof(DevHeader), 256);
  h.off_tiles = off;
  off = round_up(off + h.n_tiles * static_cast<int64_t>(sizeof(TileDesc)), 256);
  h.off_btile = off;
  off = round_up(off + (h.n_buckets + 1) * 8, 256);
  h.off_decay = off;
  off = round_up(off + static_cast<int64_t>(pl.decay_bits.size()) * 4, 256);
  pl.table_bytes = off;
  h.off_sumsq = off;
  off = round_up(off + h.n_tiles * 8 * kSubTiles, 256);
  h.off_fin = off;
  off = round_up(off + int64_t(8) * kFinMaxCtas, 256);
  h.off_stage = off;
  off = round_up(off + pl.L * 4, 256);
  pl.workspace_bytes = off;
  h.coef = 1.0f;

  pl.image.assign(pl.table_bytes, 0);
  std::memcpy(pl.image.data(), &h, sizeof(h));
  if (!pl.tiles.empty())
    std::memcpy(pl.image.data() + h.off_tiles, pl.tiles.data(), pl.tiles.size() * sizeof(TileDesc));
  std::memcpy(pl.image.data() + h.off_btile, pl.b_tile0.data(), pl.b_tile0.size() * 8);
  if (!pl.decay_bits.empty())
    std::memcpy(pl.image.data() + h.off_decay, pl.decay_bits.data(), pl.decay_bits.size() * 4);
}

// 64-bit FNV-1a over the layout, each value as 8 little-endian bytes, so the
// result does not depend on the host's byte order or word size.
class LayoutHash {
 public:
  void add(int64_t v) {
    const uint64_t u = static_cast<uint64_t>(v);
    for (int i = 0; i < 8; ++i) {
      h_ ^= (u >> (8 * i)) & 0xffu;
      h_ *= 0x100000001b3ull;   // FNV-1a 64-bit prime
    }
  }
  uint64_t value() const { return h_; }

 private:
  uint64_t h_ = 0xcbf29ce484222325ull;   // FNV-1a 64-bit offset basis
};

uint64_t layout_fingerprint(const Plan& pl) {
  LayoutHash h;
  h.add(0x31544e4946504c44ll);   // format tag ("DLPFINT1")
  h.add(pl.P);
  h.add(pl.R);
  h.add(pl.S);
  h.add(pl.L);
  h.add(static_cast<int64_t>(pl.sizes.size()));
  for (size_t t = 0; t < pl.sizes.size(); ++t) {
    h.add(pl.sizes[t]);
    h.add(pl.decay[t]);
    h.add(pl.t_off[t]);
    h.add(pl.t_bucket[t]);
  }
  h.add(static_cast<int64_t>(pl.b_off.size()));
  for (size_t b = 0; b < pl.b_off.size(); ++b) {
    h.add(pl.b_off[b]);
    h.add(pl.b_len[b]);
  }
  return h.value();
}

}  // namespace
}  // namespace dps

using namespace dps;

extern "C" {

int dp_plan_buckets_mesh(const int64_t* sizes, const uint8_t* decay, int32_t n_tensors,
                         int64_t bucket_bytes, int32_t R, int32_t S, int64_t replica_stride,
                         dp_plan** out) {
  clear_error();
  if (!out) return fail(DP_EINVAL, "dp_plan_buckets: out is NULL");
  *out = nullptr;
  if (n_tensors < 0 || (n_tensors > 0 && !sizes))
    return fail(DP_EINVAL, "dp_plan_buckets: bad tensor list");
  if (R < 1 || S < 1 || static_cast<int64_t>(R) * S > kMaxP)
    return fail(DP_EINVAL, "dp_plan_buckets: need R, S >= 1 and P = R*S in 1..64");
  const int32_t P = R * S;
  if (bucket_bytes < 2) return fail(DP_EINVAL, "dp_plan_buckets: bucket_bytes must be >= 2");
  Plan* pl = new (std::nothrow) Plan();
  if (!pl) return fail(DP_ENOMEM, "dp_plan_buckets: out of host memory");
  try {
    pl->P = P;
    pl->R = R;
    pl->S = S;
    pl->bucket_bytes = bucket_bytes;
    pl->sizes.assign(sizes, sizes + n_tensors);
    pl->decay.assign(n_tensors, 1);
    for (int t = 0; t < n_tensors; ++t) {
      if (sizes[t] < 0) {
        delete pl;
        return fail(DP_EINVAL, "dp_plan_buckets: negative tensor size");
      }
      pl->n_params += sizes[t];
      if (decay) pl->decay[t] = decay[t] ? 1 : 0;
    }
    assign_buckets(*pl);
    // vector indices are kept in 32 bits inside a bucket and 63 bits overall
    for (size_t b = 0; b < pl->b_len.size(); ++b)
      if (pl->b_len[b] / kVecElems >= (int64_t(1) << 31)) {
        delete pl;
        return fail(DP_EINVAL, "dp_plan_buckets: a bucket exceeds 2^31 vectors");
      }
    const int64_t min_stride = round_up(pl->L, 128);
    if (replica_stride == 0) {
      pl->stride = min_stride + 128;
    } else {
      if (replica_stride < pl->L || replica_stride % 128) {
        delete pl;
        return fail(DP_EINVAL, "dp_plan_buckets: replica_stride must be >= L and a multiple of 128");
      }
      pl->stride = replica_stride;
    }
    pl->id = fresh_plan_id();
    build_tiles(*pl);
    build_decay_bits(*pl);
    build_image(*pl);
  } catch (const std::bad_alloc&) {
    delete pl;
    return fail(DP_ENOMEM, "dp_plan_buckets: out of host memory");
  }
  *out = reinterpret_cast<dp_plan*>(pl);
  return DP_OK;
}

int dp_plan_buckets_ex(const int64_t* sizes, const uint8_t* decay, int32_t n_tensors,
                       int64_t bucket_bytes, int32_t P, int64_t replica_stride, dp_plan** out) {
  if (P < 1 || P > kMaxP) {
    clear_error();
    if (out) *out = nullptr;
    return fail(DP_EINVAL, "dp_plan_buckets: P must be in 1..64");
  }
  return dp_plan_buckets_mesh(sizes, decay, n_tensors, bucket_bytes, 1, P, replica_stride, out);
}

int dp_plan_buckets(const int64_t* sizes, const uint8_t* decay, int32_t n_tensors,
                    int64_t bucket_bytes, int32_t P, dp_plan** out) {
  return dp_plan_buckets_ex(sizes, decay, n_tensors, bucket_bytes, P, 0, out);
}

int dp_plan_info(const dp_plan* plan, dp_plan_info_t* out) {
  clear_error();
  const Plan* pl = as_plan(plan);
  if (!pl || !out) return fail(DP_EINVAL, "dp_plan_info: NULL argument");
  out->n_params = pl->n_params;
  out->padded_len = pl->L;
  out->replica_stride = pl->stride;
  out->bucket_bytes = pl->bucket_bytes;
  out->n_tensors = static_cast<int32_t>(pl->sizes.size());
  out->n_buckets = static_cast<int32_t>(pl->b_off.size());
  out->P = pl->P;
  out->tile_elems = kTileElems;
  out->R = pl->R;
  out->S = pl->S;
  out->pad_ = 0;
  out->n_tiles = static_cast<int64_t>(pl->tiles.size());
  out->table_bytes = pl->table_bytes;
  out->workspace_bytes = pl->workspace_bytes;
  return DP_OK;
}

int dp_plan_tensor(const dp_plan* plan, int32_t t, int32_t* bucket, int64_t* offset) {
  clear_error();
  const Plan* pl = as_plan(plan);
  if (!pl) return fail(DP_EINVAL, "dp_plan_tensor: NULL plan");
  if (t < 0 || t >= static_cast<int32_t>(pl->sizes.size()))
    return fail(DP_EINVAL, "dp_plan_tensor: tensor index out of range");
  if (bucket) *bucket = pl->t_bucket[t];
  if (offset) *offset = pl->t_off[t];
  return DP_OK;
}

int dp_plan_bucket(const dp_plan* plan, int32_t b, int64_t* offset, int64_t* padded_len,
                   int64_t* shard_len) {
  clear_error();
  const Plan* pl = as_plan(plan);
  if (!pl) return fail(DP_EINVAL, "dp_plan_bucket: NULL plan");
  if (b < 0 || b >= static_cast<int32_t>(pl->b_off.size()))
    return fail(DP_EINVAL, "dp_plan_bucket: bucket index out of range");
  if (offset) *offset = pl->b_off[b];
  if (padded_len) *padded_len = pl->b_len[b];
  if (shard_len) *shard_len = pl->b_len[b] / pl->S;
  return DP_OK;
}

int dp_plan_fingerprint(const dp_plan* plan, uint64_t* out) {
  clear_error();
  const Plan* pl = as_plan(plan);
  if (!pl || !out) return fail(DP_EINVAL, "dp_plan_fingerprint: NULL argument");
  *out = layout_fingerprint(*pl);
  return DP_OK;
}

int dp_plan_check_match(const dp_plan* plan, const uint64_t* fingerprints, int32_t n_ranks) {
  clear_error();
  const Plan* pl = as_plan(plan);
  if (!pl) return fail(DP_EINVAL, "dp_plan_check_match: NULL plan");
  if (n_ranks < 0 || (n_ranks > 0 && !fingerprints))
    return fail(DP_EINVAL, "dp_plan_check_match: bad fingerprint list");
  const uint64_t mine = layout_fingerprint(*pl);
  for (int32_t r = 0; r < n_ranks; ++r) {
    if (fingerprints[r] != mine) {
      char buf[160];
      std::snprintf(buf, sizeof(buf),
                    "dp_plan_check_match: rank %d's bucket layout differs (fingerprint %016llx, "
                    "this plan %016llx)",
                    r, static_cast<unsigned long long>(fingerprints[r]),
                    static_cast<unsigned long long>(mine));
      return fail(DP_EPLAN, buf);
    }
  }
  return DP_OK;
}

void dp_plan_free(dp_plan* plan) { delete reinterpret_cast<Plan*>(plan); }

const char* dp_last_error(void) { return dps::last_error_text(); }

int dp_version(void) { return 2; }

}  // extern "C"

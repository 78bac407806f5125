// Checkpoint and resume of the sharded optimizer state.
//
// The fp32 master weights and AdamW moments are the only state a ZeRO-1/2 step
// carries from one step to the next ("Data Parallelism: DDP, ZeRO and FSDP",
// "The three stages": the optimizer state is what ZeRO shards first; "4.1 Data
// parallelism in depth", sec. 7: 12 of the 16 bytes per parameter), together
// with the step count t that the bias corrections use.  A checkpoint stores them
// in tensor order, without the plan's padding, so it can be loaded into a plan
// with another bucket size, rank count or mesh (an elastic restart): each
// element's value and the step are all a plan needs to continue.
//
// File layout (little-endian):
//   header (80 bytes): magic "DPSYNCK1", u32 version = 1, u32 arrays (bit 0
//     master, bit 1 m, bit 2 v), i64 n_tensors, i64 n_params, i64 step,
//     u64 checksum, i32 P, R, S of the saving plan, i32 0, i64 bucket_bytes,
//     8 zero bytes;
//   i64 sizes[n_tensors];
//   for each array present, in the order master, m, v: f32 [n_params], tensor
//     0 first, each tensor's elements in order.
// checksum: 64-bit FNV-1a over the bytes after the header taken as 8-byte
// little-endian words (the last one zero-padded), each step
// h = (h ^ w) * 0x100000001b3, starting from 0xcbf29ce484222325.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "internal.h"

namespace dps {
namespace {

constexpr char kCkptMagic[8] = {'D', 'P', 'S', 'Y', 'N', 'C', 'K', '1'};
constexpr uint32_t kCkptVersion = 1;

struct CkptHeader {
  char magic[8];
  uint32_t version;
  uint32_t arrays;
  int64_t n_tensors;
  int64_t n_params;
  int64_t step;
  uint64_t checksum;
  int32_t P, R, S, pad_;
  int64_t bucket_bytes;
  int64_t reserved_;
};
static_assert(sizeof(CkptHeader) == 80, "checkpoint header is 80 bytes");

class Hasher {
 public:
  void update(const void* p, size_t n) {
    const uint8_t* b = static_cast<const uint8_t*>(p);
    while (n > 0 && fill_ > 0) {  // finish a partial word
      word_[fill_++] = *b++;
      --n;
      if (fill_ == 8) mix_word();
    }
    while (n >= 8) {
      uint64_t w;
      std::memcpy(&w, b, 8);
      mix(w);
      b += 8;
      n -= 8;
    }
    while (n > 0) {
      word_[fill_++] = *b++;
      --n;
    }
  }
  uint64_t digest() {
    if (fill_ > 0) {
      while (fill_ < 8) word_[fill_++] = 0;
      mix_word();
    }
    return h_;
  }

 private:
  void mix(uint64_t w) { h_ = (h_ ^ w) * 0x100000001b3ull; }
  void mix_word() {
    uint64_t w = 0;
    for (int i = 7; i >= 0; --i) w = (w << 8) | word_[i];
    mix(w);
    fill_ = 0;
  }
  uint64_t h_ = 0xcbf29ce484222325ull;
  uint8_t word_[8] = {};
  int fill_ = 0;
};

struct File {
  FILE* f = nullptr;
  ~File() {
    if (f) std::fclose(f);
  }
};

bool host_mode(int32_t flags) { return (flags & DP_CKPT_HOST) != 0; }

// dst[0..n) <- src (host), on the device or the host.
int put(float* dst, const float* src, int64_t n, bool host, cudaStream_t s) {
  if (n == 0) return DP_OK;
  if (host) {
    std::memcpy(dst, src, static_cast<size_t>(n) * 4);
    return DP_OK;
  }
  cudaError_t e = cudaMemcpyAsync(dst, src, static_cast<size_t>(n) * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? DP_OK : fail(DP_ECUDA, std::string("dp_checkpoint_load: ") + cudaGetErrorString(e));
}

int get(float* dst, const float* src, int64_t n, bool host, cudaStream_t s) {
  if (n == 0) return DP_OK;
  if (host) {
    std::memcpy(dst, src, static_cast<size_t>(n) * 4);
    return DP_OK;
  }
  cudaError_t e = cudaMemcpyAsync(dst, src, static_cast<size_t>(n) * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? DP_OK : fail(DP_ECUDA, std::string("dp_checkpoint_save: ") + cudaGetErrorString(e));
}

int64_t max_tensor(const Plan& pl) {
  int64_t m = 0;
  for (int64_t s : pl.sizes) m = s > m ? s : m;
  return m;
}

}  // namespace
}  // namespace dps

using namespace dps;

extern "C" {

int dp_checkpoint_save(const dp_plan* plan, const char* path, const float* master, const float* m,
                       const float* v, int64_t step, int32_t flags, void* stream) {
  clear_error();
  const Plan* pl = as_plan(plan);
  if (!pl) return fail(DP_EINVAL, "dp_checkpoint_save: NULL plan");
  if (!path || !*path) return fail(DP_EINVAL, "dp_checkpoint_save: empty path");
  if (flags & ~DP_CKPT_HOST) return fail(DP_EINVAL, "dp_checkpoint_save: unknown flags");
  const float* arr[3] = {master, m, v};
  uint32_t arrays = 0;
  for (int i = 0; i < 3; ++i)
    if (arr[i]) arrays |= 1u << i;
  if (!arrays) return fail(DP_EINVAL, "dp_checkpoint_save: no array to save");
  if (step < 0) return fail(DP_EINVAL, "dp_checkpoint_save: step must be >= 0");
  const bool host = host_mode(flags);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!host) {
    const cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(DP_ECUDA, std::string("dp_checkpoint_save: ") + cudaGetErrorString(e));
  }
  const std::string tmp = std::string(path) + ".tmp";
  File fh;
  fh.f = std::fopen(tmp.c_str(), "wb");
  if (!fh.f) return fail(DP_EINVAL, "dp_checkpoint_save: cannot open " + tmp + " for writing");
  CkptHeader h{};
  std::memcpy(h.magic, kCkptMagic, 8);
  h.version = kCkptVersion;
  h.arrays = arrays;
  h.n_tensors = static_cast<int64_t>(pl->sizes.size());
  h.n_params = pl->n_params;
  h.step = step;
  h.P = pl->P;
  h.R = pl->R;
  h.S = pl->S;
  h.bucket_bytes = pl->bucket_bytes;
  Hasher hs;
  bool ok = std::fwrite(&h, sizeof h, 1, fh.f) == 1;
  const size_t nt = pl->sizes.size();
  if (ok && nt) {
    ok = std::fwrite(pl->sizes.data(), 8, nt, fh.f) == nt;
    hs.update(pl->sizes.data(), 8 * nt);
  }
  std::vector<float> buf;
  try {
    buf.resize(static_cast<size_t>(max_tensor(*pl)));
  } catch (const std::bad_alloc&) {
    std::fclose(fh.f);
    fh.f = nullptr;
    std::remove(tmp.c_str());
    return fail(DP_ENOMEM, "dp_checkpoint_save: out of host memory");
  }
  for (int i = 0; i < 3 && ok; ++i) {
    if (!arr[i]) continue;
    for (size_t t = 0; t < nt && ok; ++t) {
      const int64_t n = pl->sizes[t];
      if (n == 0) continue;
      const int rc = get(buf.data(), arr[i] + pl->t_off[t], n, host, s);
      if (rc) {
        std::fclose(fh.f);
        fh.f = nullptr;
        std::remove(tmp.c_str());
        return rc;
      }
      hs.update(buf.data(), static_cast<size_t>(n) * 4);
      ok = std::fwrite(buf.data(), 4, static_cast<size_t>(n), fh.f) == static_cast<size_t>(n);
    }
  }
  h.checksum = hs.digest();
  ok = ok && std::fseek(fh.f, 0, SEEK_SET) == 0 && std::fwrite(&h, sizeof h, 1, fh.f) == 1;
  ok = ok && std::fflush(fh.f) == 0;
  const int closed = std::fclose(fh.f);
  fh.f = nullptr;
  if (!ok || closed != 0) {
    std::remove(tmp.c_str());
    return fail(DP_EINVAL, "dp_checkpoint_save: write to " + tmp + " failed");
  }
  if (std::rename(tmp.c_str(), path) != 0) {
    std::remove(tmp.c_str());
    return fail(DP_EINVAL, std::string("dp_checkpoint_save: cannot rename to ") + path);
  }
  return DP_OK;
}

int dp_checkpoint_load(const dp_plan* plan, const char* path, float* master, float* m, float* v,
                       int64_t* step, int32_t flags, void* stream) {
  clear_error();
  const Plan* pl = as_plan(plan);
  if (!pl) return fail(DP_EINVAL, "dp_checkpoint_load: NULL plan");
  if (!path || !*path) return fail(DP_EINVAL, "dp_checkpoint_load: empty path");
  if (flags & ~DP_CKPT_HOST) return fail(DP_EINVAL, "dp_checkpoint_load: unknown flags");
  File fh;
  fh.f = std::fopen(path, "rb");
  if (!fh.f) return fail(DP_EINVAL, std::string("dp_checkpoint_load: cannot open ") + path);
  CkptHeader h{};
  if (std::fread(&h, sizeof h, 1, fh.f) != 1 || std::memcmp(h.magic, kCkptMagic, 8) != 0)
    return fail(DP_EINVAL, std::string("dp_checkpoint_load: ") + path + " is not a checkpoint");
  if (h.version != kCkptVersion)
    return fail(DP_EINVAL, "dp_checkpoint_load: unsupported version " + std::to_string(h.version));
  if ((h.arrays & ~7u) || h.n_tensors < 0 || h.n_params < 0 || h.step < 0)
    return fail(DP_EINVAL, "dp_checkpoint_load: corrupt header");
  const size_t nt = pl->sizes.size();
  if (h.n_tensors != static_cast<int64_t>(nt) || h.n_params != pl->n_params)
    return fail(DP_EPLAN, "dp_checkpoint_load: the file holds " + std::to_string(h.n_tensors) +
                              " tensors / " + std::to_string(h.n_params) + " parameters, the plan " +
                              std::to_string(nt) + " / " + std::to_string(pl->n_params));
  std::vector<int64_t> sizes(nt);
  if (nt && std::fread(sizes.data(), 8, nt, fh.f) != nt)
    return fail(DP_EINVAL, "dp_checkpoint_load: truncated file");
  for (size_t t = 0; t < nt; ++t)
    if (sizes[t] != pl->sizes[t])
      return fail(DP_EPLAN, "dp_checkpoint_load: tensor " + std::to_string(t) + " has " +
                                std::to_string(sizes[t]) + " elements in the file and " +
                                std::to_string(pl->sizes[t]) + " in the plan");
  float* dst[3] = {master, m, v};
  for (int i = 0; i < 3; ++i)
    if (dst[i] && !(h.arrays & (1u << i)))
      return fail(DP_EINVAL, std::string("dp_checkpoint_load: the file has no ") +
                                 (i == 0 ? "master" : i == 1 ? "m" : "v") + " array");
  // the file's length must match what the header announces
  int n_arrays = 0;
  for (int i = 0; i < 3; ++i) n_arrays += (h.arrays >> i) & 1;
  const long long want = static_cast<long long>(sizeof h) + 8LL * static_cast<long long>(nt) +
                         4LL * n_arrays * h.n_params;
  if (std::fseek(fh.f, 0, SEEK_END) != 0 || std::ftell(fh.f) != want)
    return fail(DP_EINVAL, "dp_checkpoint_load: file length does not match its header");
  if (std::fseek(fh.f, static_cast<long>(sizeof h + 8 * nt), SEEK_SET) != 0)
    return fail(DP_EINVAL, "dp_checkpoint_load: seek failed");
  const bool host = host_mode(flags);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // padding slots of the destination hold zeros
  for (int i = 0; i < 3; ++i) {
    if (!dst[i] || pl->L == 0) continue;
    if (host) {
      std::memset(dst[i], 0, static_cast<size_t>(pl->L) * 4);
    } else {
      const cudaError_t e = cudaMemsetAsync(dst[i], 0, static_cast<size_t>(pl->L) * 4, s);
      if (e != cudaSuccess) return fail(DP_ECUDA, std::string("dp_checkpoint_load: ") + cudaGetErrorString(e));
    }
  }
  Hasher hs;
  if (nt) hs.update(sizes.data(), 8 * nt);
  std::vector<float> buf;
  try {
    buf.resize(static_cast<size_t>(max_tensor(*pl)));
  } catch (const std::bad_alloc&) {
    return fail(DP_ENOMEM, "dp_checkpoint_load: out of host memory");
  }
  for (int i = 0; i < 3; ++i) {
    if (!(h.arrays & (1u << i))) continue;
    for (size_t t = 0; t < nt; ++t) {
      const int64_t n = pl->sizes[t];
      if (n == 0) continue;
      if (std::fread(buf.data(), 4, static_cast<size_t>(n), fh.f) != static_cast<size_t>(n))
        return fail(DP_EINVAL, "dp_checkpoint_load: truncated file");
      hs.update(buf.data(), static_cast<size_t>(n) * 4);
      if (dst[i]) {
        const int rc = put(dst[i] + pl->t_off[t], buf.data(), n, host, s);
        if (rc) return rc;
      }
    }
  }
  if (!host) {
    const cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(DP_ECUDA, std::string("dp_checkpoint_load: ") + cudaGetErrorString(e));
  }
  if (hs.digest() != h.checksum)
    return fail(DP_EINVAL, "dp_checkpoint_load: checksum mismatch (the file is corrupt; the "
                           "destination arrays hold partial data)");
  if (step) *step = h.step;
  return DP_OK;
}

}  // extern "C"

// Oracle for the data-parallel gradient synchronisation step.
//
// TEST INFRASTRUCTURE ONLY.  Plain, slow, obviously-correct CPU code that the
// GPU path is checked against.  Only the tests, the smoke check and the bench's
// CPU-baseline leg may load it; the product path never does.  It shares no code,
// header, table or helper with the CUDA library.
//
// What it computes (sources are the four pages on data parallelism):
//  * "4.1 Data parallelism in depth", sec. 2: the averaged
//    gradient g_bar = (1/N) sum_k g_k equals the full-batch gradient when every
//    rank averages over an equal local batch (eqs. for L, g, g_k, g_bar); sec. 4.2:
//    gradients are packed into ~25 MB buckets in reverse compute order; sec. 5:
//    all-reduce = reduce-scatter + all-gather, ring volume 2(N-1)/N * Psi;
//    sec. 6.1 and 7: the ZeRO stages and the 16-byte/parameter ledger; sec. 8.2:
//    ZeRO-3 moves 3 Psi.
//  * "Data Parallelism: From Parameter Server to Ring All-Reduce", sec. 1: the
//    synchronised gradient is the average over the N ranks, and every rank applies
//    the same optimizer step with it; sec. 5: at each ring step a rank passes one
//    chunk to its neighbour, which adds it to its own running sum, so after N-1
//    steps each rank holds one chunk's complete sum, and N-1 more steps pass the
//    reduced chunks on until every rank has all of them; per-rank traffic
//    2(N-1)/N * M; sec. 6: 2(N-1) steps.
//  * "Data Parallelism: DDP, ZeRO and FSDP", "The three stages": ZeRO-1/2
//    reduce-scatter, update the owned shard, all-gather the updated parameters.
//  * "Distributed Training: Data Parallel, Model Parallel and FSDP Strategies", "Inside DDP":
//    AdamW with learning rate 2e-4 and weight decay 0.1, clipping to norm 1.0 after the
//    averaged gradients; "FSDP1 vs FSDP2": MixedPrecisionPolicy(param bf16,
//    reduce fp32).
//
// Readings where the pages leave a step open (each is also listed in the design
// notes):
//  R1 ring schedule: at step s (0..P-2) rank r sends chunk (r-1-s) mod P to rank
//     r+1, which adds it into its own copy; rank c ends owning chunk c.  The
//     all-gather sends chunk (r-s) mod P at step s.
//  R2 reduction in fp32 (reduce_dtype=float32); bf16 -> fp32 is exact.
//  R3 the 1/P is applied after the sum, as an IEEE fp32 division.
//  R4 fp32 -> bf16 rounds to nearest even.
//  R5 bucket rule: walk tensors last to first, 8-element aligned slots, close the
//     bucket when a non-empty bucket would exceed the cap; a tensor is never
//     split; a bucket is padded to a multiple of 16P, so each of its P equal,
//     contiguous shards is a whole number of 32-byte bf16 blocks; padding holds
//     zeros.
//  R6 AdamW is torch.optim.AdamW's algorithm (decoupled decay, bias-corrected
//     Adam, eps outside the square root), with per-element op order
//        theta *= (1 - lr*wd)                     [decayed tensors only]
//        m = b1*m + (1-b1)*g
//        v = b2*v + (1-b2)*(g*g)
//        theta -= (lr/bc1) * (m / (sqrt(v)/sqrt(bc2) + eps))
//     in fp32 without fused multiply-add; the scalar factors are formed in
//     double and rounded to fp32 once.
//  R7 clipping is clip_grad_norm_: norm = ||mean||_2 over the fp32 mean
//     gradient (squares summed in double with Neumaier's compensated
//     summation), coef = min(1, max_norm/(norm+1e-6))
//     rounded to fp32 once; g = mean * coef.  max_norm <= 0 disables it.  A
//     non-finite norm gives coef = NaN, so the bad step shows in every output.
//
// Parity status: planner, ring sums/ownership/counters, AdamW closed form at
// t=1, ledger and volumes, least-squares identity are pinned by tests that use
// the pages' printed values, closed forms and brute force.  The AdamW op order
// (R6) and the clip form (R7) are readings, pinned algebraically only.
//
// Build: g++ -std=c++17 -O2 -ffp-contract=off -fPIC -shared -pthread
// (-ffp-contract=off keeps every multiply and add separately rounded).

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

constexpr int kMaxRanks = 64;

int mod(int a, int p) { return ((a % p) + p) % p; }

float bf16_bits_to_f32(uint16_t h) {
  uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Round-to-nearest-even to the upper 16 bits (R4).  NaN stays NaN (quietened).
uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x0040u);
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return static_cast<uint16_t>(u >> 16);
}

struct Plan {
  int P = 0;
  int64_t L = 0;
  std::vector<int64_t> t_off;     // flat padded offset of each tensor
  std::vector<int32_t> t_bucket;  // bucket of each tensor
  std::vector<int64_t> b_off, b_len;
  std::vector<std::vector<int32_t>> b_tensors;  // tensors of each bucket
};

// R5.  DDP fills buckets of about 25 MB in the reverse of the forward pass's
// order ("4.1 Data parallelism in depth", sec. 4.2); buckets fire in that order.
bool make_plan(const int64_t* sizes, int n, int64_t bucket_bytes, int P, Plan* pl) {
  if (n < 0 || P < 1 || P > kMaxRanks || bucket_bytes < 1) return false;
  for (int t = 0; t < n; ++t)
    if (sizes[t] < 0) return false;
  const int64_t cap = bucket_bytes / 2;  // bf16 elements
  const int64_t quantum = 16 * static_cast<int64_t>(P);
  pl->P = P;
  pl->t_off.assign(n, 0);
  pl->t_bucket.assign(n, -1);
  pl->b_off.clear();
  pl->b_len.clear();
  pl->b_tensors.clear();
  int64_t start = 0, used = 0;
  bool open = false;
  auto close_bucket = [&]() {
    const int64_t padded = (used + quantum - 1) / quantum * quantum;
    pl->b_off.push_back(start);
    pl->b_len.push_back(padded);
    start += padded;
    used = 0;
    open = false;
  };
  for (int t = n - 1; t >= 0; --t) {
    const int64_t slot = (sizes[t] + 7) / 8 * 8;
    if (open && used > 0 && used + slot > cap) close_bucket();
    if (!open) {
      open = true;
      pl->b_tensors.emplace_back();
    }
    pl->t_off[t] = start + used;
    pl->t_bucket[t] = static_cast<int32_t>(pl->b_tensors.size()) - 1;
    pl->b_tensors.back().push_back(t);
    used += slot;
  }
  if (open) close_bucket();
  pl->L = start;
  return true;
}

// Literal ring reduce-scatter over P buffers ("Data Parallelism: From Parameter Server to Ring All-Reduce", sec. 5, R1): P-1 steps, each
// rank sends one chunk to its clockwise neighbour, which adds it into its local
// partial sum.  X is [P][len] fp32; S = len/P.
void ring_reduce_scatter(int P, int64_t len, float* X, int64_t* sent, int64_t* steps) {
  const int64_t S = len / P;
  std::vector<float> msg(static_cast<size_t>(P) * S);
  for (int s = 0; s + 1 < P; ++s) {
    for (int r = 0; r < P; ++r) {  // everybody sends
      const int c = mod(r - 1 - s, P);
      std::memcpy(&msg[static_cast<size_t>(r) * S], X + static_cast<size_t>(r) * len + c * S,
                  sizeof(float) * S);
      sent[r] += S;
    }
    for (int r = 0; r < P; ++r) {  // everybody receives and accumulates
      const int dst = (r + 1) % P;
      const int c = mod(r - 1 - s, P);
      float* mine = X + static_cast<size_t>(dst) * len + c * S;
      const float* in = &msg[static_cast<size_t>(r) * S];
      for (int64_t i = 0; i < S; ++i) mine[i] = mine[i] + in[i];
    }
    ++*steps;
  }
}

// Literal ring all-gather ("Data Parallelism: From Parameter Server to Ring All-Reduce", sec. 5): P-1 steps, each rank forwards the
// reduced chunk it received last (its own chunk at step 0).  Y is [P][len] bf16.
void ring_all_gather(int P, int64_t len, uint16_t* Y, int64_t* sent, int64_t* steps) {
  const int64_t S = len / P;
  std::vector<uint16_t> msg(static_cast<size_t>(P) * S);
  for (int s = 0; s + 1 < P; ++s) {
    for (int r = 0; r < P; ++r) {
      const int c = mod(r - s, P);
      std::memcpy(&msg[static_cast<size_t>(r) * S], Y + static_cast<size_t>(r) * len + c * S,
                  sizeof(uint16_t) * S);
      sent[r] += S;
    }
    for (int r = 0; r < P; ++r) {
      const int dst = (r + 1) % P;
      const int c = mod(r - s, P);
      std::memcpy(Y + static_cast<size_t>(dst) * len + c * S, &msg[static_cast<size_t>(r) * S],
                  sizeof(uint16_t) * S);
    }
    ++*steps;
  }
}

// The same ring all-gather carrying fp32 partial results (used by the
// cross-group all-reduce of the hybrid mesh).
void ring_all_gather_f32(int P, int64_t len, float* Y, int64_t* sent, int64_t* steps) {
  const int64_t S = len / P;
  std::vector<float> msg(static_cast<size_t>(P) * S);
  for (int s = 0; s + 1 < P; ++s) {
    for (int r = 0; r < P; ++r) {
      const int c = mod(r - s, P);
      std::memcpy(&msg[static_cast<size_t>(r) * S], Y + static_cast<size_t>(r) * len + c * S,
                  sizeof(float) * S);
      sent[r] += S;
    }
    for (int r = 0; r < P; ++r) {
      const int dst = (r + 1) % P;
      const int c = mod(r - s, P);
      std::memcpy(Y + static_cast<size_t>(dst) * len + c * S, &msg[static_cast<size_t>(r) * S],
                  sizeof(float) * S);
    }
    ++*steps;
  }
}

}  // namespace

extern "C" {

struct orc_adamw {
  double lr, beta1, beta2, eps, weight_decay, max_norm;
  int64_t step;  // t >= 1
};

struct orc_stats {
  double sumsq;  // sum of mean^2 (double) over the padded elements used for the clip
  double norm;
  float coef;
  int32_t n_buckets;
  int64_t padded_len;
  int64_t rs_steps, ag_steps;  // ring steps, summed over buckets
  int32_t replicas_equal;      // 1 when all P replicas are bit-identical afterwards
  int32_t pad_;
  int64_t rs_sent[kMaxRanks];  // elements sent per rank, reduce-scatter phase
  int64_t ag_sent[kMaxRanks];  // elements sent per rank, all-gather phase
};

}  // extern "C"

namespace {

struct AdamScalars {
  float wd_factor, b1, omb1, b2, omb2, step_size, sqrt_bc2, eps;
};

AdamScalars adam_scalars(const orc_adamw& c) {
  AdamScalars s;
  const double t = static_cast<double>(c.step);
  s.wd_factor = static_cast<float>(1.0 - c.lr * c.weight_decay);
  s.b1 = static_cast<float>(c.beta1);
  s.omb1 = static_cast<float>(1.0 - c.beta1);
  s.b2 = static_cast<float>(c.beta2);
  s.omb2 = static_cast<float>(1.0 - c.beta2);
  s.step_size = static_cast<float>(c.lr / (1.0 - std::pow(c.beta1, t)));
  s.sqrt_bc2 = static_cast<float>(std::sqrt(1.0 - std::pow(c.beta2, t)));
  s.eps = static_cast<float>(c.eps);
  return s;
}

// R6: one element of AdamW ("Distributed Training: Data Parallel, Model Parallel and FSDP Strategies", "Inside DDP": torch.optim.AdamW).
void adamw_element(float g, float& theta, float& m, float& v, bool decay, const AdamScalars& s) {
  if (decay) theta = theta * s.wd_factor;
  m = s.b1 * m + s.omb1 * g;
  v = s.b2 * v + s.omb2 * (g * g);
  const float denom = std::sqrt(v) / s.sqrt_bc2 + s.eps;
  theta = theta - s.step_size * (m / denom);
}

// R7.
float clip_coef(double sumsq, double max_norm, double* norm_out) {
  const double norm = std::sqrt(sumsq);
  if (norm_out) *norm_out = norm;
  if (!(max_norm > 0.0)) return 1.0f;
  if (!std::isfinite(norm)) return std::nanf("");  // a non-finite norm poisons the step
  return static_cast<float>(std::min(1.0, max_norm / (norm + 1e-6)));
}

template <class F>
void parallel_for(int n, int n_threads, F&& f) {
  if (n_threads <= 0) n_threads = static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
  n_threads = std::min(n_threads, std::max(n, 1));
  if (n_threads <= 1) {
    for (int i = 0; i < n; ++i) f(i);
    return;
  }
  std::atomic<int> next{0};
  std::vector<std::thread> pool;
  for (int w = 0; w < n_threads; ++w)
    pool.emplace_back([&]() {
      for (int i = next++; i < n; i = next++) f(i);
    });
  for (auto& th : pool) th.join();
}

// Per bucket: the P ranks' fp32 copies of their gradients, packed in bucket order.
void pack_bucket(const Plan& pl, int b, const int64_t* sizes, const std::vector<int64_t>& base,
                 int64_t n_params, const uint16_t* grads, std::vector<float>& X) {
  const int P = pl.P;
  const int64_t len = pl.b_len[b];
  X.assign(static_cast<size_t>(P) * len, 0.0f);
  for (int t : pl.b_tensors[b]) {
    const int64_t o = pl.t_off[t] - pl.b_off[b];
    for (int r = 0; r < P; ++r) {
      const uint16_t* src = grads + static_cast<size_t>(r) * n_params + base[t];
      float* dst = X.data() + static_cast<size_t>(r) * len + o;
      for (int64_t j = 0; j < sizes[t]; ++j) dst[j] = bf16_bits_to_f32(src[j]);
    }
  }
}

std::vector<int64_t> tensor_bases(const int64_t* sizes, int n, int64_t* total) {
  std::vector<int64_t> base(n + 1, 0);
  for (int t = 0; t < n; ++t) base[t + 1] = base[t] + sizes[t];
  if (total) *total = base[n];
  return base;
}

// Reduce-scatter + 1/P of one bucket: returns the fp32 mean at every flat slot of
// the bucket (slot i taken from the owner of its chunk) and the counters.
void bucket_mean(const Plan& pl, int b, std::vector<float>& X, std::vector<float>& mean,
                 int64_t* rs_sent, int64_t* rs_steps) {
  const int P = pl.P;
  const int64_t len = pl.b_len[b];
  const int64_t S = len / P;
  ring_reduce_scatter(P, len, X.data(), rs_sent, rs_steps);
  mean.assign(len, 0.0f);
  for (int c = 0; c < P; ++c) {
    const float* own = X.data() + static_cast<size_t>(c) * len + c * S;  // rank c owns chunk c
    for (int64_t i = 0; i < S; ++i) mean[c * S + i] = own[i] / static_cast<float>(P);
  }
}

// Neumaier's compensated summation (an improved Kahan-Babuska sum): the running
// compensation keeps the result within a few ulps of the exact sum, where a
// plain running double sum of ~1e8 squares can drift by ~1e-10 relative.
struct CompensatedSum {
  double sum = 0.0, comp = 0.0;
  void add(double x) {
    const double t = sum + x;
    if (std::fabs(sum) >= std::fabs(x))
      comp += (sum - t) + x;
    else
      comp += (x - t) + sum;
    sum = t;
  }
  double value() const { return sum + comp; }
};

// sum of mean^2; each square of an fp32 value is exact in double.
double sumsq_of(const std::vector<float>& mean) {
  CompensatedSum acc;
  for (float x : mean) acc.add(static_cast<double>(x) * static_cast<double>(x));
  return acc.value();
}

}  // namespace

extern "C" {

// ---- planner ---------------------------------------------------------------
// Outputs: t_off[n], t_bucket[n], b_off[n], b_len[n] (at most n buckets), *nb, *L.
int orc_plan(const int64_t* sizes, int32_t n, int64_t bucket_bytes, int32_t P, int64_t* t_off,
             int32_t* t_bucket, int64_t* b_off, int64_t* b_len, int32_t* nb, int64_t* L) {
  Plan pl;
  if (!make_plan(sizes, n, bucket_bytes, P, &pl)) return -1;
  for (int t = 0; t < n; ++t) {
    t_off[t] = pl.t_off[t];
    t_bucket[t] = pl.t_bucket[t];
  }
  for (size_t b = 0; b < pl.b_off.size(); ++b) {
    b_off[b] = pl.b_off[b];
    b_len[b] = pl.b_len[b];
  }
  *nb = static_cast<int32_t>(pl.b_off.size());
  *L = pl.L;
  return 0;
}

// ---- ring primitives, exposed for the pins ---------------------------------
int orc_ring_reduce_scatter_f32(int32_t P, int64_t len, float* X, int64_t* sent, int64_t* steps) {
  if (P < 1 || P > kMaxRanks || len < 0 || len % P) return -1;
  ring_reduce_scatter(P, len, X, sent, steps);
  return 0;
}

int orc_ring_all_gather_u16(int32_t P, int64_t len, uint16_t* Y, int64_t* sent, int64_t* steps) {
  if (P < 1 || P > kMaxRanks || len < 0 || len % P) return -1;
  ring_all_gather(P, len, Y, sent, steps);
  return 0;
}

uint16_t orc_bf16_rne(float f) { return f32_to_bf16_rne(f); }

// One AdamW element; state[0..2] = theta, m, v (in/out).
void orc_adamw_element(float g, float* state, int32_t decay, const orc_adamw* cfg) {
  const AdamScalars s = adam_scalars(*cfg);
  adamw_element(g, state[0], state[1], state[2], decay != 0, s);
}

float orc_clip_coef(const double* bucket_sumsq, int32_t nb, double max_norm, double* norm) {
  CompensatedSum acc;
  for (int b = 0; b < nb; ++b) acc.add(bucket_sumsq[b]);
  return clip_coef(acc.value(), max_norm, norm);
}

// The compensated total of per-bucket sums (what orc_zero_step takes as sumsq_total).
double orc_sum(const double* x, int64_t n) {
  CompensatedSum acc;
  for (int64_t i = 0; i < n; ++i) acc.add(x[i]);
  return acc.value();
}

// ---- the mean all-reduce (DDP / NO_SHARD) ----------------------------------
// grads: [P][n_params] bf16 bits, tensors concatenated in list order, replaced by
// bf16(mean) on every replica.  mean_out (nullable): fp32 mean [n_params].
int orc_allreduce_mean(const int64_t* sizes, int32_t n, int64_t bucket_bytes, int32_t P,
                       uint16_t* grads, float* mean_out, orc_stats* st, int32_t n_threads) {
  Plan pl;
  if (!make_plan(sizes, n, bucket_bytes, P, &pl)) return -1;
  int64_t n_params = 0;
  const std::vector<int64_t> base = tensor_bases(sizes, n, &n_params);
  const int nb = static_cast<int>(pl.b_off.size());
  std::vector<std::vector<int64_t>> rs_sent(nb, std::vector<int64_t>(P, 0)),
      ag_sent(nb, std::vector<int64_t>(P, 0));
  std::vector<int64_t> rs_steps(nb, 0), ag_steps(nb, 0);
  std::vector<int> equal(nb, 1);
  parallel_for(nb, n_threads, [&](int b) {
    std::vector<float> X, mean;
    pack_bucket(pl, b, sizes, base, n_params, grads, X);
    bucket_mean(pl, b, X, mean, rs_sent[b].data(), &rs_steps[b]);
    const int64_t len = pl.b_len[b], S = len / P;
    std::vector<uint16_t> Y(static_cast<size_t>(P) * len, 0);
    for (int c = 0; c < P; ++c)  // the owner's payload is bf16(mean) of its chunk
      for (int64_t i = 0; i < S; ++i)
        Y[static_cast<size_t>(c) * len + c * S + i] = f32_to_bf16_rne(mean[c * S + i]);
    ring_all_gather(P, len, Y.data(), ag_sent[b].data(), &ag_steps[b]);
    for (int r = 1; r < P; ++r)
      if (std::memcmp(Y.data(), Y.data() + static_cast<size_t>(r) * len, 2 * len)) equal[b] = 0;
    for (int t : pl.b_tensors[b]) {
      const int64_t o = pl.t_off[t] - pl.b_off[b];
      for (int r = 0; r < P; ++r)
        std::memcpy(grads + static_cast<size_t>(r) * n_params + base[t],
                    Y.data() + static_cast<size_t>(r) * len + o, 2 * sizes[t]);
      if (mean_out) std::memcpy(mean_out + base[t], mean.data() + o, 4 * sizes[t]);
    }
  });
  if (st) {
    std::memset(st, 0, sizeof(*st));
    st->n_buckets = nb;
    st->padded_len = pl.L;
    st->replicas_equal = 1;
    st->coef = 1.0f;
    for (int b = 0; b < nb; ++b) {
      for (int r = 0; r < P; ++r) {
        st->rs_sent[r] += rs_sent[b][r];
        st->ag_sent[r] += ag_sent[b][r];
      }
      st->rs_steps += rs_steps[b];
      st->ag_steps += ag_steps[b];
      st->replicas_equal &= equal[b];
    }
  }
  return 0;
}

// Sum of mean^2 (double) of each bucket of the problem, bucket order; the input
// to orc_clip_coef when a problem is streamed bucket by bucket.
int orc_bucket_sumsq(const int64_t* sizes, int32_t n, int64_t bucket_bytes, int32_t P,
                     const uint16_t* grads, double* sumsq_out, int32_t n_threads) {
  Plan pl;
  if (!make_plan(sizes, n, bucket_bytes, P, &pl)) return -1;
  int64_t n_params = 0;
  const std::vector<int64_t> base = tensor_bases(sizes, n, &n_params);
  const int nb = static_cast<int>(pl.b_off.size());
  parallel_for(nb, n_threads, [&](int b) {
    std::vector<float> X, mean;
    int64_t sent[kMaxRanks] = {0}, steps = 0;
    pack_bucket(pl, b, sizes, base, n_params, grads, X);
    bucket_mean(pl, b, X, mean, sent, &steps);
    sumsq_out[b] = sumsq_of(mean);
  });
  return 0;
}

// ---- the fused ZeRO-1/2 step ------------------------------------------------
// ZeRO-1/2 keep DDP's reduce-scatter, have each rank update the shard it owns,
// then all-gather the new parameters ("Data Parallelism: DDP, ZeRO and FSDP",
// "The three stages").  grads [P][n_params] bf16 (in), master/m/v [n_params] fp32 (in/out),
// params [P][n_params] bf16 (out, all replicas), mean_out [n_params] (nullable,
// pre-clip fp32 mean).  sumsq_total < 0: the clip norm is taken over this
// problem; >= 0: that value is used (a streamed problem's total from
// orc_bucket_sumsq + orc_clip_coef's sum).
int orc_zero_step(const int64_t* sizes, const uint8_t* decay, int32_t n, int64_t bucket_bytes,
                  int32_t P, const uint16_t* grads, float* master, float* m, float* v,
                  uint16_t* params, const orc_adamw* cfg, float* mean_out, double sumsq_total,
                  orc_stats* st, int32_t n_threads) {
  Plan pl;
  if (!make_plan(sizes, n, bucket_bytes, P, &pl) || cfg->step < 1) return -1;
  int64_t n_params = 0;
  const std::vector<int64_t> base = tensor_bases(sizes, n, &n_params);
  const int nb = static_cast<int>(pl.b_off.size());
  std::vector<std::vector<float>> means(nb);
  std::vector<std::vector<int64_t>> rs_sent(nb, std::vector<int64_t>(P, 0)),
      ag_sent(nb, std::vector<int64_t>(P, 0));
  std::vector<int64_t> rs_steps(nb, 0), ag_steps(nb, 0);
  std::vector<double> bsum(nb, 0.0);
  std::vector<int> equal(nb, 1);

  // phase 1: reduce-scatter + mean, per bucket
  parallel_for(nb, n_threads, [&](int b) {
    std::vector<float> X;
    pack_bucket(pl, b, sizes, base, n_params, grads, X);
    bucket_mean(pl, b, X, means[b], rs_sent[b].data(), &rs_steps[b]);
    bsum[b] = sumsq_of(means[b]);
  });

  // global norm and clip coefficient ("Distributed Training: Data Parallel, Model Parallel and FSDP Strategies", "Inside DDP": clip after the
  // gradients are averaged)
  CompensatedSum total;
  for (int b = 0; b < nb; ++b) total.add(bsum[b]);
  double sumsq = total.value();
  if (sumsq_total >= 0.0) sumsq = sumsq_total;
  double norm = 0.0;
  const float coef = clip_coef(sumsq, cfg->max_norm, &norm);
  const AdamScalars s = adam_scalars(*cfg);

  // phase 2: each owner updates its shard, then the ring all-gathers bf16 params
  parallel_for(nb, n_threads, [&](int b) {
    const int64_t len = pl.b_len[b], S = len / P;
    // per flat slot of the bucket: tensor index (or -1 for padding) and element
    std::vector<int32_t> slot_t(len, -1);
    std::vector<int64_t> slot_j(len, 0);
    for (int t : pl.b_tensors[b]) {
      const int64_t o = pl.t_off[t] - pl.b_off[b];
      for (int64_t j = 0; j < sizes[t]; ++j) {
        slot_t[o + j] = t;
        slot_j[o + j] = j;
      }
    }
    std::vector<uint16_t> Y(static_cast<size_t>(P) * len, 0);
    for (int c = 0; c < P; ++c) {  // rank c updates the shard it owns
      for (int64_t i = c * S; i < (c + 1) * S; ++i) {
        const float g = means[b][i] * coef;
        float theta = 0.0f, mm = 0.0f, vv = 0.0f;
        const int t = slot_t[i];
        const int64_t e = t >= 0 ? base[t] + slot_j[i] : -1;
        if (t >= 0) {
          theta = master[e];
          mm = m[e];
          vv = v[e];
        }
        adamw_element(g, theta, mm, vv, t >= 0 && decay[t] != 0, s);
        if (t >= 0) {
          master[e] = theta;
          m[e] = mm;
          v[e] = vv;
        }
        Y[static_cast<size_t>(c) * len + i] = f32_to_bf16_rne(theta);
      }
    }
    ring_all_gather(P, len, Y.data(), ag_sent[b].data(), &ag_steps[b]);
    for (int r = 1; r < P; ++r)
      if (std::memcmp(Y.data(), Y.data() + static_cast<size_t>(r) * len, 2 * len)) equal[b] = 0;
    for (int t : pl.b_tensors[b]) {
      const int64_t o = pl.t_off[t] - pl.b_off[b];
      for (int r = 0; r < P; ++r)
        std::memcpy(params + static_cast<size_t>(r) * n_params + base[t],
                    Y.data() + static_cast<size_t>(r) * len + o, 2 * sizes[t]);
      if (mean_out) std::memcpy(mean_out + base[t], means[b].data() + o, 4 * sizes[t]);
    }
  });

  if (st) {
    std::memset(st, 0, sizeof(*st));
    st->sumsq = sumsq;
    st->norm = norm;
    st->coef = coef;
    st->n_buckets = nb;
    st->padded_len = pl.L;
    st->replicas_equal = 1;
    for (int b = 0; b < nb; ++b) {
      for (int r = 0; r < P; ++r) {
        st->rs_sent[r] += rs_sent[b][r];
        st->ag_sent[r] += ag_sent[b][r];
      }
      st->rs_steps += rs_steps[b];
      st->ag_steps += ag_steps[b];
      st->replicas_equal &= equal[b];
    }
  }
  return 0;
}

// ---- hybrid sharding on an R x S mesh -------------------------------------------
// HYBRID_SHARD: shard within a group, data-parallel all-reduce across groups
// ("4.1 Data parallelism in depth", sec. 6.3 table and tip; "Distributed Training:
// Data Parallel, Model Parallel and FSDP Strategies", FSDP2 DeviceMesh
// mesh_shape=(2, 4) with dims ("replicate", "shard"), and "Selecting and Tuning":
// sharding inside each group of ranks, an ordinary data-parallel all-reduce
// between the groups;
// "Data Parallelism: DDP, ZeRO and FSDP", "Hybrid sharding").  Rank (g, s) =
// g*S + s.  Per bucket, literally:
//   1. in every group g, a ring reduce-scatter over its S ranks: rank (g, s)
//      holds the group's sum of shard s (S equal shards);
//   2. for every shard s, a ring all-reduce over the R ranks (0..R-1, s):
//      reduce-scatter over R sub-chunks of the shard, then all-gather;
//   3. mean = sum / P; rank (g, s) updates shard s (every group the same);
//   4. in every group, a ring all-gather of the bf16 shards.
// rs_sent counts steps 1 and the cross reduce-scatter, ag_sent the cross
// all-gather and step 4; cross_sent only the cross-group (step 2) traffic.
struct orc_mesh_stats {
  int64_t rs_sent[kMaxRanks];
  int64_t ag_sent[kMaxRanks];
  int64_t cross_sent[kMaxRanks];
  int32_t groups_equal;     // 1 when every group's updated shard state agreed
  int32_t replicas_equal;   // 1 when all P replicas are bit-identical afterwards
  double sumsq;
  double norm;
  float coef;
  int32_t pad_;
};

}  // extern "C"

namespace {

// Steps 1-2 for one bucket: X [P][len] fp32 per rank -> the total of every slot
// as held by rank (g, s) after the cross all-reduce (identical for all g).
void mesh_reduce(int R, int S, int64_t len, std::vector<float>& X, std::vector<float>& total,
                 int64_t* rs_sent, int64_t* ag_sent, int64_t* cross_sent) {
  const int P = R * S;
  const int64_t sh = len / S;  // shard length
  int64_t steps = 0;
  std::vector<float> G(static_cast<size_t>(S) * len);
  for (int g = 0; g < R; ++g) {  // 1. ring reduce-scatter inside group g
    std::memcpy(G.data(), X.data() + static_cast<size_t>(g) * S * len, sizeof(float) * S * len);
    int64_t sent[kMaxRanks] = {0};
    ring_reduce_scatter(S, len, G.data(), sent, &steps);
    std::memcpy(X.data() + static_cast<size_t>(g) * S * len, G.data(), sizeof(float) * S * len);
    for (int s = 0; s < S; ++s) rs_sent[g * S + s] += sent[s];
  }
  total.assign(len, 0.0f);
  std::vector<float> C(static_cast<size_t>(R) * sh);
  for (int s = 0; s < S; ++s) {  // 2. ring all-reduce of shard s across the groups
    for (int g = 0; g < R; ++g)
      std::memcpy(C.data() + static_cast<size_t>(g) * sh,
                  X.data() + static_cast<size_t>(g * S + s) * len + s * sh, sizeof(float) * sh);
    int64_t sent_rs[kMaxRanks] = {0}, sent_ag[kMaxRanks] = {0};
    ring_reduce_scatter(R, sh, C.data(), sent_rs, &steps);
    ring_all_gather_f32(R, sh, C.data(), sent_ag, &steps);
    for (int g = 0; g < R; ++g) {
      rs_sent[g * S + s] += sent_rs[g];
      ag_sent[g * S + s] += sent_ag[g];
      cross_sent[g * S + s] += sent_rs[g] + sent_ag[g];
    }
    for (int g = 1; g < R; ++g)  // every group now holds the same totals
      if (std::memcmp(C.data(), C.data() + static_cast<size_t>(g) * sh, sizeof(float) * sh))
        total.assign(len, std::nanf(""));
    std::memcpy(total.data() + s * sh, C.data(), sizeof(float) * sh);
  }
  (void)P;
}

// Step 4: ring all-gather of bf16 shards inside every group; Y [P][len].
void mesh_all_gather(int R, int S, int64_t len, std::vector<uint16_t>& Y, int64_t* ag_sent) {
  int64_t steps = 0;
  std::vector<uint16_t> G(static_cast<size_t>(S) * len);
  for (int g = 0; g < R; ++g) {
    std::memcpy(G.data(), Y.data() + static_cast<size_t>(g) * S * len, 2 * S * len);
    int64_t sent[kMaxRanks] = {0};
    ring_all_gather(S, len, G.data(), sent, &steps);
    std::memcpy(Y.data() + static_cast<size_t>(g) * S * len, G.data(), 2 * S * len);
    for (int s = 0; s < S; ++s) ag_sent[g * S + s] += sent[s];
  }
}

}  // namespace

extern "C" {

// Mean all-reduce on the R x S mesh (HYBRID with NO_SHARD state): every replica
// ends with bf16(mean).  grads [P][n_params] in/out, mean_out nullable.
int orc_mesh_allreduce_mean(const int64_t* sizes, int32_t n, int64_t bucket_bytes, int32_t R,
                            int32_t S, uint16_t* grads, float* mean_out, orc_mesh_stats* st) {
  const int P = R * S;
  Plan pl;
  if (R < 1 || S < 1 || !make_plan(sizes, n, bucket_bytes, P, &pl)) return -1;
  int64_t n_params = 0;
  const std::vector<int64_t> base = tensor_bases(sizes, n, &n_params);
  orc_mesh_stats acc;
  std::memset(&acc, 0, sizeof(acc));
  acc.groups_equal = 1;
  acc.replicas_equal = 1;
  for (size_t b = 0; b < pl.b_off.size(); ++b) {
    const int64_t len = pl.b_len[b], sh = len / S;
    std::vector<float> X, total;
    pack_bucket(pl, static_cast<int>(b), sizes, base, n_params, grads, X);
    mesh_reduce(R, S, len, X, total, acc.rs_sent, acc.ag_sent, acc.cross_sent);
    std::vector<uint16_t> Y(static_cast<size_t>(P) * len, 0);
    for (int g = 0; g < R; ++g)
      for (int s = 0; s < S; ++s)
        for (int64_t i = s * sh; i < (s + 1) * sh; ++i)
          Y[static_cast<size_t>(g * S + s) * len + i] = f32_to_bf16_rne(total[i] / static_cast<float>(P));
    mesh_all_gather(R, S, len, Y, acc.ag_sent);
    for (int r = 1; r < P; ++r)
      if (std::memcmp(Y.data(), Y.data() + static_cast<size_t>(r) * len, 2 * len)) acc.replicas_equal = 0;
    for (int t : pl.b_tensors[b]) {
      const int64_t o = pl.t_off[t] - pl.b_off[b];
      for (int r = 0; r < P; ++r)
        std::memcpy(grads + static_cast<size_t>(r) * n_params + base[t],
                    Y.data() + static_cast<size_t>(r) * len + o, 2 * sizes[t]);
      if (mean_out)
        for (int64_t j = 0; j < sizes[t]; ++j) mean_out[base[t] + j] = total[o + j] / static_cast<float>(P);
    }
  }
  if (st) *st = acc;
  return 0;
}

// The ZeRO-2 step on the R x S mesh: every group's rank (g, s) updates shard s
// of its own copy of master/m/v (they must agree across groups) and the bf16
// parameters are all-gathered inside every group.  Clip norm over the mean,
// as in orc_zero_step.
int orc_mesh_zero_step(const int64_t* sizes, const uint8_t* decay, int32_t n, int64_t bucket_bytes,
                       int32_t R, int32_t S, const uint16_t* grads, float* master, float* m,
                       float* v, uint16_t* params, const orc_adamw* cfg, orc_mesh_stats* st) {
  const int P = R * S;
  Plan pl;
  if (R < 1 || S < 1 || !make_plan(sizes, n, bucket_bytes, P, &pl) || cfg->step < 1) return -1;
  int64_t n_params = 0;
  const std::vector<int64_t> base = tensor_bases(sizes, n, &n_params);
  const int nb = static_cast<int>(pl.b_off.size());
  orc_mesh_stats acc;
  std::memset(&acc, 0, sizeof(acc));
  acc.groups_equal = 1;
  acc.replicas_equal = 1;
  std::vector<std::vector<float>> means(nb);
  CompensatedSum total_sq;
  for (int b = 0; b < nb; ++b) {
    std::vector<float> X, total;
    pack_bucket(pl, b, sizes, base, n_params, grads, X);
    mesh_reduce(R, S, pl.b_len[b], X, total, acc.rs_sent, acc.ag_sent, acc.cross_sent);
    means[b].resize(pl.b_len[b]);
    for (int64_t i = 0; i < pl.b_len[b]; ++i) means[b][i] = total[i] / static_cast<float>(P);
    total_sq.add(sumsq_of(means[b]));
  }
  acc.sumsq = total_sq.value();
  acc.coef = clip_coef(acc.sumsq, cfg->max_norm, &acc.norm);
  const AdamScalars sc = adam_scalars(*cfg);
  for (int b = 0; b < nb; ++b) {
    const int64_t len = pl.b_len[b], sh = len / S;
    std::vector<int32_t> slot_t(len, -1);
    std::vector<int64_t> slot_j(len, 0);
    for (int t : pl.b_tensors[b]) {
      const int64_t o = pl.t_off[t] - pl.b_off[b];
      for (int64_t j = 0; j < sizes[t]; ++j) {
        slot_t[o + j] = t;
        slot_j[o + j] = j;
      }
    }
    std::vector<uint16_t> Y(static_cast<size_t>(P) * len, 0);
    for (int s = 0; s < S; ++s) {
      for (int64_t i = s * sh; i < (s + 1) * sh; ++i) {
        const int t = slot_t[i];
        const int64_t e = t >= 0 ? base[t] + slot_j[i] : -1;
        float first[3] = {0, 0, 0};
        for (int g = 0; g < R; ++g) {  // each group's owner of shard s, own state copy
          float th = t >= 0 ? master[e] : 0.0f, mm = t >= 0 ? m[e] : 0.0f, vv = t >= 0 ? v[e] : 0.0f;
          adamw_element(means[b][i] * acc.coef, th, mm, vv, t >= 0 && decay[t] != 0, sc);
          if (g == 0) {
            first[0] = th;
            first[1] = mm;
            first[2] = vv;
          } else if (std::memcmp(first, &th, 4) || std::memcmp(first + 1, &mm, 4) ||
                     std::memcmp(first + 2, &vv, 4)) {
            acc.groups_equal = 0;
          }
          Y[static_cast<size_t>(g * S + s) * len + i] = f32_to_bf16_rne(th);
        }
        if (t >= 0) {
          master[e] = first[0];
          m[e] = first[1];
          v[e] = first[2];
        }
      }
    }
    mesh_all_gather(R, S, len, Y, acc.ag_sent);
    for (int r = 1; r < P; ++r)
      if (std::memcmp(Y.data(), Y.data() + static_cast<size_t>(r) * len, 2 * len)) acc.replicas_equal = 0;
    for (int t : pl.b_tensors[b]) {
      const int64_t o = pl.t_off[t] - pl.b_off[b];
      for (int r = 0; r < P; ++r)
        std::memcpy(params + static_cast<size_t>(r) * n_params + base[t],
                    Y.data() + static_cast<size_t>(r) * len + o, 2 * sizes[t]);
    }
  }
  if (st) *st = acc;
  return 0;
}

// ---- ZeRO-3 / FULL_SHARD unit flow ------------------------------------------
// FSDP applies ZeRO-3 unit by unit: before a unit's forward its parameter shards
// are all-gathered into the whole unit, before its backward they are gathered
// again and afterwards its gradients are reduce-scattered, and the optimizer on
// each rank updates only that rank's shard ("Data Parallelism: DDP, ZeRO and
// FSDP", "How FSDP actually runs" and
// "The three stages": 3N; "4.1 Data parallelism in depth", sec. 6.2 and 8.2).
// Units are the plan's buckets; forward visits them from the last bucket to the
// first (buckets hold layers in reverse), backward from the first to the last.
// param_shards [n_params] bf16: each element as held by its shard owner (in/out);
// grads [P][n_params]: every rank's full gradients of this step.  Outputs the
// same master/m/v and bf16 values as orc_zero_step.
struct orc_zero3_stats {
  int64_t ag_fwd_sent[kMaxRanks];
  int64_t ag_bwd_sent[kMaxRanks];
  int64_t rs_sent[kMaxRanks];
  int32_t gathered_ok;   // 1 when every rank's gathered unit equals the shards' values
  int32_t pad_;
  double norm;
  float coef;
  int32_t pad2_;
};

int orc_zero3_step(const int64_t* sizes, const uint8_t* decay, int32_t n, int64_t bucket_bytes,
                   int32_t P, const uint16_t* grads, uint16_t* param_shards, float* master,
                   float* m, float* v, const orc_adamw* cfg, orc_zero3_stats* st) {
  Plan pl;
  if (!make_plan(sizes, n, bucket_bytes, P, &pl) || cfg->step < 1) return -1;
  int64_t n_params = 0;
  const std::vector<int64_t> base = tensor_bases(sizes, n, &n_params);
  const int nb = static_cast<int>(pl.b_off.size());
  orc_zero3_stats acc;
  std::memset(&acc, 0, sizeof(acc));
  acc.gathered_ok = 1;
  // the unit's bf16 shards laid out flat in the bucket (padding 0)
  auto unit_values = [&](int b, std::vector<uint16_t>& u) {
    u.assign(pl.b_len[b], 0);
    for (int t : pl.b_tensors[b]) {
      const int64_t o = pl.t_off[t] - pl.b_off[b];
      for (int64_t j = 0; j < sizes[t]; ++j) u[o + j] = param_shards[base[t] + j];
    }
  };
  // one all-gather of unit b: rank c starts with only its shard; check the result
  auto gather = [&](int b, int64_t* sent) {
    const int64_t len = pl.b_len[b], S = len / P;
    std::vector<uint16_t> u, Y(static_cast<size_t>(P) * len, 0);
    unit_values(b, u);
    for (int c = 0; c < P; ++c)
      std::memcpy(Y.data() + static_cast<size_t>(c) * len + c * S, u.data() + c * S, 2 * S);
    int64_t steps = 0;
    ring_all_gather(P, len, Y.data(), sent, &steps);
    for (int r = 0; r < P; ++r)
      if (std::memcmp(Y.data() + static_cast<size_t>(r) * len, u.data(), 2 * len)) acc.gathered_ok = 0;
  };
  for (int b = nb - 1; b >= 0; --b) gather(b, acc.ag_fwd_sent);     // forward
  std::vector<std::vector<float>> means(nb);
  CompensatedSum total;
  for (int b = 0; b < nb; ++b) {                                    // backward
    gather(b, acc.ag_bwd_sent);
    std::vector<float> X;
    int64_t steps = 0;
    pack_bucket(pl, b, sizes, base, n_params, grads, X);
    bucket_mean(pl, b, X, means[b], acc.rs_sent, &steps);
    total.add(sumsq_of(means[b]));
  }
  acc.coef = clip_coef(total.value(), cfg->max_norm, &acc.norm);
  const AdamScalars sc = adam_scalars(*cfg);
  for (int b = 0; b < nb; ++b) {                                    // each owner's shard
    for (int t : pl.b_tensors[b]) {
      const int64_t o = pl.t_off[t] - pl.b_off[b];
      for (int64_t j = 0; j < sizes[t]; ++j) {
        const int64_t e = base[t] + j;
        adamw_element(means[b][o + j] * acc.coef, master[e], m[e], v[e], decay[t] != 0, sc);
        param_shards[e] = f32_to_bf16_rne(master[e]);
      }
    }
  }
  if (st) *st = acc;
  return 0;
}

// ---- gradient accumulation and the bf16 wire ----------------------------------
// Gradient accumulation keeps the global batch large at a fixed memory cost,
// synchronising only on the last micro-batch ("Distributed Training: Data
// Parallel, Model Parallel and FSDP Strategies", "Selecting and Tuning": no_sync
// on every micro-batch but the last).  Each rank's bf16 gradient buffer accumulates the
// micro-batch gradients as autograd does for bf16 gradients: acc = bf16(acc + g),
// the add in fp32.  acc, micro: [P][n] bf16 bits.
void orc_accumulate(int32_t P, int64_t n, uint16_t* acc, const uint16_t* micro) {
  for (int64_t i = 0; i < static_cast<int64_t>(P) * n; ++i)
    acc[i] = f32_to_bf16_rne(bf16_bits_to_f32(acc[i]) + bf16_bits_to_f32(micro[i]));
}

// The dtype gradients are communicated in changes both the bytes moved and the
// numerics ("Data Parallelism: From Parameter Server to Ring All-Reduce",
// sec. 8).  The ring with bf16 on the wire: every hop's partial sum
// is rounded to bf16 before it is sent (the receiver adds in fp32 and rounds),
// the owner's final sum is divided by P in fp32 and rounded to bf16 for the
// all-gather.  grads [P][n_params] in/out; mean_out: the fp32 quotient before
// its bf16 rounding (nullable).
int orc_allreduce_mean_bf16wire(const int64_t* sizes, int32_t n, int64_t bucket_bytes, int32_t P,
                                uint16_t* grads, float* mean_out) {
  Plan pl;
  if (!make_plan(sizes, n, bucket_bytes, P, &pl)) return -1;
  int64_t n_params = 0;
  const std::vector<int64_t> base = tensor_bases(sizes, n, &n_params);
  for (size_t b = 0; b < pl.b_off.size(); ++b) {
    const int64_t len = pl.b_len[b], S = len / P;
    std::vector<float> X;
    pack_bucket(pl, static_cast<int>(b), sizes, base, n_params, grads, X);
    std::vector<uint16_t> W(static_cast<size_t>(P) * len);   // what each rank holds, bf16
    for (size_t i = 0; i < W.size(); ++i) W[i] = f32_to_bf16_rne(X[i]);
    std::vector<uint16_t> msg(static_cast<size_t>(P) * S);
    for (int s = 0; s + 1 < P; ++s) {
      for (int r = 0; r < P; ++r) {
        const int c = mod(r - 1 - s, P);
        std::memcpy(&msg[static_cast<size_t>(r) * S], W.data() + static_cast<size_t>(r) * len + c * S, 2 * S);
      }
      for (int r = 0; r < P; ++r) {
        const int dst = (r + 1) % P, c = mod(r - 1 - s, P);
        uint16_t* mine = W.data() + static_cast<size_t>(dst) * len + c * S;
        for (int64_t i = 0; i < S; ++i)
          mine[i] = f32_to_bf16_rne(bf16_bits_to_f32(mine[i]) + bf16_bits_to_f32(msg[static_cast<size_t>(r) * S + i]));
      }
    }
    std::vector<float> q(len);
    std::vector<uint16_t> Y(static_cast<size_t>(P) * len, 0);
    for (int c = 0; c < P; ++c)
      for (int64_t i = c * S; i < (c + 1) * S; ++i) {
        q[i] = bf16_bits_to_f32(W[static_cast<size_t>(c) * len + i]) / static_cast<float>(P);
        Y[static_cast<size_t>(c) * len + i] = f32_to_bf16_rne(q[i]);
      }
    int64_t sent[kMaxRanks] = {0}, steps = 0;
    ring_all_gather(P, len, Y.data(), sent, &steps);
    for (int t : pl.b_tensors[b]) {
      const int64_t o = pl.t_off[t] - pl.b_off[b];
      for (int r = 0; r < P; ++r)
        std::memcpy(grads + static_cast<size_t>(r) * n_params + base[t],
                    Y.data() + static_cast<size_t>(r) * len + o, 2 * sizes[t]);
      if (mean_out) std::memcpy(mean_out + base[t], q.data() + o, 4 * sizes[t]);
    }
  }
  return 0;
}

// ---- ledger and volumes ------------------------------------------------------
// Per-rank model-state bytes for `psi` parameters on P ranks, summing the
// buffers each stage keeps ("4.1 Data parallelism in depth", sec. 6.1 table and sec. 7; "Data Parallelism: DDP, ZeRO and FSDP",
// "The three stages").  comp[5] = bytes per parameter of (params, grads,
// master, m, v).  stage: 0 DDP, 1 ZeRO-1 (optimizer state sharded), 2 ZeRO-2
// (+ gradients), 3 ZeRO-3 (+ parameters).
double orc_ledger_bytes(int32_t stage, double psi, int32_t P, const double* comp) {
  const bool shard_params = stage >= 3, shard_grads = stage >= 2, shard_opt = stage >= 1;
  double total = 0.0;
  total += comp[0] * psi / (shard_params ? P : 1);
  total += comp[1] * psi / (shard_grads ? P : 1);
  for (int k = 2; k < 5; ++k) total += comp[k] * psi / (shard_opt ? P : 1);
  return total;
}

// Elements each rank sends in one training step's synchronisation, simulated
// with the ring primitives on M elements: DDP / ZeRO-1 / ZeRO-2 run one
// reduce-scatter and one all-gather; ZeRO-3 runs an all-gather before the
// forward, another before the backward, and a reduce-scatter of the gradients
// ("4.1 Data parallelism in depth", sec. 8.2; "Data Parallelism: DDP, ZeRO and FSDP", "The three stages").
int orc_stage_traffic(int32_t stage, int32_t P, int64_t M, int64_t* sent, int64_t* steps) {
  if (P < 1 || P > kMaxRanks || M % P) return -1;
  std::vector<float> X(static_cast<size_t>(P) * M, 1.0f);
  std::vector<uint16_t> Y(static_cast<size_t>(P) * M, 0);
  for (int r = 0; r < P; ++r) sent[r] = 0;
  *steps = 0;
  if (stage == 3) {
    ring_all_gather(P, M, Y.data(), sent, steps);
    ring_all_gather(P, M, Y.data(), sent, steps);
    ring_reduce_scatter(P, M, X.data(), sent, steps);
  } else {
    ring_reduce_scatter(P, M, X.data(), sent, steps);
    ring_all_gather(P, M, Y.data(), sent, steps);
  }
  return 0;
}

// ---- least-squares identity ("4.1 Data parallelism in depth", sec. 2) ----------------------------
// l_i = 1/2 (x_i . theta - y_i)^2, grad_i = (x_i . theta - y_i) x_i, in double.
// Ranks take consecutive blocks of split[k] samples.  Outputs (each [F]):
// g_full = (1/B) sum_i grad_i; g_k[k][F] = (1/|D_k|) sum_{i in D_k} grad_i
// (= N/B sum for an equal split); g_bar = (1/N) sum_k g_k; g_sum = sum_k g_k.
int orc_lsq_identity(int32_t B, int32_t F, int32_t N, const double* x, const double* y,
                     const double* theta, const int32_t* split, double* g_full, double* g_k,
                     double* g_bar, double* g_sum) {
  int32_t tot = 0;
  for (int k = 0; k < N; ++k) tot += split[k];
  if (tot != B) return -1;
  std::vector<double> gi(static_cast<size_t>(B) * F);
  for (int i = 0; i < B; ++i) {
    double pred = 0.0;
    for (int f = 0; f < F; ++f) pred += x[i * F + f] * theta[f];
    const double res = pred - y[i];
    for (int f = 0; f < F; ++f) gi[static_cast<size_t>(i) * F + f] = res * x[i * F + f];
  }
  for (int f = 0; f < F; ++f) {
    double acc = 0.0;
    for (int i = 0; i < B; ++i) acc += gi[static_cast<size_t>(i) * F + f];
    g_full[f] = acc / B;
  }
  int32_t start = 0;
  for (int k = 0; k < N; ++k) {
    for (int f = 0; f < F; ++f) {
      double acc = 0.0;
      for (int i = start; i < start + split[k]; ++i) acc += gi[static_cast<size_t>(i) * F + f];
      g_k[k * F + f] = acc / split[k];
    }
    start += split[k];
  }
  for (int f = 0; f < F; ++f) {
    double acc = 0.0;
    for (int k = 0; k < N; ++k) acc += g_k[k * F + f];
    g_sum[f] = acc;
    g_bar[f] = acc / N;
  }
  return 0;
}

int orc_version(void) { return 1; }

}  // extern "C"

/*
 * dpsync.h - C ABI of the GB300 data-parallel gradient synchronisation library
 * (libdpsync.so).
 *
 * P "virtual ranks" are data-parallel replicas whose bf16 gradient and bf16
 * parameter copies all live in one GPU's HBM.  The library performs, as CUDA
 * kernels over those replicas, the synchronisation step that the pages on
 * data parallelism define:
 *   - gradients packed into buckets in reverse layer order
 *     ("4.1 Data parallelism in depth", sec. 4.2 "The Bucket mechanism");
 *   - the mean all-reduce G = sum_i G_i / N, decomposed into a reduce-scatter
 *     and an all-gather ("Data Parallelism: From Parameter Server to Ring All-Reduce", sec. 1
 *     and sec. 5, the ring's two phases);
 *   - the ZeRO-1/2 step: reduce-scatter, update the owned shard with AdamW on
 *     fp32 master/m/v, all-gather the updated bf16 parameters ("Data
 *     Parallelism: DDP, ZeRO and FSDP", "The three stages"), with optional
 *     global gradient-norm clipping ("Distributed Training: Data Parallel, Model Parallel and FSDP Strategies",
 *     "Inside DDP": the gradients are clipped to norm 1.0 after averaging).
 *
 * Conventions shared by every call
 * --------------------------------
 * Ownership.  The caller owns all device memory and the stream.  The library
 *   allocates no device memory: the workspace is a caller buffer of
 *   dp_plan_info().workspace_bytes bytes.  A plan is host memory owned by the
 *   library, immutable after dp_plan_buckets() and safe to share between
 *   threads.
 * Layout.  Element i of the "flat padded index space" [0, L) is defined by the
 *   plan (dp_plan_tensor, dp_plan_bucket).  Replica buffers (gradients,
 *   parameters) are bf16 arrays [P][replica_stride]: replica r's element i is at
 *   r * replica_stride + i.  master, m, v and fp32 mean buffers are fp32 [L].
 *   Bucket b covers [offset_b, offset_b + len_b); its shard c is
 *   [offset_b + c*S_b, offset_b + (c+1)*S_b) with S_b = len_b / P, and rank c
 *   owns shard c (on a hybrid mesh, see dp_plan_buckets_mesh: S shards, shard s
 *   owned by rank (g, s) of every group g).  Padding slots (between tensors and at a bucket's end) must
 *   hold zeros in gradients and in master/m/v; the calls keep them zero.
 * Alignment.  Every device pointer must be 32-byte aligned (DP_EALIGN); the
 *   kernels move 32 bytes per access.
 * Streams.  `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   Every compute call only enqueues work on it and never synchronises the
 *   device, except dp_read_norm, which synchronises `stream`.  Kernel-side
 *   errors surface when the caller synchronises; dp_read_norm reports the
 *   workspace's status bits.  Kernels are launched as programmatic dependents
 *   of the previous kernel in the stream: a launch is prepared while that
 *   kernel runs, but no kernel of the library reads or writes memory before
 *   its predecessor has finished and its writes are visible, so the stream's
 *   ordering is that of plain launches, with other libraries' kernels too.
 *   The environment variable DPSYNC_PDL=0 (read once per process) gives plain
 *   launches.
 * Buckets.  [b0, b1) selects a range of buckets (0 <= b0 <= b1 <= n_buckets),
 *   so a caller can launch per bucket (DDP's bucket-ready semantics) or once
 *   for all buckets.
 * Errors.  0 is success; negative values are DP_E*.  dp_last_error() returns a
 *   thread-local message for the last failing call on this thread.
 * Numerics.  Sums are fp32, taken for shard c of every bucket in the ring's
 *   order: rank c+1 first, then c+2, ..., ending with rank c (indices mod P);
 *   the mean is that sum divided by P in IEEE fp32; bf16 results round to
 *   nearest even.  AdamW runs in fp32 without fused multiply-add.
 */
#ifndef DPSYNC_H
#define DPSYNC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  DP_OK = 0,
  DP_EINVAL = -1,      /* bad argument, size, rank or bucket range */
  DP_EALIGN = -2,      /* a device pointer is not 32-byte aligned */
  DP_EPLAN = -3,       /* workspace does not hold this plan's uploaded image */
  DP_ECUDA = -4,       /* a CUDA runtime call or kernel launch failed */
  DP_ENONFINITE = -5,  /* the global gradient norm was not finite */
  DP_ENOMEM = -6,      /* host allocation failed */
  DP_ETIMEOUT = -7     /* a kernel's bounded wait on its own copies gave up */
};

/* Status bits written by kernels into the workspace, read by dp_read_norm. */
enum {
  DP_STATUS_PLAN_MISMATCH = 1,
  DP_STATUS_NONFINITE = 2,
  DP_STATUS_TIMEOUT = 4,
  DP_STATUS_NO_SCALARS = 8   /* an update ran without a cfg before dp_set_adamw_cfg */
};

/*
 * Where a workspace keeps the results the kernels write, as byte offsets from
 * the workspace's start (device memory): the squared global norm (double), the
 * norm (double), the clip coefficient (float) and the status bits (int32,
 * DP_STATUS_*).  dp_read_norm synchronises and reads them; a caller may instead
 * copy them itself after ordering the copy after the kernels, or pass
 * workspace + DP_WS_COEF_OFFSET as an update's coef_dev.
 * dp_workspace_result_offsets reports the same four values from the library.
 */
enum {
  DP_WS_NORM2_OFFSET = 112,
  DP_WS_NORM_OFFSET = 120,
  DP_WS_COEF_OFFSET = 128,
  DP_WS_STATUS_OFFSET = 132
};

typedef struct dp_plan dp_plan;

typedef struct {
  int64_t n_params;         /* sum of the tensor sizes */
  int64_t padded_len;       /* L: length of the flat padded index space */
  int64_t replica_stride;   /* elements between consecutive replicas, >= L, multiple of 128 */
  int64_t bucket_bytes;     /* the cap the plan was made with */
  int32_t n_tensors;
  int32_t n_buckets;
  int32_t P;
  int32_t tile_elems;       /* elements per work tile (tiles never cross a bucket) */
  int32_t R, S;             /* mesh: R replicate groups x S shards (flat plans: 1 x P) */
  int32_t pad_;
  int64_t n_tiles;
  int64_t table_bytes;      /* device plan image at the start of the workspace */
  int64_t workspace_bytes;  /* whole workspace: image + norm scratch + fp32 mean stage [L] */
} dp_plan_info_t;

/* AdamW hyperparameters for one step.  max_norm <= 0 disables clipping. */
typedef struct {
  double lr, beta1, beta2, eps, weight_decay, max_norm;
  int64_t step; /* t >= 1 */
} dp_adamw_cfg;

/*
 * Bucket planner.  Gradients are packed into buckets of about 25 MB (one
 * collective per bucket), filled in the reverse of the order the forward pass
 * computes them ("4.1 Data parallelism in depth", sec. 4.2; PyTorch's
 * bucket_cap_mb).  Rule: walk tensors n-1 ... 0; each takes a
 * slot of ceil(size/8)*8 elements (16-byte aligned); a non-empty bucket is
 * closed when adding the next slot would exceed bucket_bytes/2 elements; a
 * tensor is never split (one larger than the cap forms its own bucket); a
 * closed bucket is padded up to a multiple of 16P, so each of its P shards is a
 * whole number of 32-byte blocks (the kernels' 256-bit access unit).
 *   sizes[n_tensors]  element count of each tensor (>= 0), host memory.
 *   decay[n_tensors]  1 = weight decay applies to the tensor, 0 = not; NULL = all.
 *   bucket_bytes      cap in bytes of bf16 gradient (>= 2).
 *   P                 number of virtual ranks, 1..64.
 *   out               receives the plan; free with dp_plan_free.
 * Returns DP_EINVAL on bad arguments, DP_ENOMEM if host memory runs out.
 */
int dp_plan_buckets(const int64_t* sizes, const uint8_t* decay, int32_t n_tensors,
                    int64_t bucket_bytes, int32_t P, dp_plan** out);

/* Same, with an explicit replica stride (elements; 0 = the default, the
 * smallest multiple of 128 >= L plus 128).  A stride < L or not a multiple of
 * 128 is DP_EINVAL. */
int dp_plan_buckets_ex(const int64_t* sizes, const uint8_t* decay, int32_t n_tensors,
                       int64_t bucket_bytes, int32_t P, int64_t replica_stride, dp_plan** out);

/*
 * Same, on a hybrid R x S device mesh (P = R * S ranks; rank (g, s) = g*S + s):
 * HYBRID_SHARD, full sharding within a group of ranks and plain data
 * parallelism between the groups ("4.1 Data parallelism in depth", sec. 6.3); FSDP2's DeviceMesh mesh_shape=(2, 4)
 * with dims ("replicate", "shard") ("Distributed Training: Data Parallel, Model
 * Parallel and FSDP Strategies", "FSDP1 vs FSDP2"); "Data Parallelism: DDP, ZeRO
 * and FSDP", "Hybrid sharding".  Each bucket is split into S shards, shard s
 * owned by rank (g, s) in every group g.  The sums follow the hierarchical
 * rings: a ring reduce-scatter inside each group of S ranks, then a ring
 * all-reduce of each shard across the R groups (R sub-chunks); so element i of
 * shard s in sub-chunk j (of R) is
 *   sum over groups g = j+1, ..., j (mod R) of
 *     [sum over members s' = s+1, ..., s (mod S) of grad(g, s')[i]]
 * in fp32, left to right.  R = 1 is the flat ring over P = S ranks.
 */
int dp_plan_buckets_mesh(const int64_t* sizes, const uint8_t* decay, int32_t n_tensors,
                         int64_t bucket_bytes, int32_t R, int32_t S, int64_t replica_stride,
                         dp_plan** out);

int dp_plan_info(const dp_plan* plan, dp_plan_info_t* out);

/* Tensor t lives in bucket *bucket at flat offset *offset (16-byte aligned). */
int dp_plan_tensor(const dp_plan* plan, int32_t t, int32_t* bucket, int64_t* offset);

/* Bucket b: flat offset, padded length len_b and shard length len_b / S (S = P
 * for flat plans). */
int dp_plan_bucket(const dp_plan* plan, int32_t b, int64_t* offset, int64_t* padded_len,
                   int64_t* shard_len);

void dp_plan_free(dp_plan* plan);

/*
 * Cross-process plan check.  Every rank must pack its gradients into the same
 * buckets in the same order, or the collectives of different ranks no longer
 * line up and the job hangs ("4.1 Data parallelism in depth", sec. 4.2 on the
 * bucket mechanism; "Data Parallelism: DDP, ZeRO and FSDP", "DDP, and why it
 * works").  Processes that each build their own plan compare them before the
 * first step and get an error instead of a hang.
 *
 * dp_plan_fingerprint: *out = a 64-bit FNV-1a hash of the layout, identical on
 *   every platform: P, the mesh shape (R, S), the padded length L, and per
 *   tensor its size, decay flag, flat offset and bucket, per bucket its offset
 *   and padded length (each as 8 little-endian bytes, in that order, after a
 *   format tag).  The bucket cap and the replica stride are not part of it: two
 *   caps that give the same buckets give the same fingerprint, and each
 *   process's replica buffers are its own.  Host only; DP_EINVAL on NULL.
 * dp_plan_check_match: fingerprints[0..n_ranks) are the values every rank
 *   computed (gathered by the caller, e.g. over torch.distributed); DP_OK if all
 *   equal this plan's, else DP_EPLAN naming the first rank that differs.
 *   DP_EINVAL for NULL fingerprints with n_ranks > 0 or n_ranks < 0.
 */
int dp_plan_fingerprint(const dp_plan* plan, uint64_t* out);
int dp_plan_check_match(const dp_plan* plan, const uint64_t* fingerprints, int32_t n_ranks);

/*
 * Copy the plan's device image (bucket/tile tables, decay bits) into the first
 * table_bytes of `workspace` (device, workspace_bytes long) on `stream`.  Must
 * run once before any compute call uses that workspace; a compute call given a
 * workspace holding another plan's image does no work and sets
 * DP_STATUS_PLAN_MISMATCH.
 */
int dp_plan_upload(const dp_plan* plan, void* workspace, void* stream);

/*
 * Launch shape of the compute calls enqueued on one stream.  DDP and FSDP run
 * their collectives beside the backward ("4.1 Data parallelism in depth",
 * sec. 4.2; "Data Parallelism: DDP, ZeRO and FSDP", "How FSDP actually runs");
 * here those collectives are kernels that share the SMs with the backward's.
 *   DP_LAUNCH_DEFAULT     (every stream's default; DP_LAUNCH_PERSISTENT is its
 *                         older name) each kernel's own shape: short-lived CTAs,
 *                         eight 64-thread CTAs per tile, one block per thread, for
 *                         the all-reduce, the reduce-scatter, the update passes and
 *                         the write-back; a persistent grid (at most the CTAs the
 *                         GPU holds at once, each walking many tiles) for the mesh
 *                         reduce-scatter, the accumulating reduce-scatter and any
 *                         launch a tracker's max_ctas caps below its pieces.
 *   DP_LAUNCH_SHORT_CTAS  short-lived CTAs for every kernel, the persistent ones
 *                         as one CTA per tile, caps ignored.  Each CTA holds its SM
 *                         for microseconds, so a kernel of a higher-priority stream
 *                         waiting for SMs (a GEMM wave) gets them almost at once.
 *                         For a stream of the lowest priority beside a compute
 *                         stream of a higher one (cudaStreamCreateWithPriority).
 * Every call enqueued on `stream` afterwards, from any host thread, takes the
 * shape, except the bulk-copy kernels selected by DPSYNC_AG_BULK / DPSYNC_REP_BULK
 * (kept for comparison) and dp_clip_coef_noalloc; a tracker whose stream is set
 * fires as with DP_TRACK_SHORT_CTAS.  Results do not depend on the shape, bit for
 * bit.  The setting is host state kept per stream handle (NULL: the legacy
 * default stream); it costs an uncontended lock per call while any stream is
 * set.  Set DP_LAUNCH_DEFAULT again before destroying a stream: CUDA may give
 * its handle to a later stream.  DP_EINVAL for another shape.
 */
enum { DP_LAUNCH_DEFAULT = 0, DP_LAUNCH_PERSISTENT = 0, DP_LAUNCH_SHORT_CTAS = 1 };
int dp_stream_set_launch(void* stream, int32_t shape);
int dp_stream_get_launch(void* stream, int32_t* shape);

/*
 * Reduce-scatter + mean ("Data Parallelism: From Parameter Server to Ring All-Reduce", sec. 5:
 * the first N-1 ring steps leave each rank holding the complete sum of one
 * chunk; sec. 1: the synchronised gradient is the ranks' average).
 *   grads   bf16 [P][replica_stride], read only.
 *   mean    fp32 [L]; for each bucket in [b0,b1), shard c's slots receive the
 *           fp32 mean that rank c owns.
 *   want_sumsq  non-zero: also store per-tile sums of mean^2 in the workspace
 *           for dp_clip_coef (warp-shuffle partials, fixed order).
 */
int dp_reduce_scatter_mean(const dp_plan* plan, void* workspace, const void* grads, float* mean,
                           int32_t b0, int32_t b1, int32_t want_sumsq, void* stream);

/*
 * Global gradient-norm clip coefficient over buckets [b0,b1) from the partials
 * of a preceding dp_reduce_scatter_mean(want_sumsq=1) over the same buckets
 * ("Distributed Training: Data Parallel, Model Parallel and FSDP Strategies", "Inside DDP":
 * the averaged gradients are clipped to a global norm of 1.0).
 * norm = sqrt(sum mean^2) (partials summed in double in tile order);
 * coef = min(1, max_norm / (norm + 1e-6)), or 1 when max_norm <= 0; a
 * non-finite norm gives coef = NaN and sets DP_STATUS_NONFINITE.  Results stay
 * in the workspace (dp_read_norm reads them).
 */
int dp_clip_coef(const dp_plan* plan, void* workspace, double max_norm, int32_t b0, int32_t b1,
                 void* stream);

/*
 * The clip coefficient of an update (use_clip_coef, coef_dev), shared by
 * dp_sharded_adamw_step, dp_adamw_all_gather and dp_shard_adamw_step:
 *   use_clip_coef = 0, coef_dev = NULL   coef = 1 (no clipping);
 *   use_clip_coef != 0, coef_dev = NULL  coef = the workspace's, from the last
 *                                        dp_clip_coef on it;
 *   use_clip_coef != 0, coef_dev != NULL coef = *coef_dev, one device float the
 *                                        caller formed itself (its own
 *                                        clip_grad_norm_), 4-byte aligned, read
 *                                        when the kernel runs (stream order);
 *   use_clip_coef = 0, coef_dev != NULL  DP_EINVAL.
 * The gradient is multiplied by coef in fp32 before AdamW
 * ("Distributed Training: Data Parallel, Model Parallel and FSDP Strategies",
 * "Inside DDP": clip after averaging, then optimizer.step()).
 */

/*
 * Sharded AdamW ("Data Parallelism: DDP, ZeRO and FSDP", "The three stages":
 * each rank updates the shard it owns; "Distributed Training: Data Parallel, Model Parallel and FSDP Strategies",
 * "Inside DDP": torch.optim.AdamW(lr, weight_decay)).  For every slot i of the
 * shards of buckets [b0,b1), owned by rank c:
 *   g = grad[i] * coef   (coef from use_clip_coef / coef_dev, above)
 *   theta = master[i] * (1 - lr*wd)          if the slot's tensor decays
 *   m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*(g*g)
 *   theta -= (lr / (1-b1^t)) * (m / (sqrt(v) / sqrt(1-b2^t) + eps))
 *   params[c][i] = bf16(theta)   (only the owner's replica is written)
 *   grad, master, m, v  fp32 [L] (master/m/v updated in place)
 *   params              bf16 [P][replica_stride]
 */
int dp_sharded_adamw_step(const dp_plan* plan, void* workspace, const float* grad, float* master,
                          float* m, float* v, void* params, const dp_adamw_cfg* cfg,
                          int32_t use_clip_coef, const float* coef_dev, int32_t b0, int32_t b1,
                          void* stream);

/*
 * All-gather, in place ("Data Parallelism: From Parameter Server to Ring All-Reduce", sec. 5:
 * the second phase passes the reduced chunks around the ring so that all ranks
 * end with the whole result): for every
 * shard c of buckets [b0,b1), copy params[c][shard c] into every other replica.
 */
int dp_all_gather(const dp_plan* plan, void* workspace, void* params, int32_t b0, int32_t b1,
                  void* stream);

/*
 * Broadcast replica `src` into every other replica over buckets [b0,b1): the
 * one-time start-up broadcast of rank 0's parameters ("4.1 Data parallelism in
 * depth", sec. 4.1: parameters are copied from one rank once at the start,
 * gradients are synchronised every step).
 */
int dp_broadcast(const dp_plan* plan, void* workspace, void* params, int32_t src, int32_t b0,
                 int32_t b1, void* stream);

/*
 * Mean all-reduce in place (DDP / NO_SHARD): reduce-scatter, mean, and the
 * all-gather of bf16(mean) fused in one pass with no shard buffer ("4.1 Data
 * parallelism in depth", sec. 5.1 AllReduce = ReduceScatter + AllGather;
 * sec. 2: averaged, not summed).  grads bf16 [P][replica_stride], in/out.
 */
int dp_allreduce_mean(const dp_plan* plan, void* workspace, void* grads, int32_t b0, int32_t b1,
                      void* stream);

/*
 * The fused ZeRO-1/2 step over all buckets ("Data Parallelism: DDP, ZeRO and
 * FSDP", "The three stages": reduce-scatter, update the owned shard, all-gather
 * the updated parameters).  Without clipping it is one kernel that reads the P
 * gradient replicas and master/m/v once and writes master/m/v and the P
 * parameter replicas once.  With clipping (cfg->max_norm > 0) it is
 * dp_reduce_scatter_mean(want_sumsq) into the workspace's fp32 stage, then
 * dp_clip_coef, then one kernel fusing AdamW with the all-gather.
 *   grads   bf16 [P][replica_stride], read only.
 *   params  bf16 [P][replica_stride], written (every replica, bit-identical).
 *   master, m, v  fp32 [L], in/out.
 *   stage_events  NULL, or dp_fused_zero_step_launches(cfg)+1 cudaEvent_t
 *           handles the call records on `stream` before its first launch and
 *           after each launch (for per-kernel timing by the caller).
 */
int dp_fused_zero_step(const dp_plan* plan, void* workspace, const void* grads, void* params,
                       float* master, float* m, float* v, const dp_adamw_cfg* cfg,
                       void* const* stage_events, void* stream);

/*
 * The clipped step's second pass on its own: AdamW on mean * coef fused with
 * the all-gather of bf16(theta) into every replica, over all buckets ("Data
 * Parallelism: DDP, ZeRO and FSDP", "The three stages").  Use after per-bucket
 * reduce-scatters (e.g. from a tracker) and dp_clip_coef.
 *   mean     fp32 [L] (input: the reduce-scatter mean of every bucket)
 *   master, m, v fp32 [L] (in/out);  params bf16 [P][replica_stride] (out)
 *   use_clip_coef, coef_dev  the clip coefficient (see above dp_sharded_adamw_step).
 */
int dp_adamw_all_gather(const dp_plan* plan, void* workspace, const float* mean, float* master,
                        float* m, float* v, void* params, const dp_adamw_cfg* cfg,
                        int32_t use_clip_coef, const float* coef_dev, void* stream);

/*
 * ZeRO-3 / FULL_SHARD unit flow ("Data Parallelism: DDP, ZeRO and FSDP", "How
 * FSDP actually runs": per unit, all-gather the parameter shards before the
 * forward, again before the backward, reduce-scatter the gradients after it,
 * then each rank steps only its shard; "4.1 Data parallelism in depth",
 * sec. 6.2).  Units are the plan's buckets.  Persistent state is sharded: one
 * flat bf16 [L] array of parameter shards (element i held by its shard owner),
 * fp32 [L] master/m/v and an fp32 [L] mean (the gradient shards): 18 bytes per
 * parameter across all P ranks.  The unit buffers are transient:
 * [P][unit_stride] bf16 (unit_stride >= the unit's padded length, a multiple of
 * 16), one row per rank.
 *
 * dp_unit_all_gather: every rank's full copy of unit `unit`:
 *   unit_buf[r][i] = param_shards[offset_unit + i], r < P, i < len_unit.
 * dp_unit_reduce_scatter: the unit's gradients, rank r's in unit_grads[r][0..len),
 *   reduced in ring order to the fp32 mean of each owner's shard:
 *   mean[offset_unit + i]; want_sumsq also stores the unit's norm partials.
 * An empty unit (a bucket of zero-size tensors only) is a no-op for both calls;
 * its buffer pointers are not checked.
 * dp_shard_adamw_step: AdamW over all buckets on mean (times the clip
 *   coefficient chosen by use_clip_coef / coef_dev, as for dp_sharded_adamw_step),
 *   writing bf16(theta) to param_shards.
 */
int dp_unit_all_gather(const dp_plan* plan, void* workspace, const void* param_shards, int32_t unit,
                       void* unit_buf, int64_t unit_stride, void* stream);
int dp_unit_reduce_scatter(const dp_plan* plan, void* workspace, const void* unit_grads,
                           int64_t unit_stride, int32_t unit, float* mean, int32_t want_sumsq,
                           void* stream);
int dp_shard_adamw_step(const dp_plan* plan, void* workspace, const float* mean, float* master,
                        float* m, float* v, void* param_shards, const dp_adamw_cfg* cfg,
                        int32_t use_clip_coef, const float* coef_dev, void* stream);
/*
 * dp_unit_backward: one backward step of the unit flow in one launch — the
 * gather of unit gather_unit into gather_buf (the next unit's parameters, FSDP's
 * prefetch) and the reduce-scatter of unit rs_unit's gradients into mean: the
 * same results as dp_unit_all_gather(gather_unit) and
 * dp_unit_reduce_scatter(rs_unit), in either order.  gather_unit = -1 or
 * rs_unit = -1 leaves that part out (one of the two calls above; both -1: no
 * work).  Arguments as for those calls; gather_buf must not overlap unit_grads
 * or mean (DP_EINVAL), and the caller must not let unit_grads alias
 * param_shards.  Units outside [-1, n_buckets) are DP_EINVAL.
 */
int dp_unit_backward(const dp_plan* plan, void* workspace, const void* param_shards,
                     int32_t gather_unit, void* gather_buf, int64_t gather_stride,
                     const void* unit_grads, int64_t grads_stride, int32_t rs_unit, float* mean,
                     int32_t want_sumsq, void* stream);

/*
 * Gradient accumulation ("Distributed Training: Data Parallel, Model Parallel and
 * FSDP Strategies", "Selecting and Tuning": no_sync on every micro-batch but the
 * last, which alone is synchronised).  Each rank accumulates its bf16
 * gradients as autograd does for bf16 gradients: acc = bf16(acc + g), the add in
 * fp32, rounding to nearest even.
 * dp_accumulate: acc[r] = bf16(acc[r] + micro[r]) for every replica, buckets [b0,b1).
 * dp_allreduce_mean_accum: the last micro-batch fused with the sync: every rank's
 *   bf16(acc + micro) is reduced (ring order, fp32) and the bf16 mean written to
 *   every replica of acc — one pass instead of dp_accumulate + dp_allreduce_mean.
 *   acc, micro: bf16 [P][replica_stride].
 */
int dp_accumulate(const dp_plan* plan, void* workspace, void* acc, const void* micro, int32_t b0,
                  int32_t b1, void* stream);
int dp_allreduce_mean_accum(const dp_plan* plan, void* workspace, void* acc, const void* micro,
                            int32_t b0, int32_t b1, void* stream);
/* The ZeRO form of the same fusion: the last micro-batch's bf16(acc + micro) of
 * every rank reduce-scattered into the fp32 mean (as dp_reduce_scatter_mean, with
 * the optional norm partials); acc and micro are only read.  Flat plans only. */
int dp_reduce_scatter_mean_accum(const dp_plan* plan, void* workspace, const void* acc,
                                 const void* micro, float* mean, int32_t b0, int32_t b1,
                                 int32_t want_sumsq, void* stream);

/*
 * The mean all-reduce with bf16 on the wire, as a precision comparison
 * ("Data Parallelism: From Parameter Server to Ring All-Reduce", sec. 8: the dtype
 * the gradients travel in affects both the bytes moved and the numerics):
 * every ring hop's partial sum is rounded to bf16 (the add in fp32),
 * the owner's sum is divided by P in fp32 and rounded to bf16.  Flat plans only.
 */
int dp_allreduce_mean_bf16wire(const dp_plan* plan, void* workspace, void* grads, int32_t b0,
                               int32_t b1, void* stream);

/*
 * Checkpoint and resume of the optimizer state (fp32 master, m, v in the plan's
 * flat layout, and the step t).  The pages name the optimizer state as what a
 * ZeRO step carries between steps ("Data Parallelism: DDP, ZeRO and FSDP", "The
 * three stages"; "4.1 Data parallelism in depth", sec. 7) and note FSDP2's clearer
 * checkpoint semantics (sec. 6.4); the file format is this library's own.
 * The file holds the arrays in tensor order without padding, so a checkpoint
 * saved under one plan loads into any plan over the same tensor sizes (another
 * bucket size, rank count or mesh).  Layout, little-endian: 80-byte header
 * (magic "DPSYNCK1", u32 version 1, u32 arrays mask: bit 0 master, 1 m, 2 v;
 * i64 n_tensors, n_params, step; u64 checksum; i32 P, R, S, 0; i64 bucket_bytes;
 * 8 zero bytes), i64 sizes[n_tensors], then each present array as f32[n_params].
 * checksum: 64-bit FNV-1a over the bytes after the header in 8-byte
 * little-endian words (last word zero-padded).
 *
 * save: a NULL array is left out (at least one is required).  Writes path.tmp,
 *   then renames it over path.  Synchronises `stream` first (device mode).
 * load: a NULL destination skips that array; a requested array the file lacks is
 *   DP_EINVAL; tensor sizes that differ from the plan's are DP_EPLAN (checked before
 *   anything is written).  Padding slots are set to 0.  A checksum mismatch is
 *   found at the end (DP_EINVAL; the destinations then hold partial data).  *step
 *   (nullable) receives t.  Synchronous on `stream`.
 * flags: DP_CKPT_HOST = the arrays are host memory (no CUDA call is made).
 * Errors: DP_EINVAL (path, I/O, format), DP_EPLAN, DP_ENOMEM, DP_ECUDA.
 */
#define DP_CKPT_HOST 1
int dp_checkpoint_save(const dp_plan* plan, const char* path, const float* master, const float* m,
                       const float* v, int64_t step, int32_t flags, void* stream);
int dp_checkpoint_load(const dp_plan* plan, const char* path, float* master, float* m, float* v,
                       int64_t* step, int32_t flags, void* stream);

/*
 * Failure detection without a GPU fault.  The pages' hangs come from waits that
 * never end (an unready bucket, "4.1 Data parallelism in depth", sec. 4.2 note);
 * here every device wait is bounded.  This call checks that path: one CTA arms a
 * shared-memory mbarrier for 16 bytes that no copy delivers, waits with the same
 * bounded wait the bulk-copy kernels use (limit_ns of the global timer, in
 * [1e3, 1e10]), writes status_dev[0] = DP_STATUS_TIMEOUT (0 had the wait
 * completed) and status_dev[1] = milliseconds waited, and returns.  The context
 * stays usable.  status_dev: device int32[2], 8-byte aligned.  Asynchronous.
 */
int dp_selftest_bounded_wait(int32_t* status_dev, int64_t limit_ns, void* stream);

/*
 * Index checks.  A library built with -DDPSYNC_CHECKED (libdpsync_checked.so)
 * tests every tile descriptor, block index, shard owner and replica index against
 * the plan before the access; a failed check is counted and the access skipped,
 * never trapped (the stand-in for a memory checker).  Returns the count since the
 * last reset (reset != 0 zeroes it; synchronises the device), -1 for a library
 * built without checks, -2 if the counters cannot be read.
 */
int64_t dp_bounds_violations(int32_t reset);

/*
 * CUDA-graph capture of whole steps.  The update kernels take AdamW's per-step
 * scalars as launch arguments, which a captured graph would freeze.  This call
 * forms them from cfg on the host (exactly as the per-call path does) and copies
 * them into the workspace on `stream`; dp_sharded_adamw_step, dp_adamw_all_gather
 * and dp_shard_adamw_step called with cfg = NULL then read them from there when
 * they run.  So: capture the step once with cfg = NULL, and before each replay call
 * dp_set_adamw_cfg with that step's cfg (outside the graph).  An update that runs
 * with cfg = NULL before any dp_set_adamw_cfg on this workspace skips its work and
 * sets DP_STATUS_NO_SCALARS.  dp_plan_upload clears the scalars.  The host copy is
 * staged by the driver before this call returns (cfg need not outlive it).
 */
int dp_set_adamw_cfg(const dp_plan* plan, void* workspace, const dp_adamw_cfg* cfg, void* stream);

/* offsets[0..3] = DP_WS_NORM2_OFFSET, DP_WS_NORM_OFFSET, DP_WS_COEF_OFFSET,
 * DP_WS_STATUS_OFFSET as the library was built (host only; DP_EINVAL on NULL). */
int dp_workspace_result_offsets(int64_t* offsets);

/* Number of kernel launches dp_fused_zero_step makes for cfg (1 or 3). */
int dp_fused_zero_step_launches(const dp_adamw_cfg* cfg);

/*
 * Streamed per-bucket synchronisation: DDP's bucket readiness.  As soon as all
 * of a bucket's gradients exist its all-reduce starts, while backward continues
 * through the earlier layers ("4.1 Data parallelism in depth", sec. 4.2); the
 * communication runs on its own stream beside the computation ("Distributed
 * Training: Data Parallel, Model Parallel and FSDP Strategies", "Inside DDP");
 * buckets fire in the same order every step ("Data Parallelism: DDP, ZeRO and
 * FSDP", "DDP, and why it works": bucket order must match).
 *
 * A tracker belongs to one plan and one set of buffers.  Each step: begin, then
 * mark every tensor ready (from any host thread) as its gradient is written,
 * passing a CUDA event recorded after that write (or NULL when the write is
 * already ordered before comm_stream's work); dp_tracker_mark_ready_batch marks
 * many tensors, each with its own event, in one call, and
 * dp_tracker_mark_ready_range a run of tensors (e.g. one layer's) with one event.
 * When bucket b and every bucket before it in plan order are complete, the
 * tracker makes comm_stream wait once for each distinct event of the bucket's
 * tensors and launches the bucket's reduction there.  Consecutive complete
 * buckets whose tensors all carry the same event (or none) become ready together
 * and go out as one launch over their tiles (the same results as one launch per
 * bucket; with DP_TRACK_SHORT_CTAS one launch per bucket all the same); a bucket
 * whose tensors carry different events goes out on its own:
 *   DP_TRACK_ALLREDUCE       the in-place mean all-reduce of `grads`;
 *   DP_TRACK_REDUCE_SCATTER  the reduce-scatter mean into `mean` with norm
 *                            partials (follow with dp_clip_coef and
 *                            dp_adamw_all_gather on comm_stream);
 *   DP_TRACK_ZERO_STEP       the whole ZeRO-1/2 step of the bucket without
 *                            clipping: reduce-scatter, AdamW on each owner's
 *                            shard and all-gather of the new parameters in one
 *                            pass over the bucket (dp_fused_zero_step on
 *                            [b, b+1)); set the targets and the step's AdamW
 *                            settings with dp_tracker_set_zero_step.  `mean` is
 *                            not used.  With clipping every update needs the
 *                            global norm of all buckets first, so a clipped step
 *                            uses DP_TRACK_REDUCE_SCATTER instead.
 * dp_tracker_wait returns once every bucket has been launched, or DP_ETIMEOUT
 * after timeout_ms naming tensors never marked (DDP would hang there).  It does
 * not synchronise the GPU: order later work after comm_stream.
 *   max_ctas   cap on each launch's grid (0 = no cap), to leave SMs to the
 *              backward running beside it: a launch whose short CTAs exceed the
 *              cap runs on a persistent grid of at most max_ctas CTAs.
 *   flags      DP_TRACK_DRY_RUN: record the firing order, launch nothing.
 *              DP_TRACK_SHORT_CTAS: every bucket goes out as its own launch
 *              (no merging of buckets that became ready together) of
 *              short-lived CTAs, as DP_LAUNCH_SHORT_CTAS gives them (eight
 *              64-thread CTAs per tile, one CTA per tile for the kernels that
 *              are otherwise persistent); max_ctas (and side_ctas) are then
 *              ignored.  Such a CTA holds its SM for microseconds, so a kernel of
 *              higher priority waiting for SMs gets them almost at once.  Meant
 *              for comm_stream at the lowest priority and the backward's stream
 *              at a higher one (cudaStreamCreateWithPriority): its GEMM waves
 *              then take the SMs first and the reductions fill the SMs the GEMMs
 *              leave idle and the gaps between them.  Results are those of the
 *              other launches, bit for bit.
 *              Other bits: DP_EINVAL.
 * Events are the caller's: keep them alive and unrecorded until their bucket
 * fires.  Marking a tensor twice in one step is DP_EINVAL.
 * Parameters that a step does not use (a skipped branch) never get a gradient,
 * so their bucket would never fire ("4.1 Data parallelism in depth", sec. 4.2
 * note).  DDP's find_unused_parameters marks them ready after the forward pass;
 * here the caller does the same: zero their gradient slots and mark them ready
 * (event NULL) as soon as it knows they are unused.
 */
typedef struct dp_tracker dp_tracker;
enum { DP_TRACK_ALLREDUCE = 0, DP_TRACK_REDUCE_SCATTER = 1, DP_TRACK_ZERO_STEP = 2 };
enum { DP_TRACK_DRY_RUN = 1, DP_TRACK_SHORT_CTAS = 2 };

int dp_tracker_create(const dp_plan* plan, int32_t mode, void* workspace, void* grads, float* mean,
                      void* comm_stream, int32_t max_ctas, int32_t flags, dp_tracker** out);
/* Gradient accumulation: with micro set (bf16 [P][replica_stride], 32-byte
 * aligned), each bucket's launch fuses the last micro-batch's add — grads holds the
 * sum of the earlier micro-batches, micro the last one's gradients as backward
 * writes them; the reduction runs on bf16(grads + micro) (dp_allreduce_mean_accum
 * / dp_reduce_scatter_mean_accum per bucket).  NULL restores the plain reduction.
 * Flat plans only; refused (DP_EINVAL) while a step has fired some but not all
 * buckets. */
int dp_tracker_set_micro(dp_tracker* tracker, const void* micro);
/* DP_TRACK_ZERO_STEP: the parameter replicas (bf16 [P][replica_stride]), the fp32
 * master, m and v [L] that each bucket's step updates, and the step's AdamW
 * settings (copied; cfg->step is this step's t).  Call before the step's first
 * bucket fires, again for every step (t changes).  DP_EINVAL for another mode,
 * a NULL pointer or cfg, cfg->max_norm > 0 (clipping needs the global norm), a
 * micro-batch buffer set, or a step that has fired some but not all buckets;
 * DP_EALIGN for a pointer that is not 32-byte aligned.  A bucket that becomes
 * ready before any call fails its launch with DP_EINVAL. */
int dp_tracker_set_zero_step(dp_tracker* tracker, void* params, float* master, float* m, float* v,
                             const dp_adamw_cfg* cfg);
int dp_tracker_begin(dp_tracker* tracker);
int dp_tracker_mark_ready(dp_tracker* tracker, int32_t tensor, void* ready_event);
/* Tensors [t0, t1) ready, all written before ready_event: one call, one event.
 * DP_EINVAL for a range outside [0, n_tensors) or a tensor already marked in
 * this step (then nothing is marked). */
int dp_tracker_mark_ready_range(dp_tracker* tracker, int32_t t0, int32_t t1, void* ready_event);
/* tensors[0..n) ready, tensor[i] written before ready_events[i] (ready_events NULL:
 * no events): the per-tensor marks of dp_tracker_mark_ready in one call.
 * DP_EINVAL for a tensor out of range, already marked, or listed twice (then
 * nothing is marked). */
int dp_tracker_mark_ready_batch(dp_tracker* tracker, const int32_t* tensors,
                                void* const* ready_events, int32_t n);
/* Fire every bucket but the plan's last on side_stream (NULL: all on the tracker's
 * stream), with each launch's grid capped at side_ctas CTAs (0: no cap).  The last
 * bucket, ready only when backward ends, fires on the tracker's stream after it
 * has waited for side_stream's work, so all reductions are still ordered before
 * the tracker's stream.  Meant for the partition stream of dp_sm_streams_create,
 * with the backward on its rest stream.  Not while a step has
 * fired some but not all buckets (DP_EINVAL). */
int dp_tracker_set_side_stream(dp_tracker* tracker, void* side_stream, int32_t side_ctas);
/* This step so far: kernel launches made and cudaStreamWaitEvent calls issued
 * (with DP_TRACK_DRY_RUN: those that would have been; either pointer may be
 * NULL). */
int dp_tracker_stats(const dp_tracker* tracker, int32_t* launches, int32_t* waits);
int dp_tracker_wait(dp_tracker* tracker, int64_t timeout_ms);
/* Buckets launched so far this step, in launch order (up to cap entries). */
int dp_tracker_fired(const dp_tracker* tracker, int32_t* order, int32_t cap, int32_t* n_fired);
void dp_tracker_free(dp_tracker* tracker);

/*
 * Streams whose kernels run only on a partition of the GPU's SMs (green
 * contexts).  The GPU's SMs are split into groups of n_sms (rounded up to the
 * driver's partition granularity, 8 on this GPU family); *part_stream runs on the
 * first group, *rest_stream (if rest_stream is not NULL) on all the others.
 * n_sms must leave SMs outside the partition.  *n_part and *n_rest (nullable)
 * receive the two SM counts.  On one GPU the streamed mode's "communication" is
 * SM work: reductions on part_stream beside a backward whose GEMMs run on
 * rest_stream never take SMs from each other ("4.1 Data parallelism in depth",
 * sec. 4.2: the bucket's collective runs while backward continues); a backward
 * left on the whole GPU can still take the partition's SMs.  Measured on a
 * GEMM-heavy synthetic backward (cuBLAS, 2-CTA clusters): its GEMMs ran 21% slower
 * on 144 of 152 SMs, more than the reductions beside them gained, so the split
 * pays only where the producer does not need every SM.  Streams belong to
 * the current device; dp_sm_streams_destroy(handle) destroys both.  DP_ECUDA when
 * the driver lacks green contexts.  The library's kernels launch on them like on
 * any stream.
 */
int dp_sm_streams_create(int32_t n_sms, int32_t priority, void** part_stream, void** rest_stream,
                         void** handle, int32_t* n_part, int32_t* n_rest);
int dp_sm_streams_destroy(void* handle);

/*
 * Synchronise `stream` and read the workspace's last clip results: norm
 * (double), coef (fp32) and the status bits.  Any pointer may be NULL.
 * Returns DP_ENONFINITE if the non-finite bit is set, DP_EPLAN if a kernel saw
 * a plan mismatch, DP_ETIMEOUT if a kernel's bounded wait for its own
 * asynchronous copies gave up (its results for that step are not valid).
 */
int dp_read_norm(const dp_plan* plan, const void* workspace, double* norm, float* coef,
                 int32_t* status, void* stream);

/*
 * The pages have no counterpart for this call: it is a library convenience.
 * dp_reduce_scatter_mean(want_sumsq=1) + dp_clip_coef over all buckets,
 * for callers that cannot allocate device memory (a plugin handed buffers by a
 * host application that owns the memory pool, a framework whose caching
 * allocator must account for every byte, a loop where a cudaMalloc/cudaFree
 * that may synchronise the device is not acceptable).  Instead of a workspace
 * it uses a 32 MiB library-owned device array, held by every GPU that loads it
 * until the process exits; plans up to about 1.2e9 parameters fit (larger ones:
 * DP_EINVAL with the sizes in dp_last_error()).  It allocates nothing.
 *   grads     bf16 [P][replica_stride] (input, 32-byte aligned)
 *   mean      fp32 [L] (output, 32-byte aligned): the reduce-scatter mean
 *   max_norm  clip threshold (<= 0: coef = 1)
 *   coef_out  device float (output): min(1, max_norm / (norm + 1e-6))
 *   norm_out  device double (output): the global L2 norm of the mean
 * The status bits the kernels set stay in the library's array, where the caller
 * cannot read them: a non-finite gradient norm still returns DP_OK, with
 * *norm_out inf or NaN and *coef_out NaN (1 when max_norm <= 0), so a caller
 * checks *norm_out itself.
 * Every call shares the array and overwrites it; calls whose work overlaps on
 * the GPU (unordered streams, concurrent host threads) race and must be
 * serialised.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it.
 */
int dp_clip_coef_noalloc(const dp_plan* plan, const void* grads, float* mean, double max_norm,
                         float* coef_out, double* norm_out, void* stream);

/* Thread-local text of the last error on this thread ("" if none). */
const char* dp_last_error(void);

/* ABI version of this header (increments on incompatible change): 2. */
int dp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DPSYNC_H */

"""Python binding of libdpsync.so, the GB300 data-parallel gradient
synchronisation library.

Argument marshalling only: every step of the synchronisation runs in the CUDA
kernels behind the C ABI declared in include/dpsync.h.  PyTorch supplies device
memory (``tensor.data_ptr()``) and streams (``torch.cuda.current_stream()``).
There is no fallback: if the shared library is missing or fails to load, import
raises.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# DPSYNC_VARIANT=checked loads the build with device index checks compiled in.
VARIANT = os.environ.get("DPSYNC_VARIANT", "")
LIB_PATH = os.path.join(HERE, "libdpsync_checked.so" if VARIANT == "checked" else "libdpsync.so")

DP_OK, DP_EINVAL, DP_EALIGN, DP_EPLAN, DP_ECUDA, DP_ENONFINITE, DP_ENOMEM, DP_ETIMEOUT = \
    0, -1, -2, -3, -4, -5, -6, -7
DP_STATUS_PLAN_MISMATCH, DP_STATUS_NONFINITE, DP_STATUS_TIMEOUT, DP_STATUS_NO_SCALARS = 1, 2, 4, 8
DP_TRACK_ALLREDUCE, DP_TRACK_REDUCE_SCATTER, DP_TRACK_ZERO_STEP, DP_TRACK_DRY_RUN = 0, 1, 2, 1
DP_TRACK_SHORT_CTAS = 2
DP_LAUNCH_DEFAULT, DP_LAUNCH_SHORT_CTAS = 0, 1
DP_LAUNCH_PERSISTENT = DP_LAUNCH_DEFAULT     # the older name
DP_CKPT_HOST = 1


class DPError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{msg} (code {code})")
        self.code = code


class PlanInfo(C.Structure):
    _fields_ = [("n_params", C.c_int64), ("padded_len", C.c_int64), ("replica_stride", C.c_int64),
                ("bucket_bytes", C.c_int64), ("n_tensors", C.c_int32), ("n_buckets", C.c_int32),
                ("P", C.c_int32), ("tile_elems", C.c_int32), ("R", C.c_int32), ("S", C.c_int32),
                ("pad_", C.c_int32), ("n_tiles", C.c_int64),
                ("table_bytes", C.c_int64), ("workspace_bytes", C.c_int64)]


class AdamWCfg(C.Structure):
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double), ("beta2", C.c_double),
                ("eps", C.c_double), ("weight_decay", C.c_double), ("max_norm", C.c_double),
                ("step", C.c_int64)]


_lib = None


def lib():
    """Load libdpsync.so (raises if it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built; run gradient_sync_zero_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        vp, i32, i64, f64 = C.c_void_p, C.c_int32, C.c_int64, C.c_double
        sig = {
            "dp_plan_buckets": [vp, vp, i32, i64, i32, vp],
            "dp_plan_buckets_ex": [vp, vp, i32, i64, i32, i64, vp],
            "dp_plan_buckets_mesh": [vp, vp, i32, i64, i32, i32, i64, vp],
            "dp_plan_info": [vp, vp],
            "dp_plan_tensor": [vp, i32, vp, vp],
            "dp_plan_bucket": [vp, i32, vp, vp, vp],
            "dp_plan_upload": [vp, vp, vp],
            "dp_reduce_scatter_mean": [vp, vp, vp, vp, i32, i32, i32, vp],
            "dp_clip_coef": [vp, vp, f64, i32, i32, vp],
            "dp_sharded_adamw_step": [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, vp],
            "dp_all_gather": [vp, vp, vp, i32, i32, vp],
            "dp_broadcast": [vp, vp, vp, i32, i32, i32, vp],
            "dp_allreduce_mean": [vp, vp, vp, i32, i32, vp],
            "dp_fused_zero_step": [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp],
            "dp_fused_zero_step_launches": [vp],
            "dp_read_norm": [vp, vp, vp, vp, vp, vp],
            "dp_clip_coef_noalloc": [vp, vp, vp, f64, vp, vp, vp],
            "dp_adamw_all_gather": [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp],
            "dp_tracker_create": [vp, i32, vp, vp, vp, vp, i32, i32, vp],
            "dp_unit_all_gather": [vp, vp, vp, i32, vp, i64, vp],
            "dp_accumulate": [vp, vp, vp, vp, i32, i32, vp],
            "dp_selftest_bounded_wait": [vp, i64, vp],
            "dp_set_adamw_cfg": [vp, vp, vp, vp],
            "dp_checkpoint_save": [vp, C.c_char_p, vp, vp, vp, i64, i32, vp],
            "dp_checkpoint_load": [vp, C.c_char_p, vp, vp, vp, C.POINTER(i64), i32, vp],
            "dp_allreduce_mean_accum": [vp, vp, vp, vp, i32, i32, vp],
            "dp_reduce_scatter_mean_accum": [vp, vp, vp, vp, vp, i32, i32, i32, vp],
            "dp_allreduce_mean_bf16wire": [vp, vp, vp, i32, i32, vp],
            "dp_unit_reduce_scatter": [vp, vp, vp, i64, i32, vp, i32, vp],
            "dp_shard_adamw_step": [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp],
            "dp_workspace_result_offsets": [vp],
            "dp_unit_backward": [vp, vp, vp, i32, vp, i64, vp, i64, i32, vp, i32, vp],
            "dp_tracker_begin": [vp],
            "dp_tracker_set_micro": [vp, vp],
            "dp_tracker_mark_ready": [vp, i32, vp],
            "dp_tracker_mark_ready_range": [vp, i32, i32, vp],
            "dp_tracker_mark_ready_batch": [vp, vp, vp, i32],
            "dp_tracker_stats": [vp, vp, vp],
            "dp_tracker_set_side_stream": [vp, vp, i32],
            "dp_sm_streams_create": [i32, i32, vp, vp, vp, vp, vp],
            "dp_sm_streams_destroy": [vp],
            "dp_tracker_wait": [vp, i64],
            "dp_tracker_fired": [vp, vp, i32, vp],
            "dp_plan_fingerprint": [vp, vp],
            "dp_plan_check_match": [vp, vp, i32],
            "dp_tracker_set_zero_step": [vp, vp, vp, vp, vp, vp],
            "dp_stream_set_launch": [vp, i32],
            "dp_stream_get_launch": [vp, vp],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = C.c_int
        L.dp_plan_free.argtypes = [vp]
        L.dp_plan_free.restype = None
        L.dp_tracker_free.argtypes = [vp]
        L.dp_tracker_free.restype = None
        L.dp_bounds_violations.argtypes = [i32]
        L.dp_bounds_violations.restype = i64
        L.dp_last_error.argtypes = []
        L.dp_last_error.restype = C.c_char_p
        L.dp_version.restype = C.c_int
        _lib = L
    return _lib


def _check(rc):
    if rc != DP_OK:
        raise DPError(rc, lib().dp_last_error().decode())
    return rc


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _cfg_ref(cfg):
    """cfg=None: the update reads the scalars set by dp_set_adamw_cfg (graph capture)."""
    return None if cfg is None else C.byref(cfg)


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def _coef(coef_dev):
    """coef_dev: None, or a 1-element float32 CUDA tensor holding a clip
    coefficient the caller formed itself."""
    if coef_dev is None:
        return None
    _need(coef_dev, torch.float32, 1, "coef_dev")
    return _ptr(coef_dev)


def workspace_result_offsets():
    """Byte offsets of (norm2, norm, coef, status) in a workspace, from the library."""
    out = (C.c_int64 * 4)()
    _check(lib().dp_workspace_result_offsets(out))
    return tuple(out)


def _need(t, dtype, numel, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {numel}")


class Plan:
    """A bucket plan (host object of the library)."""

    def __init__(self, sizes, bucket_bytes, P, decay=None, replica_stride=0, mesh=None):
        """mesh=(R, S) with R*S == P gives a hybrid R x S plan (R groups of S shards)."""
        sizes = [int(s) for s in sizes]
        n = len(sizes)
        arr = (C.c_int64 * max(n, 1))(*sizes)
        dec = None
        if decay is not None:
            dec = (C.c_uint8 * max(n, 1))(*[1 if d else 0 for d in decay])
        h = C.c_void_p()
        if mesh is None:
            _check(lib().dp_plan_buckets_ex(arr, dec, n, int(bucket_bytes), int(P),
                                            int(replica_stride), C.byref(h)))
        else:
            R, S = (int(x) for x in mesh)
            if R * S != int(P):
                raise ValueError(f"mesh {mesh} does not multiply to P={P}")
            _check(lib().dp_plan_buckets_mesh(arr, dec, n, int(bucket_bytes), R, S,
                                              int(replica_stride), C.byref(h)))
        self._h = h
        info = PlanInfo()
        _check(lib().dp_plan_info(h, C.byref(info)))
        self.info = info
        self.sizes = sizes

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.dp_plan_free(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    P = property(lambda self: self.info.P)
    L = property(lambda self: self.info.padded_len)
    stride = property(lambda self: self.info.replica_stride)
    n_buckets = property(lambda self: self.info.n_buckets)

    def tensor(self, t):
        b, o = C.c_int32(), C.c_int64()
        _check(lib().dp_plan_tensor(self._h, int(t), C.byref(b), C.byref(o)))
        return b.value, o.value

    def bucket(self, b):
        o, n, s = C.c_int64(), C.c_int64(), C.c_int64()
        _check(lib().dp_plan_bucket(self._h, int(b), C.byref(o), C.byref(n), C.byref(s)))
        return o.value, n.value, s.value

    def tensor_offsets(self):
        return [self.tensor(t)[1] for t in range(len(self.sizes))]

    @property
    def fingerprint(self):
        """64-bit layout fingerprint (dp_plan_fingerprint), as a Python int."""
        out = C.c_uint64()
        _check(lib().dp_plan_fingerprint(self._h, C.byref(out)))
        return out.value

    def check_match(self, fingerprints):
        """dp_plan_check_match over a list of fingerprints (one per rank)."""
        fps = [int(f) for f in fingerprints]
        arr = (C.c_uint64 * max(len(fps), 1))(*fps)
        _check(lib().dp_plan_check_match(self._h, arr, len(fps)))

    # ---- device buffers (torch plumbing) ----
    def new_replicas(self, device="cuda", dtype=torch.bfloat16):
        return torch.zeros(self.P, self.stride, dtype=dtype, device=device)

    def new_state(self, device="cuda"):
        return torch.zeros(self.L, dtype=torch.float32, device=device)

    def new_workspace(self, device="cuda", stream=None):
        ws = torch.empty(self.info.workspace_bytes, dtype=torch.uint8, device=device)
        self.upload(ws, stream)
        return ws


def check_plans_match(plan, group=None):
    """Gather every process's plan fingerprint over torch.distributed and check
    them with dp_plan_check_match: raises DPError (DP_EPLAN) on every rank when
    one rank built a different bucket layout, instead of the mismatched
    collectives hanging.  Without an initialised process group only this plan
    is checked."""
    import torch.distributed as dist
    fp = plan.fingerprint
    if dist.is_available() and dist.is_initialized():
        fps = [None] * dist.get_world_size(group)
        dist.all_gather_object(fps, fp, group=group)
    else:
        fps = [fp]
    plan.check_match(fps)


def adamw_cfg(lr=2e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=0.0, step=1):
    return AdamWCfg(float(lr), float(beta1), float(beta2), float(eps), float(weight_decay),
                    float(max_norm), int(step))


def _ws(plan, ws):
    _need(ws, torch.uint8, plan.info.workspace_bytes, "workspace")
    return _ptr(ws)


def _range(plan, b0, b1):
    return int(b0), int(plan.n_buckets if b1 is None else b1)


def set_stream_launch(stream, short_ctas):
    """Launch shape of every later compute call on `stream` (dp_stream_set_launch):
    short_ctas=True for short-lived CTAs in every kernel (a low-priority stream
    beside a high-priority compute stream), False for each kernel's default shape.
    Set False again before the stream is destroyed."""
    _check(lib().dp_stream_set_launch(_stream(stream),
                                      DP_LAUNCH_SHORT_CTAS if short_ctas else DP_LAUNCH_DEFAULT))


def stream_launch(stream):
    """True when `stream` is set to short-lived CTAs."""
    out = C.c_int32()
    _check(lib().dp_stream_get_launch(_stream(stream), C.byref(out)))
    return out.value == DP_LAUNCH_SHORT_CTAS


def dp_plan_upload(plan, ws, stream=None):
    _check(lib().dp_plan_upload(plan.handle, _ws(plan, ws), _stream(stream)))


Plan.upload = lambda self, ws, stream=None: dp_plan_upload(self, ws, stream)


def dp_reduce_scatter_mean(plan, ws, grads, mean, b0=0, b1=None, want_sumsq=False, stream=None):
    _need(grads, torch.bfloat16, plan.P * plan.stride, "grads")
    _need(mean, torch.float32, plan.L, "mean")
    b0, b1 = _range(plan, b0, b1)
    _check(lib().dp_reduce_scatter_mean(plan.handle, _ws(plan, ws), _ptr(grads), _ptr(mean), b0, b1,
                                        1 if want_sumsq else 0, _stream(stream)))


def dp_clip_coef(plan, ws, max_norm, b0=0, b1=None, stream=None):
    b0, b1 = _range(plan, b0, b1)
    _check(lib().dp_clip_coef(plan.handle, _ws(plan, ws), float(max_norm), b0, b1, _stream(stream)))


def dp_sharded_adamw_step(plan, ws, grad, master, m, v, params, cfg, use_clip_coef=False, b0=0,
                          b1=None, stream=None, coef_dev=None):
    """coef_dev: a float32 CUDA tensor [1] with the caller's own clip coefficient
    (needs use_clip_coef=True); None with use_clip_coef: the workspace's."""
    for t, name in ((grad, "grad"), (master, "master"), (m, "m"), (v, "v")):
        _need(t, torch.float32, plan.L, name)
    _need(params, torch.bfloat16, plan.P * plan.stride, "params")
    b0, b1 = _range(plan, b0, b1)
    _check(lib().dp_sharded_adamw_step(plan.handle, _ws(plan, ws), _ptr(grad), _ptr(master), _ptr(m),
                                       _ptr(v), _ptr(params), _cfg_ref(cfg),
                                       1 if use_clip_coef else 0, _coef(coef_dev), b0, b1,
                                       _stream(stream)))


def dp_all_gather(plan, ws, params, b0=0, b1=None, stream=None):
    _need(params, torch.bfloat16, plan.P * plan.stride, "params")
    b0, b1 = _range(plan, b0, b1)
    _check(lib().dp_all_gather(plan.handle, _ws(plan, ws), _ptr(params), b0, b1, _stream(stream)))


def dp_broadcast(plan, ws, params, src=0, b0=0, b1=None, stream=None):
    _need(params, torch.bfloat16, plan.P * plan.stride, "params")
    b0, b1 = _range(plan, b0, b1)
    _check(lib().dp_broadcast(plan.handle, _ws(plan, ws), _ptr(params), int(src), b0, b1,
                              _stream(stream)))


def dp_allreduce_mean(plan, ws, grads, b0=0, b1=None, stream=None):
    _need(grads, torch.bfloat16, plan.P * plan.stride, "grads")
    b0, b1 = _range(plan, b0, b1)
    _check(lib().dp_allreduce_mean(plan.handle, _ws(plan, ws), _ptr(grads), b0, b1, _stream(stream)))


def dp_adamw_all_gather(plan, ws, mean, master, m, v, params, cfg, use_clip_coef=True, stream=None,
                        coef_dev=None):
    for t, name in ((mean, "mean"), (master, "master"), (m, "m"), (v, "v")):
        _need(t, torch.float32, plan.L, name)
    _need(params, torch.bfloat16, plan.P * plan.stride, "params")
    _check(lib().dp_adamw_all_gather(plan.handle, _ws(plan, ws), _ptr(mean), _ptr(master), _ptr(m),
                                     _ptr(v), _ptr(params), _cfg_ref(cfg), 1 if use_clip_coef else 0,
                                     _coef(coef_dev), _stream(stream)))


def dp_unit_all_gather(plan, ws, param_shards, unit, unit_buf, stream=None):
    """ZeRO-3: every rank's row of unit_buf [P][>= len] gets unit `unit`'s values."""
    _need(param_shards, torch.bfloat16, plan.L, "param_shards")
    if unit_buf.dim() != 2 or unit_buf.shape[0] < plan.P or not unit_buf.is_contiguous():
        raise ValueError("unit_buf must be a contiguous [P][unit_stride] tensor")
    _need(unit_buf, torch.bfloat16, plan.P * unit_buf.shape[1], "unit_buf")
    _check(lib().dp_unit_all_gather(plan.handle, _ws(plan, ws), _ptr(param_shards), int(unit),
                                    _ptr(unit_buf), int(unit_buf.shape[1]), _stream(stream)))


def dp_unit_reduce_scatter(plan, ws, unit_grads, unit, mean, want_sumsq=False, stream=None):
    """ZeRO-3: unit_grads [P][>= len] (a 2-D view, rows may be strided) -> mean shards."""
    if unit_grads.dim() != 2 or unit_grads.shape[0] < plan.P or unit_grads.stride(1) != 1:
        raise ValueError("unit_grads must be a [P][stride] view with unit element stride")
    if unit_grads.dtype != torch.bfloat16 or not unit_grads.is_cuda:
        raise TypeError("unit_grads must be a CUDA bf16 tensor")
    _need(mean, torch.float32, plan.L, "mean")
    _check(lib().dp_unit_reduce_scatter(plan.handle, _ws(plan, ws), _ptr(unit_grads),
                                        int(unit_grads.stride(0)), int(unit), _ptr(mean),
                                        1 if want_sumsq else 0, _stream(stream)))


def dp_unit_backward(plan, ws, param_shards, gather_unit, gather_buf, unit_grads, rs_unit, mean,
                     want_sumsq=False, stream=None):
    """ZeRO-3 backward in one launch: gather unit `gather_unit` into gather_buf
    [P][>= len] and reduce-scatter unit `rs_unit`'s gradients (unit_grads, a
    [P][stride] view) into mean.  Either unit may be -1 (that part left out)."""
    _need(param_shards, torch.bfloat16, plan.L, "param_shards")
    gb, gstride = None, 0
    if gather_unit >= 0:
        if gather_buf.dim() != 2 or gather_buf.shape[0] < plan.P or not gather_buf.is_contiguous():
            raise ValueError("gather_buf must be a contiguous [P][unit_stride] tensor")
        _need(gather_buf, torch.bfloat16, plan.P * gather_buf.shape[1], "gather_buf")
        gb, gstride = _ptr(gather_buf), int(gather_buf.shape[1])
    ug, ustride = None, 0
    if rs_unit >= 0:
        if unit_grads.dim() != 2 or unit_grads.shape[0] < plan.P or unit_grads.stride(1) != 1:
            raise ValueError("unit_grads must be a [P][stride] view with unit element stride")
        if unit_grads.dtype != torch.bfloat16 or not unit_grads.is_cuda:
            raise TypeError("unit_grads must be a CUDA bf16 tensor")
        _need(mean, torch.float32, plan.L, "mean")
        ug, ustride = _ptr(unit_grads), int(unit_grads.stride(0))
    _check(lib().dp_unit_backward(plan.handle, _ws(plan, ws), _ptr(param_shards), int(gather_unit),
                                  gb, gstride, ug, ustride, int(rs_unit),
                                  _ptr(mean) if mean is not None else None,
                                  1 if want_sumsq else 0, _stream(stream)))


def dp_shard_adamw_step(plan, ws, mean, master, m, v, param_shards, cfg, use_clip_coef=False,
                        stream=None, coef_dev=None):
    for t, name in ((mean, "mean"), (master, "master"), (m, "m"), (v, "v")):
        _need(t, torch.float32, plan.L, name)
    _need(param_shards, torch.bfloat16, plan.L, "param_shards")
    _check(lib().dp_shard_adamw_step(plan.handle, _ws(plan, ws), _ptr(mean), _ptr(master), _ptr(m),
                                     _ptr(v), _ptr(param_shards), _cfg_ref(cfg),
                                     1 if use_clip_coef else 0, _coef(coef_dev), _stream(stream)))


class Tracker:
    """Bucket readiness tracker (streamed per-bucket synchronisation).

    mode: DP_TRACK_ALLREDUCE (in place on `grads`), DP_TRACK_REDUCE_SCATTER
    (into `mean`, with norm partials) or DP_TRACK_ZERO_STEP (each bucket's whole
    unclipped ZeRO step; targets from set_zero_step).  dry_run=True records the
    firing order and launches nothing (no GPU needed).  short_ctas=True launches
    each bucket as short-lived CTAs (DP_TRACK_SHORT_CTAS): pair it with a
    low-priority `stream` and a higher-priority stream for the backward."""

    def __init__(self, plan, mode, ws=None, grads=None, mean=None, stream=None, max_ctas=0,
                 dry_run=False, short_ctas=False):
        self.plan = plan
        self._keep = (ws, grads, mean, stream)
        if not dry_run:
            _ws(plan, ws)
            _need(grads, torch.bfloat16, plan.P * plan.stride, "grads")
            if mode == DP_TRACK_REDUCE_SCATTER:
                _need(mean, torch.float32, plan.L, "mean")
            s = _stream(stream)
        else:
            s = None
        h = C.c_void_p()
        _check(lib().dp_tracker_create(plan.handle, int(mode), _ptr(ws), _ptr(grads), _ptr(mean), s,
                                       int(max_ctas),
                                       (DP_TRACK_DRY_RUN if dry_run else 0) |
                                       (DP_TRACK_SHORT_CTAS if short_ctas else 0),
                                       C.byref(h)))
        self._h = h
        self._dry = dry_run

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.dp_tracker_free(h)
            self._h = None

    def begin(self):
        _check(lib().dp_tracker_begin(self._h))

    def set_micro(self, micro):
        """Last micro-batch of accumulation: fire the fused bf16(grads + micro)
        reduction per bucket (None: the plain reduction)."""
        if micro is not None and not getattr(self, "_dry", False):
            _need(micro, torch.bfloat16, self.plan.P * self.plan.stride, "micro")
        self._micro = micro
        _check(lib().dp_tracker_set_micro(self._h, _ptr(micro) if micro is not None else None))

    def set_zero_step(self, params, master, m, v, cfg):
        """DP_TRACK_ZERO_STEP: the replicas and fp32 state each bucket's step
        updates, and this step's AdamW settings (cfg.max_norm must be <= 0)."""
        if not getattr(self, "_dry", False):
            _need(params, torch.bfloat16, self.plan.P * self.plan.stride, "params")
            for t, name in ((master, "master"), (m, "m"), (v, "v")):
                _need(t, torch.float32, self.plan.L, name)
        self._zero = (params, master, m, v)
        _check(lib().dp_tracker_set_zero_step(self._h, _ptr(params), _ptr(master), _ptr(m), _ptr(v),
                                              _cfg_ref(cfg)))

    def mark_ready(self, tensor, event=None):
        """event: torch.cuda.Event recorded after the tensor's gradient was written."""
        ev = C.c_void_p(event.cuda_event) if event is not None else None
        _check(lib().dp_tracker_mark_ready(self._h, int(tensor), ev))

    def mark_ready_range(self, t0, t1, event=None):
        """Tensors [t0, t1) ready, all written before `event` (one call, one event)."""
        ev = C.c_void_p(event.cuda_event) if event is not None else None
        _check(lib().dp_tracker_mark_ready_range(self._h, int(t0), int(t1), ev))

    def mark_ready_batch(self, tensors, events=None):
        """Tensors ready, each written before its own event (events: a list of
        torch.cuda.Event, or None), in one call."""
        ts = [int(t) for t in tensors]
        arr = (C.c_int32 * max(len(ts), 1))(*ts)
        evs = None
        if events is not None:
            if len(events) != len(ts):
                raise ValueError("one event per tensor")
            evs = (C.c_void_p * max(len(ts), 1))(*[e.cuda_event for e in events])
        _check(lib().dp_tracker_mark_ready_batch(self._h, arr, evs, len(ts)))

    def set_side_stream(self, stream, max_ctas=0):
        """Every bucket but the last fires on `stream` (a torch stream, an SmStream,
        or None to undo), grids capped at max_ctas."""
        self._side = stream
        _check(lib().dp_tracker_set_side_stream(self._h, None if stream is None else _stream(stream),
                                                int(max_ctas)))

    def stats(self):
        """(launches, cudaStreamWaitEvent calls) of this step so far."""
        n, w = C.c_int32(), C.c_int32()
        _check(lib().dp_tracker_stats(self._h, C.byref(n), C.byref(w)))
        return n.value, w.value

    def wait(self, timeout_ms=10000):
        _check(lib().dp_tracker_wait(self._h, int(timeout_ms)))

    def fired(self):
        n = C.c_int32()
        cap = self.plan.n_buckets
        arr = (C.c_int32 * max(cap, 1))()
        _check(lib().dp_tracker_fired(self._h, arr, cap, C.byref(n)))
        return list(arr[:n.value])


class SmStreams:
    """CUDA streams confined to SM partitions (dp_sm_streams_create): .part runs on
    n_sms SMs, .rest (with_rest=True) on all the others.  Each is a
    torch.cuda.ExternalStream; close() (or garbage collection) destroys them."""

    def __init__(self, n_sms, priority=0, with_rest=False):
        s, r, h = C.c_void_p(), C.c_void_p(), C.c_void_p()
        n_part, n_rest = C.c_int32(), C.c_int32()
        _check(lib().dp_sm_streams_create(int(n_sms), int(priority), C.byref(s),
                                          C.byref(r) if with_rest else None, C.byref(h),
                                          C.byref(n_part), C.byref(n_rest)))
        self._h = h
        self.n_part, self.n_rest = n_part.value, n_rest.value
        self.part = torch.cuda.ExternalStream(s.value)
        self.rest = torch.cuda.ExternalStream(r.value) if with_rest else None

    def close(self):
        if getattr(self, "_h", None) is not None and _lib is not None:
            _lib.dp_sm_streams_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()


def dp_accumulate(plan, ws, acc, micro, b0=0, b1=None, stream=None):
    """acc[r] = bf16(acc[r] + micro[r]) (local gradient accumulation, no sync)."""
    _need(acc, torch.bfloat16, plan.P * plan.stride, "acc")
    _need(micro, torch.bfloat16, plan.P * plan.stride, "micro")
    b0, b1 = _range(plan, b0, b1)
    _check(lib().dp_accumulate(plan.handle, _ws(plan, ws), _ptr(acc), _ptr(micro), b0, b1,
                               _stream(stream)))


def dp_allreduce_mean_accum(plan, ws, acc, micro, b0=0, b1=None, stream=None):
    """Last micro-batch: accumulate and mean all-reduce in one pass (result in acc)."""
    _need(acc, torch.bfloat16, plan.P * plan.stride, "acc")
    _need(micro, torch.bfloat16, plan.P * plan.stride, "micro")
    b0, b1 = _range(plan, b0, b1)
    _check(lib().dp_allreduce_mean_accum(plan.handle, _ws(plan, ws), _ptr(acc), _ptr(micro), b0,
                                         b1, _stream(stream)))


def dp_reduce_scatter_mean_accum(plan, ws, acc, micro, mean, b0=0, b1=None, want_sumsq=False,
                                 stream=None):
    """Last micro-batch (ZeRO): reduce-scatter every rank's bf16(acc + micro) into mean."""
    _need(acc, torch.bfloat16, plan.P * plan.stride, "acc")
    _need(micro, torch.bfloat16, plan.P * plan.stride, "micro")
    _need(mean, torch.float32, plan.L, "mean")
    b0, b1 = _range(plan, b0, b1)
    _check(lib().dp_reduce_scatter_mean_accum(plan.handle, _ws(plan, ws), _ptr(acc), _ptr(micro),
                                              _ptr(mean), b0, b1, 1 if want_sumsq else 0,
                                              _stream(stream)))


def dp_allreduce_mean_bf16wire(plan, ws, grads, b0=0, b1=None, stream=None):
    _need(grads, torch.bfloat16, plan.P * plan.stride, "grads")
    b0, b1 = _range(plan, b0, b1)
    _check(lib().dp_allreduce_mean_bf16wire(plan.handle, _ws(plan, ws), _ptr(grads), b0, b1,
                                            _stream(stream)))


def _state_arrays(plan, arrays, fn):
    """The optimizer-state arrays for a checkpoint call: fp32, contiguous, >= L
    elements, all on the host or all on the GPU.  Returns (pointers, host?)."""
    host = None
    for name, t in zip(("master", "m", "v"), arrays):
        if t is None:
            continue
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_contiguous():
            raise TypeError(f"{fn}: {name} must be a contiguous float32 tensor")
        if t.numel() < plan.L:
            raise ValueError(f"{fn}: {name} holds {t.numel()} elements, needs {plan.L}")
        h = t.device.type == "cpu"
        if host is not None and h != host:
            raise ValueError(f"{fn}: arrays must all be on the host or all on the GPU")
        host = h
    return [_ptr(t) for t in arrays], host is None or host   # no array: refused, no CUDA call


def dp_checkpoint_save(plan, path, master=None, m=None, v=None, step=0, stream=None):
    """Write master/m/v (flat layout of `plan`, tensor order in the file) and t."""
    ptrs, host = _state_arrays(plan, (master, m, v), "dp_checkpoint_save")
    _check(lib().dp_checkpoint_save(plan.handle, os.fsencode(path), *ptrs, int(step),
                                    DP_CKPT_HOST if host else 0,
                                    None if host else _stream(stream)))


def dp_checkpoint_load(plan, path, master=None, m=None, v=None, stream=None):
    """Read a checkpoint into master/m/v (any plan over the same tensor sizes);
    returns the saved step t."""
    ptrs, host = _state_arrays(plan, (master, m, v), "dp_checkpoint_load")
    step = C.c_int64(0)
    _check(lib().dp_checkpoint_load(plan.handle, os.fsencode(path), *ptrs, C.byref(step),
                                    DP_CKPT_HOST if host else 0,
                                    None if host else _stream(stream)))
    return step.value


def dp_selftest_bounded_wait(limit_ns=1_000_000, stream=None):
    """Run the bounded-wait failure path once; returns (status, ms waited)."""
    st = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    _check(lib().dp_selftest_bounded_wait(_ptr(st), int(limit_ns), _stream(stream)))
    s, ms = st.tolist()
    return s, ms


def dp_bounds_violations(reset=False):
    """Failed device index checks since the last reset (-1: library built without checks)."""
    n = lib().dp_bounds_violations(1 if reset else 0)
    if n == -2:
        raise DPError(DP_ECUDA, "dp_bounds_violations: cannot read the device counters")
    return n


def dp_set_adamw_cfg(plan, ws, cfg, stream=None):
    """Store this step's AdamW scalars in the workspace; updates called with cfg=None
    (e.g. inside a captured CUDA graph) use them.  Call outside the graph, before
    each replay."""
    _check(lib().dp_set_adamw_cfg(plan.handle, _ws(plan, ws), C.byref(cfg), _stream(stream)))


def dp_fused_zero_step_launches(cfg):
    return lib().dp_fused_zero_step_launches(C.byref(cfg))


def dp_fused_zero_step(plan, ws, grads, params, master, m, v, cfg, events=None, stream=None):
    """One fused ZeRO-1/2 step over all buckets.  `events`: optional list of
    dp_fused_zero_step_launches(cfg)+1 torch.cuda.Event objects recorded around
    each launch."""
    _need(grads, torch.bfloat16, plan.P * plan.stride, "grads")
    _need(params, torch.bfloat16, plan.P * plan.stride, "params")
    for t, name in ((master, "master"), (m, "m"), (v, "v")):
        _need(t, torch.float32, plan.L, name)
    ev = None
    if events is not None:
        n = dp_fused_zero_step_launches(cfg) + 1
        if len(events) != n:
            raise ValueError(f"need {n} events, got {len(events)}")
        for e in events:
            if e.cuda_event == 0:
                raise ValueError("events must have been recorded once (so they exist)")
        ev = (C.c_void_p * n)(*[e.cuda_event for e in events])
    _check(lib().dp_fused_zero_step(plan.handle, _ws(plan, ws), _ptr(grads), _ptr(params),
                                    _ptr(master), _ptr(m), _ptr(v), C.byref(cfg), ev,
                                    _stream(stream)))


def dp_read_norm(plan, ws, stream=None, raise_on_status=True):
    """Synchronises the stream; returns (norm, coef, status)."""
    norm, coef, status = C.c_double(), C.c_float(), C.c_int32()
    rc = lib().dp_read_norm(plan.handle, _ptr(ws), C.byref(norm), C.byref(coef), C.byref(status),
                            _stream(stream))
    if raise_on_status:
        _check(rc)
    return norm.value, coef.value, status.value


def dp_clip_coef_noalloc(plan, grads, mean, max_norm, coef_out, norm_out, stream=None):
    """Reduce-scatter mean + clip coefficient without a workspace (library-owned
    static device scratch; see include/dpsync.h).  coef_out: 1-element float32
    CUDA tensor, norm_out: 1-element float64 CUDA tensor."""
    _need(grads, torch.bfloat16, plan.P * plan.stride, "grads")
    _need(mean, torch.float32, plan.L, "mean")
    _need(coef_out, torch.float32, 1, "coef_out")
    _need(norm_out, torch.float64, 1, "norm_out")
    _check(lib().dp_clip_coef_noalloc(plan.handle, _ptr(grads), _ptr(mean), float(max_norm),
                                      _ptr(coef_out), _ptr(norm_out), _stream(stream)))


def dp_version():
    return lib().dp_version()

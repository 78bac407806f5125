"""CPU oracle for the data-parallel gradient synchronisation step.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
bench's CPU-baseline leg, never by the product path.  It loads
``liboracle.so`` (built from ``oracle.cpp`` by :func:`build`), a plain C++17
program that shares no code with the CUDA library.  This module only marshals
numpy arrays in and out; every step of the computation is in ``oracle.cpp``.

``Oracle(path)`` binds one compiled copy; the module-level functions use the
default build.  The mutation tests bind deliberately broken copies to show that
the pins catch plausible mistakes.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.cpp")
LIB = os.path.join(HERE, "liboracle.so")
MAX_RANKS = 64


def build_cmd(src: str = SRC, out: str = LIB):
    return ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
            "-o", out, src]


def build(force: bool = False, src: str = SRC, out: str = LIB):
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        subprocess.run(build_cmd(src, out), check=True)


class AdamWCfg(C.Structure):
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double), ("beta2", C.c_double),
                ("eps", C.c_double), ("weight_decay", C.c_double), ("max_norm", C.c_double),
                ("step", C.c_int64)]


class Stats(C.Structure):
    _fields_ = [("sumsq", C.c_double), ("norm", C.c_double), ("coef", C.c_float),
                ("n_buckets", C.c_int32), ("padded_len", C.c_int64), ("rs_steps", C.c_int64),
                ("ag_steps", C.c_int64), ("replicas_equal", C.c_int32), ("pad_", C.c_int32),
                ("rs_sent", C.c_int64 * MAX_RANKS), ("ag_sent", C.c_int64 * MAX_RANKS)]


class MeshStats(C.Structure):
    _fields_ = [("rs_sent", C.c_int64 * MAX_RANKS), ("ag_sent", C.c_int64 * MAX_RANKS),
                ("cross_sent", C.c_int64 * MAX_RANKS), ("groups_equal", C.c_int32),
                ("replicas_equal", C.c_int32), ("sumsq", C.c_double), ("norm", C.c_double),
                ("coef", C.c_float), ("pad_", C.c_int32)]


class Zero3Stats(C.Structure):
    _fields_ = [("ag_fwd_sent", C.c_int64 * MAX_RANKS), ("ag_bwd_sent", C.c_int64 * MAX_RANKS),
                ("rs_sent", C.c_int64 * MAX_RANKS), ("gathered_ok", C.c_int32), ("pad_", C.c_int32),
                ("norm", C.c_double), ("coef", C.c_float), ("pad2_", C.c_int32)]


def adamw_cfg(adamw, step):
    return AdamWCfg(adamw.lr, adamw.beta1, adamw.beta2, adamw.eps, adamw.weight_decay,
                    adamw.max_norm, int(step))


def _p(a):
    return a.ctypes.data_as(C.c_void_p) if a is not None else None


def _i64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


class Oracle:
    """One compiled copy of the oracle."""

    def __init__(self, path: str = LIB):
        L = C.CDLL(path)
        P = C.c_void_p
        L.orc_plan.argtypes = [P, C.c_int32, C.c_int64, C.c_int32, P, P, P, P, P, P]
        L.orc_ring_reduce_scatter_f32.argtypes = [C.c_int32, C.c_int64, P, P, P]
        L.orc_ring_all_gather_u16.argtypes = [C.c_int32, C.c_int64, P, P, P]
        L.orc_bf16_rne.argtypes = [C.c_float]
        L.orc_bf16_rne.restype = C.c_uint16
        L.orc_adamw_element.argtypes = [C.c_float, P, C.c_int32, P]
        L.orc_adamw_element.restype = None
        L.orc_clip_coef.argtypes = [P, C.c_int32, C.c_double, P]
        L.orc_clip_coef.restype = C.c_float
        L.orc_allreduce_mean.argtypes = [P, C.c_int32, C.c_int64, C.c_int32, P, P, P, C.c_int32]
        L.orc_bucket_sumsq.argtypes = [P, C.c_int32, C.c_int64, C.c_int32, P, P, C.c_int32]
        L.orc_zero_step.argtypes = [P, P, C.c_int32, C.c_int64, C.c_int32, P, P, P, P, P, P, P,
                                    C.c_double, P, C.c_int32]
        L.orc_ledger_bytes.argtypes = [C.c_int32, C.c_double, C.c_int32, P]
        L.orc_ledger_bytes.restype = C.c_double
        L.orc_mesh_allreduce_mean.argtypes = [P, C.c_int32, C.c_int64, C.c_int32, C.c_int32, P,
                                              P, P]
        L.orc_mesh_zero_step.argtypes = [P, P, C.c_int32, C.c_int64, C.c_int32, C.c_int32, P, P,
                                         P, P, P, P, P]
        L.orc_zero3_step.argtypes = [P, P, C.c_int32, C.c_int64, C.c_int32, P, P, P, P, P, P, P]
        L.orc_accumulate.argtypes = [C.c_int32, C.c_int64, P, P]
        L.orc_accumulate.restype = None
        L.orc_allreduce_mean_bf16wire.argtypes = [P, C.c_int32, C.c_int64, C.c_int32, P, P]
        L.orc_sum.argtypes = [P, C.c_int64]
        L.orc_sum.restype = C.c_double
        L.orc_stage_traffic.argtypes = [C.c_int32, C.c_int32, C.c_int64, P, P]
        L.orc_lsq_identity.argtypes = [C.c_int32, C.c_int32, C.c_int32, P, P, P, P, P, P, P, P]
        self.L = L
        self.path = path

    def plan(self, sizes, bucket_bytes, P):
        """The oracle's own bucket plan: dict of t_off, t_bucket, b_off, b_len, L."""
        s = _i64(sizes)
        n = len(s)
        t_off = np.zeros(max(n, 1), np.int64)
        t_b = np.zeros(max(n, 1), np.int32)
        b_off = np.zeros(max(n, 1), np.int64)
        b_len = np.zeros(max(n, 1), np.int64)
        nb = C.c_int32()
        L = C.c_int64()
        _check(self.L.orc_plan(_p(s), n, int(bucket_bytes), int(P), _p(t_off), _p(t_b),
                               _p(b_off), _p(b_len), C.byref(nb), C.byref(L)), "plan")
        return dict(t_off=t_off[:n].copy(), t_bucket=t_b[:n].copy(),
                    b_off=b_off[:nb.value].copy(), b_len=b_len[:nb.value].copy(), L=L.value,
                    n_buckets=nb.value)

    def ring_reduce_scatter(self, X):
        """Literal ring on X [P][len] fp32. Returns (X after, sent[P], steps)."""
        X = np.array(X, dtype=np.float32, copy=True, order="C")
        P, n = X.shape
        sent = np.zeros(P, np.int64)
        steps = C.c_int64(0)
        _check(self.L.orc_ring_reduce_scatter_f32(P, n, _p(X), _p(sent), C.byref(steps)),
               "ring RS")
        return X, sent, steps.value

    def ring_all_gather(self, Y):
        Y = np.array(Y, dtype=np.uint16, copy=True, order="C")
        P, n = Y.shape
        sent = np.zeros(P, np.int64)
        steps = C.c_int64(0)
        _check(self.L.orc_ring_all_gather_u16(P, n, _p(Y), _p(sent), C.byref(steps)), "ring AG")
        return Y, sent, steps.value

    def bf16_rne(self, x: float) -> int:
        return int(self.L.orc_bf16_rne(float(x)))

    def adamw_element(self, g, theta, m, v, decay, cfg):
        st = np.array([theta, m, v], np.float32)
        self.L.orc_adamw_element(float(np.float32(g)), _p(st), int(decay), C.byref(cfg))
        return st

    def clip_coef(self, bucket_sumsq, max_norm):
        a = np.ascontiguousarray(bucket_sumsq, np.float64)
        norm = C.c_double()
        coef = self.L.orc_clip_coef(_p(a), len(a), float(max_norm), C.byref(norm))
        return coef, norm.value

    def allreduce_mean(self, sizes, bucket_bytes, P, grads_u16, want_mean=True, n_threads=0):
        """grads_u16 [P][n_params] bf16 bits (tensor order). Returns (out, mean, stats)."""
        s = _i64(sizes)
        g = np.array(grads_u16, dtype=np.uint16, copy=True, order="C")
        mean = np.zeros(g.shape[1], np.float32) if want_mean else None
        st = Stats()
        _check(self.L.orc_allreduce_mean(_p(s), len(s), int(bucket_bytes), int(P), _p(g),
                                         _p(mean), C.byref(st), int(n_threads)), "allreduce")
        return g, mean, st

    def bucket_sumsq(self, sizes, bucket_bytes, P, grads_u16, n_threads=0):
        s = _i64(sizes)
        g = np.ascontiguousarray(grads_u16, dtype=np.uint16)
        nb = self.plan(sizes, bucket_bytes, P)["n_buckets"]
        out = np.zeros(nb, np.float64)
        _check(self.L.orc_bucket_sumsq(_p(s), len(s), int(bucket_bytes), int(P), _p(g), _p(out),
                                       int(n_threads)), "bucket sumsq")
        return out

    def zero_step(self, sizes, decay, bucket_bytes, P, grads_u16, master, m, v, cfg,
                  sumsq_total=-1.0, want_mean=True, n_threads=0):
        """One fused ZeRO-1/2 step on copies of master/m/v.
        Returns (params [P][n] u16, master, m, v, mean, stats)."""
        s = _i64(sizes)
        d = np.ascontiguousarray(decay, dtype=np.uint8)
        g = np.ascontiguousarray(grads_u16, dtype=np.uint16)
        master = np.array(master, dtype=np.float32, copy=True)
        m = np.array(m, dtype=np.float32, copy=True)
        v = np.array(v, dtype=np.float32, copy=True)
        params = np.zeros_like(g)
        mean = np.zeros(g.shape[1], np.float32) if want_mean else None
        st = Stats()
        _check(self.L.orc_zero_step(_p(s), _p(d), len(s), int(bucket_bytes), int(P), _p(g),
                                    _p(master), _p(m), _p(v), _p(params), C.byref(cfg), _p(mean),
                                    float(sumsq_total), C.byref(st), int(n_threads)), "zero step")
        return params, master, m, v, mean, st

    def sum(self, x):
        """The oracle's compensated sum of doubles (e.g. per-bucket sums of squares)."""
        a = np.ascontiguousarray(x, np.float64)
        return self.L.orc_sum(_p(a), len(a))

    def mesh_allreduce_mean(self, sizes, bucket_bytes, R, S, grads_u16):
        """Mean all-reduce on an R x S mesh (rank = g*S + s). Returns (out, mean, stats)."""
        s = _i64(sizes)
        g = np.array(grads_u16, dtype=np.uint16, copy=True, order="C")
        mean = np.zeros(g.shape[1], np.float32)
        st = MeshStats()
        _check(self.L.orc_mesh_allreduce_mean(_p(s), len(s), int(bucket_bytes), int(R), int(S),
                                              _p(g), _p(mean), C.byref(st)), "mesh allreduce")
        return g, mean, st

    def mesh_zero_step(self, sizes, decay, bucket_bytes, R, S, grads_u16, master, m, v, cfg):
        """ZeRO-2 step on an R x S mesh. Returns (params, master, m, v, stats)."""
        s = _i64(sizes)
        d = np.ascontiguousarray(decay, dtype=np.uint8)
        g = np.ascontiguousarray(grads_u16, dtype=np.uint16)
        master = np.array(master, dtype=np.float32, copy=True)
        m = np.array(m, dtype=np.float32, copy=True)
        v = np.array(v, dtype=np.float32, copy=True)
        params = np.zeros_like(g)
        st = MeshStats()
        _check(self.L.orc_mesh_zero_step(_p(s), _p(d), len(s), int(bucket_bytes), int(R), int(S),
                                         _p(g), _p(master), _p(m), _p(v), _p(params), C.byref(cfg),
                                         C.byref(st)), "mesh zero step")
        return params, master, m, v, st

    def zero3_step(self, sizes, decay, bucket_bytes, P, grads_u16, param_shards, master, m, v,
                   cfg):
        """ZeRO-3 unit flow. Returns (param_shards, master, m, v, stats)."""
        s = _i64(sizes)
        d = np.ascontiguousarray(decay, dtype=np.uint8)
        g = np.ascontiguousarray(grads_u16, dtype=np.uint16)
        ps = np.array(param_shards, dtype=np.uint16, copy=True)
        master = np.array(master, dtype=np.float32, copy=True)
        m = np.array(m, dtype=np.float32, copy=True)
        v = np.array(v, dtype=np.float32, copy=True)
        st = Zero3Stats()
        _check(self.L.orc_zero3_step(_p(s), _p(d), len(s), int(bucket_bytes), int(P), _p(g), _p(ps),
                                     _p(master), _p(m), _p(v), C.byref(cfg), C.byref(st)),
               "zero3 step")
        return ps, master, m, v, st

    def accumulate(self, acc_u16, micro_u16):
        """acc = bf16(acc + micro), element by element ([P][n] bf16 bits)."""
        acc = np.array(acc_u16, dtype=np.uint16, copy=True, order="C")
        micro = np.ascontiguousarray(micro_u16, dtype=np.uint16)
        P, n = acc.shape
        self.L.orc_accumulate(P, n, _p(acc), _p(micro))
        return acc

    def allreduce_mean_bf16wire(self, sizes, bucket_bytes, P, grads_u16):
        """The ring with bf16 partial sums. Returns (out, fp32 quotient)."""
        s = _i64(sizes)
        g = np.array(grads_u16, dtype=np.uint16, copy=True, order="C")
        q = np.zeros(g.shape[1], np.float32)
        _check(self.L.orc_allreduce_mean_bf16wire(_p(s), len(s), int(bucket_bytes), int(P), _p(g),
                                                  _p(q)), "bf16 wire allreduce")
        return g, q

    def ledger_bytes(self, stage, psi, P, comp=(2, 2, 4, 4, 4)):
        c = np.asarray(comp, np.float64)
        return self.L.orc_ledger_bytes(int(stage), float(psi), int(P), _p(c))

    def stage_traffic(self, stage, P, M):
        sent = np.zeros(P, np.int64)
        steps = C.c_int64()
        _check(self.L.orc_stage_traffic(int(stage), int(P), int(M), _p(sent), C.byref(steps)),
               "stage traffic")
        return sent, steps.value

    def lsq_identity(self, x, y, theta, split):
        x = np.ascontiguousarray(x, np.float64)
        y = np.ascontiguousarray(y, np.float64)
        th = np.ascontiguousarray(theta, np.float64)
        sp = np.ascontiguousarray(split, np.int32)
        B, F = x.shape
        N = len(sp)
        g_full, g_k = np.zeros(F), np.zeros((N, F))
        g_bar, g_sum = np.zeros(F), np.zeros(F)
        _check(self.L.orc_lsq_identity(B, F, N, _p(x), _p(y), _p(th), _p(sp), _p(g_full),
                                       _p(g_k), _p(g_bar), _p(g_sum)), "least squares")
        return g_full, g_k, g_bar, g_sum


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        build()
        _default = Oracle(LIB)
    return _default

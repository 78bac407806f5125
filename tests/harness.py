"""Test harness: one workload laid out for the library and for the oracle.

Inputs come from workloads.gen (the shared seeded generator); the layout
offsets come from the plan under test only to place those inputs on the device
and to read results back.  Nothing here computes any part of the method.
"""
from __future__ import annotations

import numpy as np
import torch

import gradient_sync_zero_gb300 as dps
from workloads import configs, device as wdev, gen


def u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bits (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def small_workload(sizes, P, bucket_bytes, sigma=1e-3, seed=0, decay=None, outlier_frac=0.0,
                   name="case"):
    wl = configs.Workload(name=name, P=P, names=[f"t{i}" for i in range(len(sizes))],
                          shapes=[(s,) for s in sizes], bucket_bytes=bucket_bytes, sigma=sigma,
                          outlier_frac=outlier_frac, seed=seed)
    if decay is not None:
        wl.decay_override = list(decay)
    return wl


def decay_of(wl):
    return list(getattr(wl, "decay_override", wl.decay))


class Case:
    """A workload, its plan and its device buffers."""

    def __init__(self, wl, stride=0, device="cuda"):
        self.wl = wl
        self.P = wl.P
        self.sizes = wl.sizes
        self.decay = decay_of(wl)
        self.plan = dps.Plan(self.sizes, wl.bucket_bytes, wl.P, self.decay, stride)
        self.off = self.plan.tensor_offsets()
        self.device = device
        self.ws = self.plan.new_workspace(device) if device == "cuda" else None

    # ---- host-side inputs (tensor order) ----
    def host_grads(self, step) -> np.ndarray:
        n = self.wl.n_params
        out = np.zeros((self.P, n), np.uint16)
        for r in range(self.P):
            out[r] = u16(gen.grad_values(self.wl, step, r, 0, n))
        return out

    def host_master(self) -> np.ndarray:
        return gen.master_values(self.wl, 0, self.wl.n_params).numpy()

    # ---- tensor order <-> device layout ----
    def to_replicas(self, g_u16: np.ndarray) -> torch.Tensor:
        buf = self.plan.new_replicas(self.device)
        src = torch.from_numpy(g_u16.view(np.int16)).view(torch.bfloat16).to(self.device)
        for r in range(self.P):
            wdev.fill_flat(buf[r], self.off, self.sizes, src[r])
        return buf

    def to_flat(self, x_f32: np.ndarray) -> torch.Tensor:
        buf = self.plan.new_state(self.device)
        wdev.fill_flat(buf, self.off, self.sizes, torch.from_numpy(x_f32).to(self.device))
        return buf

    def from_replicas(self, buf: torch.Tensor) -> np.ndarray:
        return u16(wdev.gather_flat(buf[:, :self.plan.L], self.off, self.sizes))

    def from_flat(self, buf: torch.Tensor) -> np.ndarray:
        return wdev.gather_flat(buf, self.off, self.sizes).cpu().numpy()

    def padding_mask(self) -> torch.Tensor:
        """True at flat slots no tensor occupies (inside [0, L))."""
        m = torch.ones(self.plan.L, dtype=torch.bool)
        for t, s in enumerate(self.sizes):
            m[self.off[t]:self.off[t] + s] = False
        return m


def assert_replicas_equal(buf: torch.Tensor, L: int):
    for r in range(1, buf.shape[0]):
        assert torch.equal(buf[0, :L], buf[r, :L]), f"replica {r} differs from replica 0"


def rel_err(a, b, tau=1e-30):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.abs(a - b) / np.maximum(np.abs(b), tau)


def bf16_ulp_diff(a_u16: np.ndarray, b_u16: np.ndarray) -> np.ndarray:
    """Distance in bf16 units in the last place (sign-magnitude ordering)."""
    def key(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u & 0x7FFF)
    return np.abs(key(a_u16) - key(b_u16))

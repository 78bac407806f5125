"""Seeded, counter-based synthetic inputs (gradients, fp32 master weights).

Every value is a pure function of (seed, stream, step, rank, element index), so a
slice can be produced anywhere without producing the rest.  The hash is
SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014): add the golden-ratio increment, then the
xor-shift-multiply finaliser.  Two 53-bit uniforms feed the Box-Muller
transform in float64; a third hash picks outliers.  The float64 sample is scaled
by sigma and rounded to bf16 (torch's round-to-nearest-even cast), or to fp32
for master weights.

The same bytes go to both the CUDA path and the oracle: large cases are
generated on the GPU with torch ops and copied back slice by slice, small ones
on the host and uploaded.  Nothing here implements the synchronisation method.
"""
from __future__ import annotations

import math

import torch

_MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB

STREAM_GRAD = 1
STREAM_MASTER = 2
STREAM_OUTLIER = 3
STREAM_DATA = 4


def _s64(u: int) -> int:
    """uint64 -> the int64 with the same bits."""
    u &= _MASK64
    return u - (1 << 64) if u >= (1 << 63) else u


def splitmix64_int(x: int) -> int:
    """Reference SplitMix64 on Python ints (used to pin the tensor version)."""
    z = (x + GOLDEN) & _MASK64
    z = ((z ^ (z >> 30)) * MIX1) & _MASK64
    z = ((z ^ (z >> 27)) * MIX2) & _MASK64
    return z ^ (z >> 31)


def _lsr(x: torch.Tensor, k: int) -> torch.Tensor:
    return (x >> k) & ((1 << (64 - k)) - 1)


def splitmix64(x: torch.Tensor) -> torch.Tensor:
    """SplitMix64 on an int64 tensor holding uint64 bit patterns (wrapping arithmetic)."""
    z = x + _s64(GOLDEN)
    z = (z ^ _lsr(z, 30)) * _s64(MIX1)
    z = (z ^ _lsr(z, 27)) * _s64(MIX2)
    return z ^ _lsr(z, 31)


def stream_key(seed: int, stream: int, step: int, rank: int) -> int:
    k = splitmix64_int(seed)
    for part in (stream, step, rank):
        k = splitmix64_int(k ^ (part & _MASK64))
    return k


def _uniform53(h: torch.Tensor) -> torch.Tensor:
    return _lsr(h, 11).to(torch.float64) * (1.0 / (1 << 53))


def normal_f64(key: int, start: int, count: int, device) -> torch.Tensor:
    """Standard normal samples for counters [start, start+count) of one stream key."""
    idx = torch.arange(start, start + count, dtype=torch.int64, device=device)
    base = _s64(key)
    h1 = splitmix64((idx * 2) ^ base)
    h2 = splitmix64((idx * 2 + 1) ^ base)
    u1 = _uniform53(h1) + (1.0 / (1 << 53))      # (0, 1]
    u2 = _uniform53(h2)                           # [0, 1)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def outlier_mask(key: int, start: int, count: int, frac: float, device) -> torch.Tensor:
    idx = torch.arange(start, start + count, dtype=torch.int64, device=device)
    h = splitmix64(idx ^ _s64(key ^ 0x5851F42D4C957F2D))
    return _uniform53(h) < frac


CHUNK = 1 << 26


def grad_values(wl, step: int, rank: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """bf16 gradient entries [start, start+count) of rank `rank` at `step`, in the
    unpadded tensor-order index space of workload `wl`."""
    out = torch.empty(count, dtype=torch.bfloat16, device=device)
    key = stream_key(wl.seed, STREAM_GRAD, step, rank)
    okey = stream_key(wl.seed, STREAM_OUTLIER, step, rank)
    for o in range(0, count, CHUNK):
        n = min(CHUNK, count - o)
        z = normal_f64(key, start + o, n, device) * wl.sigma
        if wl.outlier_frac > 0:
            m = outlier_mask(okey, start + o, n, wl.outlier_frac, device)
            z = torch.where(m, z * wl.outlier_scale, z)
        out[o:o + n] = z.to(torch.bfloat16)
    return out


def master_values(wl, start: int, count: int, device="cpu") -> torch.Tensor:
    """fp32 master-weight entries [start, start+count), N(0, master_sigma)."""
    out = torch.empty(count, dtype=torch.float32, device=device)
    key = stream_key(wl.seed, STREAM_MASTER, 0, 0)
    for o in range(0, count, CHUNK):
        n = min(CHUNK, count - o)
        out[o:o + n] = (normal_f64(key, start + o, n, device) * wl.master_sigma).to(torch.float32)
    return out


def small_ints(seed: int, stream: int, count: int, lo: int, hi: int) -> list:
    """Deterministic small integers in [lo, hi] (least-squares identity data)."""
    key = stream_key(seed, STREAM_DATA, stream, 0)
    span = hi - lo + 1
    return [lo + (splitmix64_int(key ^ i) % span) for i in range(count)]

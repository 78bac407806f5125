"""Place generated inputs into a replica layout (device or host tensors).

The layout (where tensor t starts in the flat padded index space) is passed in
as a list of offsets; nothing here depends on the library under test.
"""
from __future__ import annotations

import torch

from . import gen


def tensor_bases(sizes):
    base, acc = [], 0
    for s in sizes:
        base.append(acc)
        acc += s
    return base


def fill_grads(buf: torch.Tensor, offsets, wl, step: int, ranks=None):
    """buf [P][stride] bf16: replica r's tensor t at offsets[t] gets the
    generator's values for (step, r); padding is left as it is (zeros)."""
    sizes = wl.sizes
    base = tensor_bases(sizes)
    for r in (range(wl.P) if ranks is None else ranks):
        vals = gen.grad_values(wl, step, r, 0, wl.n_params, device=buf.device)
        row = buf[r]
        for t, s in enumerate(sizes):
            if s:
                row[offsets[t]:offsets[t] + s].copy_(vals[base[t]:base[t] + s])
        del vals


def fill_flat(buf: torch.Tensor, offsets, sizes, values: torch.Tensor):
    """Scatter a tensor-order vector into the flat padded layout (1-D buf)."""
    base = tensor_bases(sizes)
    for t, s in enumerate(sizes):
        if s:
            buf[offsets[t]:offsets[t] + s].copy_(values[base[t]:base[t] + s])


def gather_flat(buf: torch.Tensor, offsets, sizes) -> torch.Tensor:
    """Inverse of fill_flat along the last dimension: tensor-order values."""
    parts = [buf[..., offsets[t]:offsets[t] + s] for t, s in enumerate(sizes) if s]
    if not parts:
        return buf[..., :0].clone()
    return torch.cat(parts, dim=-1)

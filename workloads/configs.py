"""Synthetic workload definitions: tensor lists, rank counts, bucket caps, AdamW settings.

This module holds shapes and hyperparameters only; it computes nothing of the
synchronisation method itself.  Both the CUDA path's tests/bench and the CPU
oracle's tests draw their inputs from here (together with ``workloads.gen``).

Readings taken where the workload text is loose:
  * "MB" for bucket caps is MiB (2**20 bytes), following PyTorch's
    ``bucket_cap_mb`` knob that the DDP pages name.
  * The tiny plumbing case lists seven sizes that add up to 1,001,003 (the text
    says 1,000,003); the list is followed.
  * The Llama-style 1.1B case orders each layer's tensors in compute order
    (input norm, q, k, v, o, post-attention norm, gate, up, down), embedding
    first and untied head last; all tensors decay.
  * The 2.5B clip case is a GPT-2-style stack (LayerNorm weight+bias twice,
    fused qkv + bias, projection + bias, fc + bias, fc-projection + bias) with a
    tied embedding, a final LayerNorm and no positional table: 387 tensors,
    2,646,430,720 parameters.  Decay applies to tensors with ndim >= 2 only.
  * The same-hyperparameters wording of the 1.1B case includes the clip at 1.0
    that the plumbing case lists among its AdamW settings.
  * The sweep case draws 6000 log-uniform sizes in [4096, 65536] and interleaves
    them as 24 groups of (one 1024x4096 matrix + 250 small tensors); the realised
    total (~234M) is reported rather than the nominal 350M.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

MiB = 1 << 20


@dataclass(frozen=True)
class AdamW:
    lr: float = 2e-4
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    max_norm: float = 1.0  # <= 0 disables clipping


@dataclass
class Workload:
    name: str
    P: int
    names: list
    shapes: list
    bucket_bytes: int
    sigma: float                      # per-rank gradient standard deviation
    outlier_frac: float = 0.0         # fraction of gradient entries scaled by outlier_scale
    outlier_scale: float = 100.0
    master_sigma: float = 0.02
    adamw: AdamW = field(default_factory=AdamW)
    steps: int = 1
    mode: str = "zero"                # "zero" (fused ZeRO-2 step) or "allreduce"
    decay_rule: str = "all"           # "all" or "ndim>=2"
    seed: int = 0

    @property
    def sizes(self):
        return [int(math.prod(s)) for s in self.shapes]

    @property
    def n_params(self):
        return sum(self.sizes)

    @property
    def decay(self):
        if self.decay_rule == "all":
            return [1] * len(self.shapes)
        return [1 if len(s) >= 2 else 0 for s in self.shapes]


def tiny_plumbing() -> Workload:
    sizes = [3, 1000, 65536, 131071, 262144, 262144, 279105]
    return Workload(name="tiny-P4-1M", P=4, names=[f"t{i}" for i in range(7)],
                    shapes=[(s,) for s in sizes], bucket_bytes=1 * MiB, sigma=1e-3,
                    steps=3, mode="zero", seed=0)


def gpt2_small_allreduce() -> Workload:
    d, ffn, vocab, ctx, L = 768, 3072, 50257, 1024, 12
    names, shapes = ["wte", "wpe"], [(vocab, d), (ctx, d)]
    for i in range(L):
        for n, s in (("ln_1.weight", (d,)), ("ln_1.bias", (d,)),
                     ("attn.c_attn.weight", (d, 3 * d)), ("attn.c_attn.bias", (3 * d,)),
                     ("attn.c_proj.weight", (d, d)), ("attn.c_proj.bias", (d,)),
                     ("ln_2.weight", (d,)), ("ln_2.bias", (d,)),
                     ("mlp.c_fc.weight", (d, ffn)), ("mlp.c_fc.bias", (ffn,)),
                     ("mlp.c_proj.weight", (ffn, d)), ("mlp.c_proj.bias", (d,))):
            names.append(f"h.{i}.{n}")
            shapes.append(s)
    names += ["ln_f.weight", "ln_f.bias"]
    shapes += [(d,), (d,)]
    return Workload(name="gpt2-small-124M-P8-allreduce", P=8, names=names, shapes=shapes,
                    bucket_bytes=25 * MiB, sigma=1e-3, outlier_frac=0.01, mode="allreduce",
                    seed=1)


def llama_1b1_zero2(layers: int = 22, embeddings: bool = True) -> Workload:
    """Llama-style 1.1B (22 layers).  `layers`/`embeddings` give the small
    profiling variant (same tensor shapes and 25 MiB buckets, fewer layers)."""
    d, ffn, vocab, L, kv = 2048, 5632, 32000, layers, 256   # 4 KV heads of 64
    names, shapes = (["embed_tokens"], [(vocab, d)]) if embeddings else ([], [])
    for i in range(L):
        for n, s in (("input_layernorm", (d,)), ("q_proj", (d, d)), ("k_proj", (kv, d)),
                     ("v_proj", (kv, d)), ("o_proj", (d, d)),
                     ("post_attention_layernorm", (d,)), ("gate_proj", (ffn, d)),
                     ("up_proj", (ffn, d)), ("down_proj", (d, ffn))):
            names.append(f"layers.{i}.{n}")
            shapes.append(s)
    names += ["norm"]
    shapes += [(d,)]
    if embeddings:
        names += ["lm_head"]
        shapes += [(vocab, d)]
    name = "llama-1.1B-P8-zero2" if (layers, embeddings) == (22, True) else \
        f"llama-{layers}L-P8-zero2"
    return Workload(name=name, P=8, names=names, shapes=shapes,
                    bucket_bytes=25 * MiB, sigma=5e-4, steps=10, mode="zero", seed=2)


def gpt_2b5_clip() -> Workload:
    d, ffn, vocab, L, P = 2560, 10240, 50304, 32, 8
    names, shapes = ["wte"], [(vocab, d)]
    for i in range(L):
        for n, s in (("ln_1.weight", (d,)), ("ln_1.bias", (d,)),
                     ("attn.qkv.weight", (3 * d, d)), ("attn.qkv.bias", (3 * d,)),
                     ("attn.proj.weight", (d, d)), ("attn.proj.bias", (d,)),
                     ("ln_2.weight", (d,)), ("ln_2.bias", (d,)),
                     ("mlp.fc.weight", (ffn, d)), ("mlp.fc.bias", (ffn,)),
                     ("mlp.proj.weight", (d, ffn)), ("mlp.proj.bias", (d,))):
            names.append(f"h.{i}.{n}")
            shapes.append(s)
    names += ["ln_f.weight", "ln_f.bias"]
    shapes += [(d,), (d,)]
    n = sum(int(math.prod(s)) for s in shapes)
    sigma = 4.0 * math.sqrt(P / n)     # E||mean|| ~= 4 so clipping to 1.0 is active
    return Workload(name="gpt-2.5B-P8-zero2-clip", P=P, names=names, shapes=shapes,
                    bucket_bytes=25 * MiB, sigma=sigma, steps=1, mode="zero",
                    decay_rule="ndim>=2", seed=3)


def sweep_small_tensors(bucket_bytes: int = 25 * MiB, mode: str = "zero",
                        groups: int = 24) -> Workload:
    """24 groups of (one 1024 x 4096 matrix + 250 log-uniform 4K-64K vectors);
    `groups` < 24 keeps the first groups only (a smaller case of the same shapes)."""
    import numpy as np
    rng = np.random.default_rng(4)
    small = np.exp(rng.uniform(math.log(4096), math.log(65536), size=6000))
    small = np.floor(small).astype(np.int64)
    names, shapes = [], []
    for g in range(groups):
        names.append(f"mat.{g}")
        shapes.append((1024, 4096))
        for j in range(250):
            k = g * 250 + j
            names.append(f"small.{k}")
            shapes.append((int(small[k]),))
    tag = "" if groups == 24 else f"-{groups}g"
    return Workload(name=f"sweep-P16-{bucket_bytes // 1024}KiB-{mode}{tag}", P=16, names=names,
                    shapes=shapes, bucket_bytes=bucket_bytes, sigma=1e-3, mode=mode, seed=4)


SWEEP_BUCKETS = [64 * 1024, 1 * MiB, 25 * MiB, 256 * MiB]


def all_workloads():
    return [tiny_plumbing(), gpt2_small_allreduce(), llama_1b1_zero2(), gpt_2b5_clip(),
            sweep_small_tensors()]

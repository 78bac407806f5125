"""Synthetic workloads: tensor counts and the counter-based generator."""
import math

import numpy as np
import torch

from workloads import configs, gen


def test_parameter_counts():
    w = configs.tiny_plumbing()
    assert (len(w.shapes), w.n_params) == (7, 1_001_003)
    w = configs.gpt2_small_allreduce()
    assert (len(w.shapes), w.n_params) == (148, 124_439_808)
    w = configs.llama_1b1_zero2()
    assert (len(w.shapes), w.n_params) == (201, 1_100_048_384)
    w = configs.gpt_2b5_clip()
    assert (len(w.shapes), w.n_params) == (387, 2_646_430_720)
    assert sum(w.decay) == 1 + 32 * 4              # matrices only
    w = configs.sweep_small_tensors()
    assert len(w.shapes) == 6024
    small = [s for s, n in zip(w.sizes, w.names) if n.startswith("small")]
    assert min(small) >= 4096 and max(small) <= 65536


def test_splitmix64_tensor_matches_definition():
    xs = [0, 1, 2, 12345678901234, (1 << 64) - 1, 1 << 63, 0xDEADBEEFCAFEBABE]
    t = torch.tensor([gen._s64(x) for x in xs], dtype=torch.int64)
    got = [v & gen._MASK64 for v in gen.splitmix64(t).tolist()]
    assert got == [gen.splitmix64_int(x) for x in xs]
    # first output of SplitMix64 seeded with 0 (published test value)
    assert gen.splitmix64_int(0) == 0xE220A8397B1DCDAF


def test_generator_is_counter_based_and_seeded():
    w = configs.tiny_plumbing()
    a = gen.grad_values(w, step=1, rank=2, start=0, count=5000)
    b = gen.grad_values(w, step=1, rank=2, start=1000, count=2000)
    assert torch.equal(a[1000:3000], b)
    c = gen.grad_values(w, step=1, rank=3, start=0, count=5000)
    assert not torch.equal(a, c)
    x = a.float().numpy().astype(np.float64)
    assert abs(x.mean()) < 4 * w.sigma / math.sqrt(len(x))
    assert abs(x.std() / w.sigma - 1) < 0.05


def test_outlier_fraction():
    w = configs.gpt2_small_allreduce()
    x = gen.grad_values(w, 1, 0, 0, 200000).float().abs()
    frac = (x > 20 * w.sigma).float().mean().item()
    assert 0.007 < frac < 0.013

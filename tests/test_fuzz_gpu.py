"""Seeded random plans against the oracle: tensor counts and sizes (zero-size,
one-element, larger than the cap), bucket caps, rank counts 1..64 and mesh shapes
drawn at random; the mean all-reduce, the clipped ZeRO-2 step and, on mesh plans,
the hybrid all-reduce must match the oracle bit for bit, on both launch shapes."""
import numpy as np
import pytest
import torch

import gradient_sync_zero_gb300 as dps
import oracle as oracle_mod
from harness import Case, small_workload
from workloads import configs

pytestmark = pytest.mark.gpu


def random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.integers(1, 12))
    kinds = rng.integers(0, 4, size=n)
    sizes = [int(x) for x in np.where(kinds == 0, rng.integers(0, 3, size=n),
                                      np.where(kinds == 1, rng.integers(1, 300, size=n),
                                               rng.integers(300, 40000, size=n)))]
    P = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16, 24, 32, 64]))
    cap = int(rng.choice([64, 1024, 8192, 65536, 1 << 20]))
    wl = small_workload(sizes, P, cap, sigma=float(rng.choice([1e-3, 0.05])), seed=seed,
                        outlier_frac=0.01)
    return wl, rng


@pytest.mark.parametrize("seed", range(12))
def test_random_plan_allreduce(orc, seed):
    wl, _ = random_case(seed)
    c = Case(wl)
    g = c.host_grads(1)
    buf = c.to_replicas(g)
    dps.dp_allreduce_mean(c.plan, c.ws, buf)
    torch.cuda.synchronize()
    want, _, _ = orc.allreduce_mean(c.sizes, wl.bucket_bytes, wl.P, g)
    assert np.array_equal(c.from_replicas(buf), want)


@pytest.mark.parametrize("seed", range(12))
def test_random_plan_zero_step_clipped(orc, seed):
    wl, _ = random_case(seed)
    wl.adamw = configs.AdamW(max_norm=0.05)
    c = Case(wl)
    g = c.host_grads(1)
    master0 = c.host_master()
    params = c.plan.new_replicas()
    st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    a = wl.adamw
    cfg = dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, 1)
    dps.dp_fused_zero_step(c.plan, c.ws, c.to_replicas(g), params, *st, cfg)
    norm, coef, status = dps.dp_read_norm(c.plan, c.ws)
    z = np.zeros_like(master0)
    p_o, m_o, mo, vo, _, so = orc.zero_step(c.sizes, c.decay, wl.bucket_bytes, wl.P, g, master0, z,
                                            z, oracle_mod.adamw_cfg(a, 1))
    assert status == 0 and coef == so.coef
    assert np.array_equal(c.from_replicas(params), p_o)
    for dev, ref in zip(st, (m_o, mo, vo)):
        assert np.array_equal(c.from_flat(dev).view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("seed", range(8))
def test_random_mesh_allreduce(orc, seed):
    wl, rng = random_case(seed)
    shapes = [(R, S) for R in (2, 3, 4, 8) for S in (1, 2, 3, 4, 8) if R * S <= 64]
    R, S = shapes[int(rng.integers(0, len(shapes)))]
    wl = small_workload(wl.sizes, R * S, wl.bucket_bytes, sigma=1e-3, seed=seed)
    c = Case.__new__(Case)
    c.wl, c.P, c.sizes, c.decay = wl, wl.P, wl.sizes, list(wl.decay)
    c.plan = dps.Plan(c.sizes, wl.bucket_bytes, c.P, c.decay, mesh=(R, S))
    c.off, c.device, c.ws = c.plan.tensor_offsets(), "cuda", c.plan.new_workspace()
    g = c.host_grads(1)
    buf = c.to_replicas(g)
    dps.dp_allreduce_mean(c.plan, c.ws, buf)
    torch.cuda.synchronize()
    want, _, _ = orc.mesh_allreduce_mean(c.sizes, wl.bucket_bytes, R, S, g)
    assert np.array_equal(c.from_replicas(buf), want)


@pytest.mark.parametrize("shape", ["persistent", "short-ctas"])
@pytest.mark.parametrize("seed", range(12))
def test_random_plan_per_bucket_launches(orc, seed, shape):
    """Random plans launched bucket by bucket in backward order (the small-launch
    kernels wherever a bucket's tiles fit, or, on a stream set to short-lived CTAs,
    always): the all-reduce and the reduce-scatter mean equal the oracle, and the
    clip norm from per-bucket norm partials equals the one from a single launch,
    bit for bit."""
    wl, _ = random_case(seed)
    c = Case(wl)
    g = c.host_grads(1)
    nb = c.plan.n_buckets
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    if shape == "short-ctas":
        dps.set_stream_launch(stream, True)
    try:
        with torch.cuda.stream(stream):
            buf = c.to_replicas(g)
            mean_a, mean_b = c.plan.new_state(), c.plan.new_state()
            dps.dp_reduce_scatter_mean(c.plan, c.ws, buf, mean_a, want_sumsq=True)
            dps.dp_clip_coef(c.plan, c.ws, 0.05)
            single = dps.dp_read_norm(c.plan, c.ws)
            for b in reversed(range(nb)):
                dps.dp_reduce_scatter_mean(c.plan, c.ws, buf, mean_b, b, b + 1, want_sumsq=True)
            dps.dp_clip_coef(c.plan, c.ws, 0.05)
            per_bucket = dps.dp_read_norm(c.plan, c.ws)
            for b in reversed(range(nb)):
                dps.dp_allreduce_mean(c.plan, c.ws, buf, b, b + 1)
        stream.synchronize()
    finally:
        dps.set_stream_launch(stream, False)
    assert per_bucket == single
    assert torch.equal(mean_a.view(torch.int32), mean_b.view(torch.int32))
    want, want_mean, _ = orc.allreduce_mean(c.sizes, wl.bucket_bytes, wl.P, g)
    assert np.array_equal(c.from_flat(mean_b).view(np.uint32), want_mean.view(np.uint32))
    assert np.array_equal(c.from_replicas(buf), want)


@pytest.mark.parametrize("seed", range(8))
def test_random_plan_unclipped_zero_step_short_ctas(orc, seed):
    """The one-pass ZeRO step (no clip) on a stream set to short-lived CTAs (one CTA
    per tile) over random plans: every replica and master/m/v equal the oracle."""
    wl, _ = random_case(seed)
    wl.adamw = configs.AdamW(max_norm=0.0)
    c = Case(wl)
    g = c.host_grads(1)
    master0 = c.host_master()
    a = wl.adamw
    cfg = dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, 0.0, 1)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    dps.set_stream_launch(stream, True)
    try:
        with torch.cuda.stream(stream):
            params = c.plan.new_replicas()
            st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
            dps.dp_fused_zero_step(c.plan, c.ws, c.to_replicas(g), params, *st, cfg)
        stream.synchronize()
    finally:
        dps.set_stream_launch(stream, False)
    z = np.zeros_like(master0)
    p_o, m_o, mo, vo, _, _ = orc.zero_step(c.sizes, c.decay, wl.bucket_bytes, wl.P, g, master0, z,
                                           z, oracle_mod.adamw_cfg(a, 1))
    assert np.array_equal(c.from_replicas(params), p_o)
    for dev, ref in zip(st, (m_o, mo, vo)):
        assert np.array_equal(c.from_flat(dev).view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("seed", range(4))
def test_random_plan_buckets_on_concurrent_streams(orc, seed):
    """Buckets touch disjoint memory, so per-bucket launches may run at once: bucket b
    on stream b mod 4 (reduce-scatter with norm partials, then all-reduce), joined
    before the clip norm.  The results equal the oracle and the single launch."""
    wl, _ = random_case(seed)
    c = Case(wl)
    g = c.host_grads(1)
    nb = c.plan.n_buckets
    buf, mean = c.to_replicas(g), c.plan.new_state()
    dps.dp_reduce_scatter_mean(c.plan, c.ws, buf, c.plan.new_state(), want_sumsq=True)
    dps.dp_clip_coef(c.plan, c.ws, 0.05)
    single = dps.dp_read_norm(c.plan, c.ws)
    streams = [torch.cuda.Stream() for _ in range(4)]
    cur = torch.cuda.current_stream()
    for s_ in streams:
        s_.wait_stream(cur)
    for b in range(nb):
        with torch.cuda.stream(streams[b % 4]):
            dps.dp_reduce_scatter_mean(c.plan, c.ws, buf, mean, b, b + 1, want_sumsq=True)
    for s_ in streams:
        cur.wait_stream(s_)
    dps.dp_clip_coef(c.plan, c.ws, 0.05)
    assert dps.dp_read_norm(c.plan, c.ws) == single
    for s_ in streams:
        s_.wait_stream(cur)
    for b in reversed(range(nb)):
        with torch.cuda.stream(streams[b % 4]):
            dps.dp_allreduce_mean(c.plan, c.ws, buf, b, b + 1)
    for s_ in streams:
        cur.wait_stream(s_)
    torch.cuda.synchronize()
    want, want_mean, _ = orc.allreduce_mean(c.sizes, wl.bucket_bytes, wl.P, g)
    assert np.array_equal(c.from_flat(mean).view(np.uint32), want_mean.view(np.uint32))
    assert np.array_equal(c.from_replicas(buf), want)

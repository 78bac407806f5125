"""Gradient accumulation and the bf16-on-the-wire ring on the GPU.

Accumulation: no sync on every micro-batch but the last, which syncs
("Distributed Training: Data Parallel, Model Parallel and FSDP Strategies",
"Selecting and Tuning"); each rank's bf16 gradient buffer accumulates as
acc = bf16(acc + g).  bf16 on the wire: every ring hop's partial sum is rounded
to bf16 ("Data Parallelism: From Parameter Server to Ring All-Reduce", sec. 8).
Both are compared with the oracle bit for bit."""
import numpy as np
import pytest
import torch

import gradient_sync_zero_gb300 as dps
from harness import Case, assert_replicas_equal, small_workload, u16
from workloads import configs

pytestmark = pytest.mark.gpu

SIZES = [3, 1000, 65536, 13107, 26214, 4097, 27910, 9000]


def micro_batches(c, k):
    return [c.host_grads(1 + i) for i in range(k)]


@pytest.mark.parametrize("P", [1, 3, 8, 12, 16])
def test_accumulate_equals_oracle(orc, P):
    wl = small_workload(SIZES, P, 32 * 1024, seed=P, outlier_frac=0.01)
    c = Case(wl)
    m = micro_batches(c, 3)
    acc = c.to_replicas(m[0])
    want = m[0]
    for x in m[1:]:
        dps.dp_accumulate(c.plan, c.ws, acc, c.to_replicas(x))
        want = orc.accumulate(want, x)
    torch.cuda.synchronize()
    assert np.array_equal(c.from_replicas(acc), want)
    assert not acc[:, :c.plan.L][:, c.padding_mask().cuda()].any()   # padding stays zero


@pytest.mark.parametrize("P", [2, 5, 8, 12, 16, 64])
def test_last_micro_batch_fused_equals_oracle(orc, P):
    """k-1 local accumulations, then one fused accumulate + mean all-reduce =
    oracle accumulate k-1 times, then its ring all-reduce."""
    wl = small_workload(SIZES, P, 32 * 1024, seed=10 + P, outlier_frac=0.01)
    c = Case(wl)
    m = micro_batches(c, 4)
    acc = c.to_replicas(m[0])
    for x in m[1:3]:
        dps.dp_accumulate(c.plan, c.ws, acc, c.to_replicas(x))
    two = acc.clone()
    last = c.to_replicas(m[3])
    dps.dp_allreduce_mean_accum(c.plan, c.ws, acc, last)
    # the unfused sequence on the GPU gives the same bits
    dps.dp_accumulate(c.plan, c.ws, two, last)
    dps.dp_allreduce_mean(c.plan, c.ws, two)
    torch.cuda.synchronize()
    assert torch.equal(acc, two)
    want = m[0]
    for x in m[1:]:
        want = orc.accumulate(want, x)
    out, _, _ = orc.allreduce_mean(c.sizes, wl.bucket_bytes, P, want, want_mean=False)
    assert np.array_equal(c.from_replicas(acc), out)
    assert_replicas_equal(acc, c.plan.L)


@pytest.mark.parametrize("P", [2, 4, 7, 8, 16, 24])
def test_bf16_wire_equals_oracle(orc, P):
    wl = small_workload(SIZES, P, 32 * 1024, seed=20 + P, outlier_frac=0.01)
    c = Case(wl)
    g = c.host_grads(1)
    buf = c.to_replicas(g)
    dps.dp_allreduce_mean_bf16wire(c.plan, c.ws, buf)
    torch.cuda.synchronize()
    want, _ = orc.allreduce_mean_bf16wire(c.sizes, wl.bucket_bytes, P, g)
    assert np.array_equal(c.from_replicas(buf), want)
    assert_replicas_equal(buf, c.plan.L)


def test_bf16_wire_bucket_range_and_error_bound():
    """Buckets outside [b0, b1) are untouched, buckets inside equal a full run.
    Against the fp32 ring, the bf16 ring's error stays inside what its roundings
    allow: each of the P-1 hops rounds a partial sum (at most sum|g|) to bf16
    (unit roundoff u = 2^-8), the quotient is divided by P, and both results take
    one final bf16 rounding: |a - b| <= (P-1) u sum|g| / P + 2 u |mean| (+ 1e-30)."""
    P = 8
    wl = small_workload(SIZES, P, 32 * 1024, seed=5, sigma=1e-2, outlier_frac=0.01)
    c = Case(wl)
    g = c.host_grads(1)
    full, part, ref = c.to_replicas(g), c.to_replicas(g), c.to_replicas(g)
    nb = c.plan.n_buckets
    assert nb >= 3
    dps.dp_allreduce_mean_bf16wire(c.plan, c.ws, full)
    dps.dp_allreduce_mean_bf16wire(c.plan, c.ws, part, 1, nb)
    torch.cuda.synchronize()
    lo = c.plan.bucket(1)[0]
    assert torch.equal(part[:, :lo], ref[:, :lo])
    assert torch.equal(part[:, lo:], full[:, lo:])
    dps.dp_allreduce_mean(c.plan, c.ws, ref)
    torch.cuda.synchronize()
    def f(u):
        return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    a, b = f(c.from_replicas(full)[0]), f(c.from_replicas(ref)[0])
    gf = f(g)
    u = 2.0 ** -8
    bound = (P - 1) * u * np.abs(gf).sum(0) / P + 2 * u * np.abs(gf.sum(0) / P) + 1e-30
    assert np.all(np.abs(a - b) <= bound)
    assert np.any(a != b)                       # the two rings do differ


def test_mesh_plans_are_refused():
    plan = dps.Plan([4096, 100], 1 << 20, 8, mesh=(2, 4))
    ws = plan.new_workspace()
    g = plan.new_replicas()
    with pytest.raises(dps.DPError) as e:
        dps.dp_allreduce_mean_bf16wire(plan, ws, g)
    assert e.value.code == dps.DP_EINVAL
    with pytest.raises(dps.DPError):
        dps.dp_allreduce_mean_accum(plan, ws, g, plan.new_replicas())


def test_full_size_gpt2_accumulation_sampled(orc):
    """GPT-2 small, P = 8, two micro-batches, fused last step: sampled tensors
    against the oracle (accumulate, then the ring all-reduce of those tensors'
    own buckets is checked through the unfused GPU path, which the oracle
    pins at full size elsewhere)."""
    wl = configs.gpt2_small_allreduce()
    c = Case(wl)
    from workloads import device as wdev
    m0, m1 = c.plan.new_replicas(), c.plan.new_replicas()
    wdev.fill_grads(m0, c.off, wl, 1)
    wdev.fill_grads(m1, c.off, wl, 2)
    acc = m0.clone()
    dps.dp_allreduce_mean_accum(c.plan, c.ws, acc, m1)
    two = m0.clone()
    dps.dp_accumulate(c.plan, c.ws, two, m1)
    summed = two.clone()
    dps.dp_allreduce_mean(c.plan, c.ws, two)
    torch.cuda.synchronize()
    assert torch.equal(acc, two)
    # the local accumulation, sampled tensors, against the oracle
    for t in (0, 1, len(wl.sizes) // 2, len(wl.sizes) - 1):
        o, s = c.off[t], wl.sizes[t]
        a = np.stack([u16(m0[r, o:o + s]) for r in range(wl.P)])
        b = np.stack([u16(m1[r, o:o + s]) for r in range(wl.P)])
        assert np.array_equal(np.stack([u16(summed[r, o:o + s]) for r in range(wl.P)]),
                              orc.accumulate(a, b))


@pytest.mark.parametrize("P", [2, 5, 8, 16, 24])
def test_last_micro_batch_reduce_scatter_equals_oracle(orc, P):
    """ZeRO form: the fused last micro-batch reduce-scatter gives the oracle's fp32
    mean of the accumulated gradients bit for bit, the same norm partials as the
    unfused path, and leaves acc and micro unchanged."""
    wl = small_workload(SIZES, P, 32 * 1024, seed=40 + P, outlier_frac=0.01)
    c = Case(wl)
    m = micro_batches(c, 3)
    acc = c.to_replicas(m[0])
    dps.dp_accumulate(c.plan, c.ws, acc, c.to_replicas(m[1]))
    last = c.to_replicas(m[2])
    acc0, last0 = acc.clone(), last.clone()
    mean = c.plan.new_state()
    dps.dp_reduce_scatter_mean_accum(c.plan, c.ws, acc, last, mean, want_sumsq=True)
    dps.dp_clip_coef(c.plan, c.ws, 1.0)
    n_fused = dps.dp_read_norm(c.plan, c.ws)
    ws2 = c.plan.new_workspace()
    two, mean2 = acc.clone(), c.plan.new_state()
    dps.dp_accumulate(c.plan, ws2, two, last)
    dps.dp_reduce_scatter_mean(c.plan, ws2, two, mean2, want_sumsq=True)
    dps.dp_clip_coef(c.plan, ws2, 1.0)
    n_two = dps.dp_read_norm(c.plan, ws2)
    torch.cuda.synchronize()
    assert torch.equal(acc, acc0) and torch.equal(last, last0)
    assert torch.equal(mean.view(torch.int32), mean2.view(torch.int32)) and n_fused == n_two
    want = orc.accumulate(orc.accumulate(m[0], m[1]), m[2])
    _, omean, _ = orc.allreduce_mean(c.sizes, wl.bucket_bytes, P, want)
    assert np.array_equal(c.from_flat(mean).view(np.uint32), omean.view(np.uint32))


def test_accumulated_zero_step_equals_oracle(orc):
    """Two micro-batches, then the fused last-micro-batch reduce-scatter, the clip
    coefficient and the AdamW + all-gather pass: the oracle's ZeRO step on the
    accumulated gradients, bit for bit."""
    import oracle as oracle_mod
    wl = configs.tiny_plumbing()
    wl.adamw = configs.AdamW(max_norm=0.3)
    c = Case(wl)
    m0, m1 = c.host_grads(1), c.host_grads(2)
    acc, last = c.to_replicas(m0), c.to_replicas(m1)
    master0 = c.host_master()
    st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    params, mean = c.plan.new_replicas(), c.plan.new_state()
    a = wl.adamw
    cfg = dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, 1)
    dps.dp_reduce_scatter_mean_accum(c.plan, c.ws, acc, last, mean, want_sumsq=True)
    dps.dp_clip_coef(c.plan, c.ws, a.max_norm)
    dps.dp_adamw_all_gather(c.plan, c.ws, mean, *st, params, cfg)
    norm, coef, status = dps.dp_read_norm(c.plan, c.ws)
    g = orc.accumulate(m0, m1)
    z = np.zeros_like(master0)
    p_o, m_o, mo, vo, _, so = orc.zero_step(c.sizes, c.decay, wl.bucket_bytes, wl.P, g, master0, z, z,
                                            oracle_mod.adamw_cfg(a, 1))
    assert status == 0 and coef == so.coef < 1.0
    assert np.array_equal(c.from_replicas(params), p_o)
    for dev, ref in zip(st, (m_o, mo, vo)):
        assert np.array_equal(c.from_flat(dev).view(np.uint32), ref.view(np.uint32))

"""GPU path against the CPU oracle, element by element, at sizes the oracle
finishes in seconds (several tiles per bucket, ragged tails, zero-size tensors,
oversized tensors, P from 1 to 16, rank counts without a dedicated
instantiation, and P = 64, the largest the planner accepts).

Tolerances (stated by the target): reduced fp32 gradients <= 1e-6 relative,
fp32 master/m/v <= 1e-5 relative after 3 steps, bf16 parameters within 1 ulp,
replica equality and layout bit-exact.  Without clipping the arithmetic is the
same op for op, so bit equality is asserted too; with clipping the norm is
summed differently (float-float tree on the GPU, sequential double in the
oracle) but both are accurate to ~1e-12, so the fp32 clip coefficient rounds
the same and bit equality is asserted as well.
"""
import math

import numpy as np
import pytest
import torch

import gradient_sync_zero_gb300 as dps
from harness import (Case, assert_replicas_equal, bf16_ulp_diff, rel_err, small_workload, u16)
from workloads import configs

pytestmark = pytest.mark.gpu

SIZE_SETS = {
    "ragged": [3, 1000, 65536, 13107, 26214, 4097, 27910],
    "zeros": [0, 517, 0, 9000, 1, 0],
    "oversized": [70000, 12, 130000, 5],
}
RANKS = [1, 2, 3, 4, 5, 7, 8, 11, 16, 64]   # 64: the largest rank count the planner accepts


def case_for(sizes_key, P, cap=64 * 1024, sigma=1e-3, seed=0, decay=None):
    sizes = SIZE_SETS[sizes_key]
    wl = small_workload(sizes, P, cap, sigma=sigma, seed=seed + P, decay=decay)
    return Case(wl)


@pytest.mark.parametrize("P", RANKS)
@pytest.mark.parametrize("sizes_key", sorted(SIZE_SETS))
def test_allreduce_matches_oracle(orc, P, sizes_key):
    c = case_for(sizes_key, P)
    g = c.host_grads(1)
    dev = c.to_replicas(g)
    dps.dp_allreduce_mean(c.plan, c.ws, dev)
    torch.cuda.synchronize()
    want, mean, st = orc.allreduce_mean(c.sizes, c.wl.bucket_bytes, P, g)
    got = c.from_replicas(dev)
    assert np.array_equal(got, want)
    assert_replicas_equal(dev, c.plan.L)
    pad = c.padding_mask().to(dev.device)
    assert not dev[:, :c.plan.L][:, pad].any(), "padding must stay zero"
    assert st.replicas_equal == 1


@pytest.mark.parametrize("P", RANKS)
def test_reduce_scatter_matches_oracle(orc, P):
    c = case_for("ragged", P)
    g = c.host_grads(2)
    dev = c.to_replicas(g)
    mean = c.plan.new_state()
    dps.dp_reduce_scatter_mean(c.plan, c.ws, dev, mean)
    torch.cuda.synchronize()
    _, want, _ = orc.allreduce_mean(c.sizes, c.wl.bucket_bytes, P, g)
    got = c.from_flat(mean)
    assert np.all(rel_err(got, want) <= 1e-6)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert not mean[c.padding_mask().cuda()].any()
    assert torch.equal(dev, c.to_replicas(g)), "reduce-scatter must not modify its input"


def run_oracle_steps(orc, c, grads_by_step, master, cfgs):
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    out = []
    for g, cfg in zip(grads_by_step, cfgs):
        params, master, m, v, mean, st = orc.zero_step(c.sizes, c.decay, c.wl.bucket_bytes, c.P, g,
                                                       master, m, v, cfg)
        out.append((params, master.copy(), m.copy(), v.copy(), st))
    return out


def ocfg(adamw, step):
    import oracle
    return oracle.adamw_cfg(adamw, step)


def dcfg(adamw, step):
    return dps.adamw_cfg(adamw.lr, adamw.beta1, adamw.beta2, adamw.eps, adamw.weight_decay,
                         adamw.max_norm, step)


def check_state(c, dev_params, dev_state, ref, exact):
    params, master, m, v, _ = ref
    got_p = c.from_replicas(dev_params)
    got = [c.from_flat(t) for t in dev_state]
    for name, a, b in zip(("master", "m", "v"), got, (master, m, v)):
        e = rel_err(a, b)
        assert np.all(e <= 1e-5), f"{name}: max rel err {e.max():.3g}"
        if exact:
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), f"{name} not bit-exact"
    assert np.all(bf16_ulp_diff(got_p, params) <= 1)
    if exact:
        assert np.array_equal(got_p, params)
    assert_replicas_equal(dev_params, c.plan.L)


@pytest.mark.parametrize("P", RANKS)
def test_fused_zero_no_clip_matches_oracle(orc, P):
    c = case_for("ragged", P, decay=[1, 0, 1, 1, 0, 1, 1])
    adamw = configs.AdamW(max_norm=0.0)
    master0 = c.host_master()
    grads = [c.host_grads(s) for s in (1, 2, 3)]
    ref = run_oracle_steps(orc, c, grads, master0, [ocfg(adamw, s) for s in (1, 2, 3)])
    params = c.plan.new_replicas()
    st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    for s, g in zip((1, 2, 3), grads):
        dps.dp_fused_zero_step(c.plan, c.ws, c.to_replicas(g), params, *st, dcfg(adamw, s))
        torch.cuda.synchronize()
        check_state(c, params, st, ref[s - 1], exact=True)
    assert not params[:, :c.plan.L][:, c.padding_mask().cuda()].any()
    assert not st[0][c.padding_mask().cuda()].any()


@pytest.mark.parametrize("P", [2, 4, 8, 11])
def test_staged_zero_equals_oracle(orc, P):
    """reduce-scatter -> sharded AdamW -> all-gather, as three calls."""
    c = case_for("oversized", P)
    adamw = configs.AdamW(max_norm=0.0)
    master0 = c.host_master()
    grads = [c.host_grads(s) for s in (1, 2)]
    ref = run_oracle_steps(orc, c, grads, master0, [ocfg(adamw, s) for s in (1, 2)])
    params = c.plan.new_replicas()
    st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    mean = c.plan.new_state()
    for s, g in zip((1, 2), grads):
        dps.dp_reduce_scatter_mean(c.plan, c.ws, c.to_replicas(g), mean)
        dps.dp_sharded_adamw_step(c.plan, c.ws, mean, *st, params, dcfg(adamw, s))
        dps.dp_all_gather(c.plan, c.ws, params)
        torch.cuda.synchronize()
        check_state(c, params, st, ref[s - 1], exact=True)


@pytest.mark.parametrize("P", [3, 4, 8, 16])
def test_fused_zero_clip_matches_oracle(orc, P):
    c = case_for("ragged", P, sigma=0.05)           # ||mean|| > 1: clipping active
    adamw = configs.AdamW(max_norm=1.0)
    master0 = c.host_master()
    grads = [c.host_grads(s) for s in (1, 2, 3)]
    ref = run_oracle_steps(orc, c, grads, master0, [ocfg(adamw, s) for s in (1, 2, 3)])
    params = c.plan.new_replicas()
    st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    for s, g in zip((1, 2, 3), grads):
        dps.dp_fused_zero_step(c.plan, c.ws, c.to_replicas(g), params, *st, dcfg(adamw, s))
        norm, coef, status = dps.dp_read_norm(c.plan, c.ws)
        ost = ref[s - 1][4]
        assert status == 0
        assert ost.coef < 1.0
        assert math.isclose(norm, ost.norm, rel_tol=1e-12)
        # the float-float norm rounds to the oracle's fp32 coefficient, after
        # which both sides run the same ops: bit equality throughout
        assert coef == ost.coef
        check_state(c, params, st, ref[s - 1], exact=True)


def test_staged_clip_equals_fused_clip():
    """RS(+partials) -> clip coef -> AdamW(coef) -> all-gather == the fused call."""
    c = case_for("zeros", 4, sigma=0.2)
    adamw = configs.AdamW(max_norm=1.0)
    master0 = c.host_master()
    g = c.to_replicas(c.host_grads(1))
    p1, p2 = c.plan.new_replicas(), c.plan.new_replicas()
    s1 = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    s2 = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    dps.dp_fused_zero_step(c.plan, c.ws, g, p1, *s1, dcfg(adamw, 1))
    n1 = dps.dp_read_norm(c.plan, c.ws)
    mean = c.plan.new_state()
    for b in range(c.plan.n_buckets):          # per-bucket launches, DDP style
        dps.dp_reduce_scatter_mean(c.plan, c.ws, g, mean, b, b + 1, want_sumsq=True)
    dps.dp_clip_coef(c.plan, c.ws, 1.0)
    dps.dp_sharded_adamw_step(c.plan, c.ws, mean, *s2, p2, dcfg(adamw, 1), use_clip_coef=True)
    dps.dp_all_gather(c.plan, c.ws, p2)
    n2 = dps.dp_read_norm(c.plan, c.ws)
    assert n1 == n2 and n1[1] < 1.0
    assert torch.equal(p1, p2)
    for a, b in zip(s1, s2):
        assert torch.equal(a, b)


@pytest.mark.parametrize("P", [4, 8])
def test_caller_given_clip_coefficient_matches_oracle(orc, P):
    """An update given the caller's own clip coefficient (coef_dev) uses it, not
    the workspace's: the workspace holds the coefficient for max_norm 1.0, the
    caller's device float is the oracle's for max_norm 0.3 on the same
    gradients, and the result equals the oracle's step at max_norm 0.3, bit for
    bit, over three steps, through dp_sharded_adamw_step + dp_all_gather and
    through dp_adamw_all_gather."""
    c = case_for("ragged", P, sigma=0.05, decay=[1, 0, 1, 1, 0, 1, 1])
    adamw_ws = configs.AdamW(max_norm=1.0)
    adamw_own = configs.AdamW(max_norm=0.3)
    master0 = c.host_master()
    grads = [c.host_grads(s) for s in (1, 2, 3)]
    ref = run_oracle_steps(orc, c, grads, master0, [ocfg(adamw_own, s) for s in (1, 2, 3)])
    pa, pb = c.plan.new_replicas(), c.plan.new_replicas()
    sa = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    sb = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    mean = c.plan.new_state()
    coef_dev = torch.empty(1, dtype=torch.float32, device="cuda")
    for s, g in zip((1, 2, 3), grads):
        sums = orc.bucket_sumsq(c.sizes, c.wl.bucket_bytes, P, g)
        own, _ = orc.clip_coef(sums, adamw_own.max_norm)
        coef_dev.fill_(own)
        dps.dp_reduce_scatter_mean(c.plan, c.ws, c.to_replicas(g), mean, want_sumsq=True)
        dps.dp_clip_coef(c.plan, c.ws, adamw_ws.max_norm)
        dps.dp_sharded_adamw_step(c.plan, c.ws, mean, *sa, pa, dcfg(adamw_own, s),
                                  use_clip_coef=True, coef_dev=coef_dev)
        dps.dp_all_gather(c.plan, c.ws, pa)
        dps.dp_adamw_all_gather(c.plan, c.ws, mean, *sb, pb, dcfg(adamw_own, s),
                                use_clip_coef=True, coef_dev=coef_dev)
        _, ws_coef, status = dps.dp_read_norm(c.plan, c.ws)
        assert status == 0
        ost = ref[s - 1][4]
        assert own == ost.coef < ws_coef < 1.0          # both clip, differently
        check_state(c, pa, sa, ref[s - 1], exact=True)
        check_state(c, pb, sb, ref[s - 1], exact=True)


@pytest.mark.parametrize("P", [3, 8])
def test_chained_per_bucket_launches_match_oracle(orc, P):
    """Hundreds of tiny launches back to back, each reading what the launch just
    before it wrote (per bucket: reduce-scatter -> AdamW on its mean -> all-gather
    of its shard), with the mean stage and the parameter replicas filled with
    garbage before every step.  A kernel that read its input before its
    predecessor's writes were visible would leave garbage or the previous
    step's values behind; the result must equal the oracle's bit for bit."""
    rng = np.random.default_rng(11)
    sizes = [int(s) for s in rng.integers(1, 3000, size=160)]
    wl = small_workload(sizes, P, 8 * 1024, sigma=1e-3, seed=40 + P)
    c = Case(wl)
    assert c.plan.n_buckets >= 50
    adamw = configs.AdamW(max_norm=0.0)
    master0 = c.host_master()
    grads = [c.host_grads(s) for s in (1, 2)]
    ref = run_oracle_steps(orc, c, grads, master0, [ocfg(adamw, s) for s in (1, 2)])
    params = c.plan.new_replicas()
    st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    mean = c.plan.new_state()
    for s, g in zip((1, 2), grads):
        dev = c.to_replicas(g)
        mean.fill_(1.0e30)
        params.fill_(7.0)
        torch.cuda.synchronize()
        for b in reversed(range(c.plan.n_buckets)):      # the order backward fills them
            dps.dp_reduce_scatter_mean(c.plan, c.ws, dev, mean, b, b + 1)
            dps.dp_sharded_adamw_step(c.plan, c.ws, mean, *st, params, dcfg(adamw, s), b0=b, b1=b + 1)
            dps.dp_all_gather(c.plan, c.ws, params, b, b + 1)
        torch.cuda.synchronize()
        check_state(c, params, st, ref[s - 1], exact=True)


def test_per_bucket_allreduce_equals_single_launch():
    c = case_for("ragged", 8, cap=16 * 1024)
    assert c.plan.n_buckets > 3
    g = c.host_grads(1)
    a, b = c.to_replicas(g), c.to_replicas(g)
    dps.dp_allreduce_mean(c.plan, c.ws, a)
    for k in reversed(range(c.plan.n_buckets)):
        dps.dp_allreduce_mean(c.plan, c.ws, b, k, k + 1)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_plumbing_workload_three_steps(orc):
    """The 7-tensor, P=4, 1 MiB plumbing case: 3 fused steps with clip 1.0."""
    wl = configs.tiny_plumbing()
    c = Case(wl)
    assert c.plan.n_buckets == 3
    master0 = c.host_master()
    grads = [c.host_grads(s) for s in (1, 2, 3)]
    ref = run_oracle_steps(orc, c, grads, master0, [ocfg(wl.adamw, s) for s in (1, 2, 3)])
    params = c.plan.new_replicas()
    st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    for s, g in zip((1, 2, 3), grads):
        dps.dp_fused_zero_step(c.plan, c.ws, c.to_replicas(g), params, *st, dcfg(wl.adamw, s))
        norm, coef, _ = dps.dp_read_norm(c.plan, c.ws)
        ost = ref[s - 1][4]
        assert math.isclose(norm, ost.norm, rel_tol=1e-6)
        # ||mean|| ~ 0.5 < 1: no clipping, so both sides use coef = 1 exactly
        assert coef == ost.coef == 1.0
        check_state(c, params, st, ref[s - 1], exact=True)


def test_least_squares_identity_through_gpu(orc):
    """bf16(g_k) of the 4-rank least-squares split through the all-reduce: the
    GPU result equals the oracle's bit for bit and the exact full-batch mean."""
    from oracle_pins import lsq_data
    x, y, th = lsq_data()
    g_full, g_k, g_bar, _ = orc.lsq_identity(x, y, th, [16, 16, 16, 16])
    gk = torch.from_numpy(g_k.astype(np.float32)).to(torch.bfloat16)
    g16 = u16(gk)
    sizes = [16]
    wl = small_workload(sizes, 4, 1024)
    c = Case(wl)
    dev = c.to_replicas(g16)
    dps.dp_allreduce_mean(c.plan, c.ws, dev)
    torch.cuda.synchronize()
    want, mean, _ = orc.allreduce_mean(sizes, 1024, 4, g16)
    assert np.array_equal(c.from_replicas(dev), want)
    exact_mean = gk.float().double().mean(0).numpy()
    assert np.array_equal(mean.astype(np.float64), exact_mean)


def test_broadcast_from_rank0():
    c = case_for("ragged", 5)
    g = c.to_replicas(c.host_grads(1))
    dps.dp_broadcast(c.plan, c.ws, g, src=0)
    torch.cuda.synchronize()
    assert_replicas_equal(g, c.plan.L)
    dps.dp_broadcast(c.plan, c.ws, g, src=3, b0=1, b1=2)


def test_empty_plan_calls_succeed():
    c = Case(small_workload([], 4, 1024))
    buf = c.plan.new_replicas()
    st = [c.plan.new_state() for _ in range(3)]
    dps.dp_allreduce_mean(c.plan, c.ws, buf)
    dps.dp_fused_zero_step(c.plan, c.ws, buf, buf.clone(), *st, dps.adamw_cfg(max_norm=1.0))
    norm, coef, status = dps.dp_read_norm(c.plan, c.ws)
    assert (norm, coef, status) == (0.0, 1.0, 0)


def test_plan_mismatch_is_refused():
    """Whole-plan launches (the small kernels over several buckets check the plan
    before they read the workspace's tile table) store nothing when the workspace
    holds another plan's image."""
    a = case_for("ragged", 4)
    b = case_for("ragged", 4)
    g = a.to_replicas(a.host_grads(1))
    before = g.clone()
    mean = torch.full((b.plan.L,), 3.0, dtype=torch.float32, device="cuda")
    dps.dp_allreduce_mean(b.plan, a.ws, g)           # a's image, b's plan
    dps.dp_reduce_scatter_mean(b.plan, a.ws, g, mean)
    dps.dp_reduce_scatter_mean(b.plan, a.ws, g, mean, want_sumsq=True)
    with pytest.raises(dps.DPError) as e:
        dps.dp_read_norm(b.plan, a.ws)
    assert e.value.code == dps.DP_EPLAN
    assert torch.equal(g, before)
    assert bool((mean == 3.0).all())


@pytest.mark.parametrize("P", [4, 16])
def test_plan_mismatch_is_refused_by_small_per_bucket_launches(P):
    """Per-bucket launches over a few tiles (the kernels that check the plan beside
    their first loads) store nothing when the workspace holds another plan's
    image: all-reduce, reduce-scatter with and without norm partials."""
    a = case_for("ragged", P)
    b = case_for("ragged", P)
    assert b.plan.n_buckets >= 2
    g = a.to_replicas(a.host_grads(1))
    before = g.clone()
    mean = torch.full((b.plan.L,), 3.0, dtype=torch.float32, device="cuda")
    for k in range(b.plan.n_buckets):
        dps.dp_allreduce_mean(b.plan, a.ws, g, k, k + 1)
        dps.dp_reduce_scatter_mean(b.plan, a.ws, g, mean, k, k + 1)
        dps.dp_reduce_scatter_mean(b.plan, a.ws, g, mean, k, k + 1, want_sumsq=True)
    with pytest.raises(dps.DPError) as e:
        dps.dp_read_norm(b.plan, a.ws)
    assert e.value.code == dps.DP_EPLAN
    assert torch.equal(g, before)
    assert bool((mean == 3.0).all())


@pytest.mark.parametrize("P", [3, 8, 16])
def test_small_per_bucket_launches_equal_the_oracle(orc, P):
    """Per-bucket launches of small buckets (tile descriptors from the launch's
    parameters, the plan checked beside the loads, every replica block loaded at
    once): the all-reduce and the reduce-scatter with norm partials equal the
    oracle bit for bit, and the norm from per-bucket partials equals the one
    from a single launch."""
    c = case_for("ragged", P, cap=16 * 1024, sigma=0.05)
    assert c.plan.n_buckets >= 5
    g = c.host_grads(1)
    dev = c.to_replicas(g)
    mean = c.plan.new_state()
    for k in reversed(range(c.plan.n_buckets)):
        dps.dp_reduce_scatter_mean(c.plan, c.ws, dev, mean, k, k + 1, want_sumsq=True)
    dps.dp_clip_coef(c.plan, c.ws, 1.0)
    norm_pb, coef_pb, st = dps.dp_read_norm(c.plan, c.ws)
    want_ar, want_mean, _ = orc.allreduce_mean(c.sizes, c.wl.bucket_bytes, P, g)
    got = c.from_flat(mean)
    assert np.array_equal(got.view(np.uint32), want_mean.view(np.uint32))
    dps.dp_reduce_scatter_mean(c.plan, c.ws, dev, mean, want_sumsq=True)
    dps.dp_clip_coef(c.plan, c.ws, 1.0)
    assert dps.dp_read_norm(c.plan, c.ws)[:2] == (norm_pb, coef_pb)
    for k in range(c.plan.n_buckets):
        dps.dp_allreduce_mean(c.plan, c.ws, dev, k, k + 1)
    torch.cuda.synchronize()
    assert np.array_equal(c.from_replicas(dev), want_ar)
    assert_replicas_equal(dev, c.plan.L)


def test_nonfinite_gradient_is_reported(orc):
    c = case_for("zeros", 4)
    g = c.host_grads(1)
    g[2, 100] = 0x7F80                                  # +inf in rank 2
    adamw = configs.AdamW(max_norm=1.0)
    master0 = c.host_master()
    params = c.plan.new_replicas()
    st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    dps.dp_fused_zero_step(c.plan, c.ws, c.to_replicas(g), params, *st, dcfg(adamw, 1))
    with pytest.raises(dps.DPError) as e:
        dps.dp_read_norm(c.plan, c.ws)
    assert e.value.code == dps.DP_ENONFINITE
    _, coef, status = dps.dp_read_norm(c.plan, c.ws, raise_on_status=False)
    assert math.isnan(coef) and status & dps.DP_STATUS_NONFINITE
    ref = run_oracle_steps(orc, c, [g], master0, [ocfg(adamw, 1)])
    assert math.isnan(ref[0][4].coef)
    assert np.isnan(c.from_flat(st[0])).all() and np.isnan(ref[0][1]).all()


def test_stage_events_time_each_launch():
    c = case_for("ragged", 8)
    cfg = dps.adamw_cfg(max_norm=1.0)
    n = dps.dp_fused_zero_step_launches(cfg) + 1
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in ev:
        e.record()
    g = c.to_replicas(c.host_grads(1))
    st = [c.plan.new_state() for _ in range(3)]
    dps.dp_fused_zero_step(c.plan, c.ws, g, c.plan.new_replicas(), *st, cfg, events=ev)
    torch.cuda.synchronize()
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(n - 1)]
    assert all(t >= 0 for t in times)

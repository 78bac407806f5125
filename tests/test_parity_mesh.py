"""Hybrid R x S mesh on the GPU against the oracle's literal hierarchical rings:
all-reduce, fused ZeRO-2 (with and without clipping) and the staged path, bit for bit."""
import numpy as np
import pytest
import torch

import gradient_sync_zero_gb300 as dps
import oracle as oracle_mod
from harness import Case, assert_replicas_equal, small_workload, u16
from workloads import configs, device as wdev

pytestmark = pytest.mark.gpu

SIZES = [3, 1000, 65536, 13107, 26214, 4097, 27910]
MESHES = [(2, 4), (4, 2), (2, 2), (8, 1), (3, 2), (2, 3), (2, 8), (4, 4), (8, 2), (5, 2), (8, 8)]


def mesh_case(R, S, sigma=1e-3, cap=64 * 1024):
    wl = small_workload(SIZES, R * S, cap, sigma=sigma, seed=10 * R + S)
    c = Case.__new__(Case)
    c.wl, c.P, c.sizes, c.decay = wl, wl.P, wl.sizes, list(wl.decay)
    c.plan = dps.Plan(c.sizes, cap, c.P, c.decay, mesh=(R, S))
    c.off = c.plan.tensor_offsets()
    c.device = "cuda"
    c.ws = c.plan.new_workspace()
    return c


@pytest.mark.parametrize("R,S", MESHES)
def test_mesh_allreduce_matches_oracle(orc, R, S):
    c = mesh_case(R, S)
    g = c.host_grads(1)
    dev = c.to_replicas(g)
    dps.dp_allreduce_mean(c.plan, c.ws, dev)
    torch.cuda.synchronize()
    want, _, st = orc.mesh_allreduce_mean(c.sizes, c.wl.bucket_bytes, R, S, g)
    assert st.replicas_equal == 1
    assert np.array_equal(c.from_replicas(dev), want)
    assert_replicas_equal(dev, c.plan.L)


@pytest.mark.parametrize("R,S", [(2, 4), (4, 2), (3, 2), (2, 8), (4, 4), (8, 2)])
@pytest.mark.parametrize("max_norm", [0.0, 1.0])
def test_mesh_fused_zero_matches_oracle(orc, R, S, max_norm):
    c = mesh_case(R, S, sigma=0.05)
    adamw = configs.AdamW(max_norm=max_norm)
    master = c.host_master()
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    params = c.plan.new_replicas()
    st = [c.to_flat(master), c.plan.new_state(), c.plan.new_state()]
    for step in (1, 2):
        g = c.host_grads(step)
        cfg = dps.adamw_cfg(adamw.lr, adamw.beta1, adamw.beta2, adamw.eps, adamw.weight_decay,
                            adamw.max_norm, step)
        dps.dp_fused_zero_step(c.plan, c.ws, c.to_replicas(g), params, *st, cfg)
        p_o, master, m, v, so = orc.mesh_zero_step(c.sizes, c.decay, c.wl.bucket_bytes, R, S, g,
                                                   master, m, v, oracle_mod.adamw_cfg(adamw, step))
        assert so.groups_equal == 1 and so.replicas_equal == 1
        if max_norm > 0:
            norm, coef, _ = dps.dp_read_norm(c.plan, c.ws)
            assert coef == so.coef and so.coef < 1.0
        torch.cuda.synchronize()
        assert np.array_equal(c.from_replicas(params), p_o)
        for dev, ref in zip(st, (master, m, v)):
            assert np.array_equal(c.from_flat(dev).view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("R,S", [(2, 4), (3, 2)])
def test_mesh_staged_equals_fused(R, S):
    """reduce-scatter -> sharded AdamW (owners of shard s in every group) ->
    in-group all-gather == the fused step."""
    c = mesh_case(R, S)
    g = c.to_replicas(c.host_grads(1))
    master = c.host_master()
    cfg = dps.adamw_cfg(max_norm=0.0)
    p1, p2 = c.plan.new_replicas(), c.plan.new_replicas()
    s1 = [c.to_flat(master), c.plan.new_state(), c.plan.new_state()]
    s2 = [c.to_flat(master), c.plan.new_state(), c.plan.new_state()]
    dps.dp_fused_zero_step(c.plan, c.ws, g, p1, *s1, cfg)
    mean = c.plan.new_state()
    dps.dp_reduce_scatter_mean(c.plan, c.ws, g, mean)
    dps.dp_sharded_adamw_step(c.plan, c.ws, mean, *s2, p2, cfg)
    dps.dp_all_gather(c.plan, c.ws, p2)
    torch.cuda.synchronize()
    assert torch.equal(p1, p2)
    for a, b in zip(s1, s2):
        assert torch.equal(a, b)


@pytest.mark.parametrize("fused", [False, True], ids=["two-launches", "fused-backward"])
@pytest.mark.parametrize("R,S", [(2, 4), (4, 2), (3, 2)])
def test_hybrid_full_shard_unit_flow_matches_oracle(orc, R, S, fused):
    """HYBRID_SHARD proper: full sharding inside each group and data parallelism
    between groups ("4.1 Data parallelism in depth", sec. 6.3) — the ZeRO-3 unit
    flow on a mesh plan.  Each unit is gathered from the flat shard array, its
    gradients are reduce-scattered with the two-level fold, and each shard is
    updated; master/m/v and the shards equal the oracle's mesh step bit for bit
    (the update is elementwise, so where the parameters live does not change it)."""
    c = mesh_case(R, S, sigma=0.05)
    adamw = configs.AdamW(max_norm=1.0)
    master = c.host_master()
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    plan, nb, P = c.plan, c.plan.n_buckets, R * S
    shards = c.plan.new_state().to(torch.bfloat16)
    wdev.fill_flat(shards, c.off, c.sizes, torch.from_numpy(master).to(torch.bfloat16).cuda())
    st = [c.to_flat(master), c.plan.new_state(), c.plan.new_state()]
    mean = c.plan.new_state()
    unit_buf = torch.zeros(P, max(plan.bucket(b)[1] for b in range(nb)), dtype=torch.bfloat16,
                           device="cuda")
    bufs = [unit_buf, torch.zeros_like(unit_buf)]
    for step in (1, 2):
        g = c.host_grads(step)
        grads = c.to_replicas(g)
        cfg = dps.adamw_cfg(adamw.lr, adamw.beta1, adamw.beta2, adamw.eps, adamw.weight_decay,
                            adamw.max_norm, step)
        before = shards.clone()
        if fused:      # the next unit's gather beside this unit's reduce-scatter, one launch
            dps.dp_unit_all_gather(plan, c.ws, shards, 0, bufs[0])
        for b in range(nb):
            o, ln, _ = plan.bucket(b)
            if not fused:
                dps.dp_unit_all_gather(plan, c.ws, shards, b, unit_buf)
            torch.cuda.synchronize()
            for r in range(P):
                assert torch.equal(bufs[b % 2 if fused else 0][r, :ln], before[o:o + ln])
            if fused:
                dps.dp_unit_backward(plan, c.ws, shards, b + 1 if b + 1 < nb else -1,
                                     bufs[(b + 1) % 2], grads[:, o:o + ln], b, mean,
                                     want_sumsq=True)
            else:
                dps.dp_unit_reduce_scatter(plan, c.ws, grads[:, o:o + ln], b, mean, want_sumsq=True)
        dps.dp_clip_coef(plan, c.ws, adamw.max_norm)
        dps.dp_shard_adamw_step(plan, c.ws, mean, *st, shards, cfg, use_clip_coef=True)
        p_o, master, m, v, so = orc.mesh_zero_step(c.sizes, c.decay, c.wl.bucket_bytes, R, S, g,
                                                   master, m, v, oracle_mod.adamw_cfg(adamw, step))
        norm, coef, status = dps.dp_read_norm(plan, c.ws)
        assert status == 0 and coef == so.coef
        torch.cuda.synchronize()
        assert np.array_equal(u16(wdev.gather_flat(shards, c.off, c.sizes)), p_o[0])
        for dev, ref in zip(st, (master, m, v)):
            assert np.array_equal(c.from_flat(dev).view(np.uint32), ref.view(np.uint32))

"""Launch shape per stream (dp_stream_set_launch).  Every compute call enqueued on
a stream set to short-lived CTAs must give the bits it gives on a stream with the
default persistent grids, and the oracle's result where the oracle has one: the
shape changes only how many CTAs walk the tiles, never a tile's arithmetic."""
import numpy as np
import pytest
import torch

import gradient_sync_zero_gb300 as dps
import oracle as oracle_mod
from harness import Case, assert_replicas_equal, small_workload
from workloads import configs, device as wdev

pytestmark = pytest.mark.gpu

# one bucket of 310000 elements next to small ones, 64 KiB-ish caps: single- and
# multi-bucket launches, the small-launch kernels and the whole-tile ones
SIZES = [3, 1000, 65536, 13107, 26214, 4097, 27910, 9000, 700, 12000, 5, 310000]


def every_call(c, g, g2, master0, stream):
    """Each compute entry point once, on `stream`: {name: result}."""
    plan, ws, nb = c.plan, c.ws, c.plan.n_buckets
    a = configs.AdamW(max_norm=0.05)
    cfg_clip = dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, 1)
    cfg = dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, 0.0, 1)
    out = {}
    with torch.cuda.stream(stream):
        x = c.to_replicas(g)
        dps.dp_allreduce_mean(plan, ws, x)
        out["allreduce"] = x
        x = c.to_replicas(g)
        for b in reversed(range(nb)):
            dps.dp_allreduce_mean(plan, ws, x, b, b + 1)
        out["allreduce_per_bucket"] = x
        x = c.to_replicas(g)
        dps.dp_allreduce_mean_bf16wire(plan, ws, x)
        out["bf16wire"] = x
        mean = plan.new_state()
        dps.dp_reduce_scatter_mean(plan, ws, c.to_replicas(g), mean, want_sumsq=True)
        dps.dp_clip_coef(plan, ws, a.max_norm)
        out["rs"], out["rs_norm"] = mean, dps.dp_read_norm(plan, ws)
        mean_b, x = plan.new_state(), c.to_replicas(g)
        for b in reversed(range(nb)):
            dps.dp_reduce_scatter_mean(plan, ws, x, mean_b, b, b + 1, want_sumsq=True)
        dps.dp_clip_coef(plan, ws, a.max_norm)
        out["rs_per_bucket"], out["rs_per_bucket_norm"] = mean_b, dps.dp_read_norm(plan, ws)
        # the staged ZeRO step: AdamW on the owners' shards, then the all-gather
        st = [c.to_flat(master0), plan.new_state(), plan.new_state()]
        params = plan.new_replicas()
        dps.dp_sharded_adamw_step(plan, ws, mean, *st, params, cfg_clip, use_clip_coef=True)
        dps.dp_all_gather(plan, ws, params)
        out["staged_params"], out["staged_master"] = params, st[0]
        bc = params.clone()
        dps.dp_broadcast(plan, ws, bc, src=plan.P - 1)
        out["broadcast"] = bc
        for clip, name in ((cfg_clip, "fused_clip"), (cfg, "fused")):
            st = [c.to_flat(master0), plan.new_state(), plan.new_state()]
            params = plan.new_replicas()
            dps.dp_fused_zero_step(plan, ws, c.to_replicas(g), params, *st, clip)
            out[name + "_params"], out[name + "_state"] = params, st
            out[name + "_norm"] = dps.dp_read_norm(plan, ws)
        # accumulation
        acc, micro = c.to_replicas(g), c.to_replicas(g2)
        dps.dp_accumulate(plan, ws, acc, micro)
        out["accumulate"] = acc
        acc = c.to_replicas(g)
        dps.dp_allreduce_mean_accum(plan, ws, acc, micro)
        out["allreduce_accum"] = acc
        mean_a = plan.new_state()
        dps.dp_reduce_scatter_mean_accum(plan, ws, c.to_replicas(g), micro, mean_a, want_sumsq=True)
        out["rs_accum"] = mean_a
        # ZeRO-3 unit flow: forward gathers, fused backward, shard update
        shards = plan.new_state().to(torch.bfloat16)
        wdev.fill_flat(shards, c.off, c.sizes, torch.from_numpy(master0).to(torch.bfloat16).cuda())
        max_len = max(plan.bucket(b)[1] for b in range(nb))
        bufs = [torch.zeros(plan.P, max_len, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        gathered = []
        for b in reversed(range(nb)):
            dps.dp_unit_all_gather(plan, ws, shards, b, bufs[0])
            gathered.append(bufs[0][:, :plan.bucket(b)[1]].clone())
        grads, mean3 = c.to_replicas(g), plan.new_state()
        dps.dp_unit_all_gather(plan, ws, shards, 0, bufs[0])
        for b in range(nb):
            o, ln, _ = plan.bucket(b)
            gathered.append(bufs[b % 2][:, :ln].clone())
            dps.dp_unit_backward(plan, ws, shards, b + 1 if b + 1 < nb else -1, bufs[(b + 1) % 2],
                                 grads[:, o:o + ln], b, mean3, want_sumsq=True)
        mean4 = plan.new_state()
        for b in range(nb):
            o, ln, _ = plan.bucket(b)
            dps.dp_unit_reduce_scatter(plan, ws, grads[:, o:o + ln], b, mean4)
        dps.dp_clip_coef(plan, ws, a.max_norm)
        st = [c.to_flat(master0), plan.new_state(), plan.new_state()]
        dps.dp_shard_adamw_step(plan, ws, mean3, *st, shards, cfg_clip, use_clip_coef=True)
        out["unit_gathered"], out["unit_mean"], out["unit_mean_rs"] = gathered, mean3, mean4
        out["unit_shards"], out["unit_state"] = shards, st
        out["unit_norm"] = dps.dp_read_norm(plan, ws)
    stream.synchronize()
    return out


def same(x, y):
    """Bit equality of results (tensors, lists of them, plain values)."""
    if isinstance(x, (list, tuple)):
        return len(x) == len(y) and all(same(a, b) for a, b in zip(x, y))
    if isinstance(x, torch.Tensor):
        return x.dtype == y.dtype and torch.equal(x.contiguous().view(torch.uint8),
                                                  y.contiguous().view(torch.uint8))
    return x == y


@pytest.mark.parametrize("P", [8, 5])
def test_every_call_short_ctas_equals_persistent_and_oracle(orc, P):
    wl = small_workload(SIZES, P, 64 * 1024, sigma=0.05, seed=70 + P)
    c = Case(wl)
    assert c.plan.n_buckets >= 4
    g, g2, master0 = c.host_grads(1), c.host_grads(2), c.host_master()
    persistent = torch.cuda.Stream()
    short = torch.cuda.Stream(priority=0)
    dps.set_stream_launch(short, True)
    try:
        assert dps.stream_launch(short) and not dps.stream_launch(persistent)
        ref = every_call(c, g, g2, master0, persistent)
        got = every_call(c, g, g2, master0, short)
    finally:
        dps.set_stream_launch(short, False)
    assert ref.keys() == got.keys()
    for k in ref:
        assert same(ref[k], got[k]), k
    # and the oracle, for the paths it defines directly
    want, want_mean, _ = orc.allreduce_mean(c.sizes, wl.bucket_bytes, P, g)
    for k in ("allreduce", "allreduce_per_bucket"):
        assert np.array_equal(c.from_replicas(got[k]), want), k
        assert_replicas_equal(got[k], c.plan.L)
    for k in ("rs", "rs_per_bucket", "unit_mean", "unit_mean_rs"):
        assert np.array_equal(c.from_flat(got[k]).view(np.uint32), want_mean.view(np.uint32)), k
    a = configs.AdamW(max_norm=0.05)
    z = np.zeros_like(master0)
    p_o, m_o, mm_o, v_o, _, so = orc.zero_step(c.sizes, c.decay, wl.bucket_bytes, P, g, master0,
                                               z, z, oracle_mod.adamw_cfg(a, 1))
    assert got["fused_clip_norm"][1] == so.coef < 1.0
    assert np.array_equal(c.from_replicas(got["fused_clip_params"]), p_o)
    for dev, o in zip(got["fused_clip_state"], (m_o, mm_o, v_o)):
        assert np.array_equal(c.from_flat(dev).view(np.uint32), o.view(np.uint32))
    assert np.array_equal(c.from_replicas(got["staged_params"]), p_o)


def test_mesh_plan_short_ctas_equals_oracle(orc):
    """Hybrid 2 x 4 plan: the mesh all-reduce and the whole ZeRO step on a short-CTA
    stream equal the oracle's two-level ring."""
    P, R, S = 8, 2, 4
    wl = small_workload(SIZES, P, 64 * 1024, sigma=0.05, seed=81)
    c = Case(wl)
    c.plan = dps.Plan(wl.sizes, wl.bucket_bytes, P, c.decay, mesh=(R, S))
    c.off, c.ws = c.plan.tensor_offsets(), c.plan.new_workspace()
    g, master0 = c.host_grads(1), c.host_master()
    short = torch.cuda.Stream(priority=0)
    dps.set_stream_launch(short, True)
    try:
        with torch.cuda.stream(short):
            x = c.to_replicas(g)
            for b in reversed(range(c.plan.n_buckets)):
                dps.dp_allreduce_mean(c.plan, c.ws, x, b, b + 1)
            a = configs.AdamW(max_norm=0.0)
            cfg = dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, 0.0, 1)
            st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
            params = c.plan.new_replicas()
            dps.dp_fused_zero_step(c.plan, c.ws, c.to_replicas(g), params, *st, cfg)
        short.synchronize()
    finally:
        dps.set_stream_launch(short, False)
    want = orc.mesh_allreduce_mean(c.sizes, wl.bucket_bytes, R, S, g)
    want = want[0] if isinstance(want, tuple) else want
    assert np.array_equal(c.from_replicas(x), want)
    z = np.zeros_like(master0)
    p_o, m_o, mm_o, v_o, _ = orc.mesh_zero_step(c.sizes, c.decay, wl.bucket_bytes, R, S, g,
                                                master0, z, z, oracle_mod.adamw_cfg(a, 1))
    assert np.array_equal(c.from_replicas(params), p_o)
    for dev, o in zip(st, (m_o, mm_o, v_o)):
        assert np.array_equal(c.from_flat(dev).view(np.uint32), o.view(np.uint32))


def test_tracker_on_a_short_ctas_stream_fires_per_bucket(orc):
    """A tracker without DP_TRACK_SHORT_CTAS whose stream is set to short CTAs fires
    one launch per bucket, as with the flag, and equals the oracle."""
    P = 8
    wl = small_workload(SIZES, P, 64 * 1024, seed=82)
    c = Case(wl)
    g = c.host_grads(1)
    grads = c.to_replicas(g)
    comm = torch.cuda.Stream(priority=0)
    torch.cuda.synchronize()
    dps.set_stream_launch(comm, True)
    try:
        tr = dps.Tracker(c.plan, dps.DP_TRACK_ALLREDUCE, c.ws, grads, stream=comm)
        tr.begin()
        tr.mark_ready_range(0, len(SIZES))                  # every bucket ready at once
        tr.wait(10000)
        comm.synchronize()
        assert tr.stats()[0] == c.plan.n_buckets
    finally:
        dps.set_stream_launch(comm, False)
    want, _, _ = orc.allreduce_mean(c.sizes, wl.bucket_bytes, P, g)
    assert np.array_equal(c.from_replicas(grads), want)

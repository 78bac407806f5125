"""Streamed per-bucket synchronisation on the GPU: a producer stream writes each
tensor's gradients in backward order (last tensor first) and records an event;
the tracker fires each complete bucket on a separate communication stream.
Results must equal the single-launch path and the oracle, bit for bit."""
import numpy as np
import pytest
import torch

import gradient_sync_zero_gb300 as dps
from harness import Case, assert_replicas_equal, small_workload
from workloads import configs, device as wdev

pytestmark = pytest.mark.gpu


def produce(c, g_u16, grads, tracker, producer, n_ranks):
    """Backward-order producer: copy tensor t of every replica, then mark it ready."""
    src = torch.from_numpy(g_u16.view(np.int16)).view(torch.bfloat16).cuda()
    base = wdev.tensor_bases(c.sizes)
    events = []
    with torch.cuda.stream(producer):
        for t in reversed(range(len(c.sizes))):
            o, s = c.off[t], c.sizes[t]
            if s:
                grads[:n_ranks, o:o + s].copy_(src[:, base[t]:base[t] + s])
            ev = torch.cuda.Event()
            ev.record(producer)
            events.append(ev)
            tracker.mark_ready(t, ev)
    return events


@pytest.mark.parametrize("P,max_ctas", [(8, 0), (5, 16), (16, 4)])
def test_streamed_allreduce_equals_oracle(orc, P, max_ctas):
    wl = small_workload([3, 1000, 65536, 13107, 26214, 4097, 27910, 9000], P, 32 * 1024, seed=P)
    c = Case(wl)
    assert c.plan.n_buckets >= 3
    g = c.host_grads(1)
    grads = c.plan.new_replicas()
    comm, producer = torch.cuda.Stream(), torch.cuda.Stream()
    tr = dps.Tracker(c.plan, dps.DP_TRACK_ALLREDUCE, c.ws, grads, stream=comm, max_ctas=max_ctas)
    for step in range(2):                                   # the tracker is reused across steps
        grads.zero_()
        torch.cuda.synchronize()
        tr.begin()
        keep = produce(c, g, grads, tr, producer, P)
        tr.wait(10000)
        assert tr.fired() == list(range(c.plan.n_buckets))
        torch.cuda.synchronize()
        want, _, _ = orc.allreduce_mean(c.sizes, wl.bucket_bytes, P, g)
        assert np.array_equal(c.from_replicas(grads), want)
        assert_replicas_equal(grads, c.plan.L)
        del keep


@pytest.mark.parametrize("mode", ["allreduce", "zero_step"])
def test_range_marks_fire_bucket_ranges_that_equal_the_oracle(orc, mode):
    """A producer that marks several tensors with one event (dp_tracker_mark_ready_range,
    groups of three in backward order) completes several buckets per mark; each
    such group is one launch over the buckets' tiles, after one stream wait.  The
    result equals the oracle bit for bit, for the all-reduce and for the whole
    unclipped ZeRO step per range."""
    import oracle as oracle_mod
    P = 4
    sizes = [3, 1000, 65536, 13107, 26214, 4097, 27910, 9000, 700, 12000, 5, 31000]
    wl = small_workload(sizes, P, 16 * 1024, seed=90)
    c = Case(wl)
    g = c.host_grads(1)
    src = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).cuda()
    base = wdev.tensor_bases(c.sizes)
    grads = c.plan.new_replicas()
    comm, producer = torch.cuda.Stream(), torch.cuda.Stream()
    zero = mode == "zero_step"
    tr = dps.Tracker(c.plan, dps.DP_TRACK_ZERO_STEP if zero else dps.DP_TRACK_ALLREDUCE, c.ws,
                     grads, stream=comm)
    adamw = configs.AdamW(max_norm=0.0)
    if zero:
        master0 = c.host_master()
        params = c.plan.new_replicas()
        st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
        cfg = dps.adamw_cfg(adamw.lr, adamw.beta1, adamw.beta2, adamw.eps, adamw.weight_decay,
                            adamw.max_norm, 1)
        tr.set_zero_step(params, *st, cfg)
    groups = [(t0, min(t0 + 3, len(sizes))) for t0 in range(0, len(sizes), 3)]
    tr.begin()
    events = []
    with torch.cuda.stream(producer):
        for t0, t1 in reversed(groups):
            for t in reversed(range(t0, t1)):
                o, n = c.off[t], c.sizes[t]
                grads[:, o:o + n].copy_(src[:, base[t]:base[t] + n])
            ev = torch.cuda.Event()
            ev.record(producer)
            events.append(ev)
            tr.mark_ready_range(t0, t1, ev)
    tr.wait(10000)
    launches, waits = tr.stats()
    assert tr.fired() == list(range(c.plan.n_buckets))
    assert launches < c.plan.n_buckets            # some marks completed several buckets
    assert waits <= len(groups)
    torch.cuda.synchronize()
    if zero:
        z = np.zeros_like(master0)
        p_ref, m_ref, mm_ref, v_ref, _, _ = orc.zero_step(c.sizes, c.decay, wl.bucket_bytes, P, g,
                                                          master0, z, z,
                                                          oracle_mod.adamw_cfg(adamw, 1))
        assert np.array_equal(c.from_replicas(params), p_ref)
        for dev, ref in zip(st, (m_ref, mm_ref, v_ref)):
            assert np.array_equal(c.from_flat(dev).view(np.uint32), ref.view(np.uint32))
    else:
        want, _, _ = orc.allreduce_mean(c.sizes, wl.bucket_bytes, P, g)
        assert np.array_equal(c.from_replicas(grads), want)
        assert_replicas_equal(grads, c.plan.L)
    del events


@pytest.mark.parametrize("side", ["stream", "sm-partition"])
@pytest.mark.parametrize("mode", ["allreduce", "reduce_scatter", "zero_step"])
def test_side_stream_results_equal_the_oracle(orc, side, mode):
    """Every bucket but the last on a side stream (a plain stream, or one confined to
    an SM partition), the last on the tracker's stream after it: the results equal
    the oracle bit for bit, and everything is ordered before the tracker's stream."""
    import oracle as oracle_mod
    P = 8
    sizes = [3, 1000, 65536, 13107, 26214, 4097, 27910, 9000, 700, 12000, 5, 31000]
    wl = small_workload(sizes, P, 16 * 1024, seed=91, sigma=0.05)
    c = Case(wl)
    g = c.host_grads(1)
    src = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).cuda()
    base = wdev.tensor_bases(c.sizes)
    grads = c.plan.new_replicas()
    comm, producer = torch.cuda.Stream(), torch.cuda.Stream()
    if side == "sm-partition":
        try:
            sm = dps.SmStreams(8, with_rest=True)
        except dps.DPError as e:                       # a driver without green contexts
            pytest.skip(f"no SM-partition stream: {e}")
        assert sm.n_part >= 8 and sm.n_part + sm.n_rest <= torch.cuda.get_device_properties(0).multi_processor_count
        side_stream, cap, producer = sm.part, 2 * sm.n_part, sm.rest   # the producer on the rest
    else:
        side_stream, cap = torch.cuda.Stream(), 0
    kinds = {"allreduce": dps.DP_TRACK_ALLREDUCE, "reduce_scatter": dps.DP_TRACK_REDUCE_SCATTER,
             "zero_step": dps.DP_TRACK_ZERO_STEP}
    mean = c.plan.new_state()
    tr = dps.Tracker(c.plan, kinds[mode], c.ws, grads, mean, stream=comm)
    tr.set_side_stream(side_stream, cap)
    adamw = configs.AdamW(max_norm=0.0)
    master0 = c.host_master()
    if mode == "zero_step":
        params = c.plan.new_replicas()
        st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
        tr.set_zero_step(params, *st, dps.adamw_cfg(adamw.lr, adamw.beta1, adamw.beta2, adamw.eps,
                                                    adamw.weight_decay, 0.0, 1))
    tr.begin()
    events = []
    with torch.cuda.stream(producer):
        for t in reversed(range(len(sizes))):
            o, n = c.off[t], c.sizes[t]
            grads[:, o:o + n].copy_(src[:, base[t]:base[t] + n])
            ev = torch.cuda.Event()
            ev.record(producer)
            events.append(ev)
            tr.mark_ready(t, ev)
    tr.wait(10000)
    assert tr.fired() == list(range(c.plan.n_buckets))
    comm.synchronize()                                 # the tracker's stream alone orders it all
    if mode == "allreduce":
        want, _, _ = orc.allreduce_mean(c.sizes, wl.bucket_bytes, P, g)
        assert np.array_equal(c.from_replicas(grads), want)
    elif mode == "reduce_scatter":
        _, want_mean, _ = orc.allreduce_mean(c.sizes, wl.bucket_bytes, P, g)
        assert np.array_equal(c.from_flat(mean).view(np.uint32), want_mean.view(np.uint32))
        dps.dp_clip_coef(c.plan, c.ws, 1.0, stream=comm)
        norm, _, _ = dps.dp_read_norm(c.plan, c.ws, stream=comm)
        _, onorm = orc.clip_coef(orc.bucket_sumsq(c.sizes, wl.bucket_bytes, P, g), 1.0)
        assert abs(norm - onorm) <= 1e-10 * onorm
    else:
        z = np.zeros_like(master0)
        p_ref, m_ref, mm_ref, v_ref, _, _ = orc.zero_step(c.sizes, c.decay, wl.bucket_bytes, P, g,
                                                          master0, z, z,
                                                          oracle_mod.adamw_cfg(adamw, 1))
        assert np.array_equal(c.from_replicas(params), p_ref)
        for dev, ref in zip(st, (m_ref, mm_ref, v_ref)):
            assert np.array_equal(c.from_flat(dev).view(np.uint32), ref.view(np.uint32))
    del events
    tr.set_side_stream(None)
    if side == "sm-partition":
        sm.close()


def test_streamed_mesh_allreduce_equals_oracle(orc):
    """The tracker on a hybrid 2 x 4 plan fires the mesh all-reduce bucket by bucket."""
    P, R, S = 8, 2, 4
    wl = small_workload([3, 1000, 65536, 13107, 26214, 4097, 27910, 9000], P, 32 * 1024, seed=77)
    plan = dps.Plan(wl.sizes, wl.bucket_bytes, P, mesh=(R, S))
    c = Case(wl)
    c.plan, c.off, c.ws = plan, plan.tensor_offsets(), plan.new_workspace()
    g = c.host_grads(1)
    grads = plan.new_replicas()
    comm, producer = torch.cuda.Stream(), torch.cuda.Stream()
    tr = dps.Tracker(plan, dps.DP_TRACK_ALLREDUCE, c.ws, grads, stream=comm)
    tr.begin()
    keep = produce(c, g, grads, tr, producer, P)
    tr.wait(10000)
    assert tr.fired() == list(range(plan.n_buckets))
    torch.cuda.synchronize()
    want = orc.mesh_allreduce_mean(c.sizes, wl.bucket_bytes, R, S, g)
    want = want[0] if isinstance(want, tuple) else want
    assert np.array_equal(c.from_replicas(grads), want)
    assert_replicas_equal(grads, plan.L)
    del keep


def test_streamed_zero_step_equals_fused(orc):
    """Tracker reduce-scatters bucket by bucket; then the clip coefficient and the
    fused AdamW + all-gather on the same stream == dp_fused_zero_step."""
    wl = configs.tiny_plumbing()
    wl.adamw = configs.AdamW(max_norm=0.3)                 # clip active
    c = Case(wl)
    g = c.host_grads(1)
    master0 = c.host_master()
    a = wl.adamw
    cfg = dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, 1)
    # reference: one fused call
    p_ref = c.plan.new_replicas()
    s_ref = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    dps.dp_fused_zero_step(c.plan, c.ws, c.to_replicas(g), p_ref, *s_ref, cfg)
    n_ref = dps.dp_read_norm(c.plan, c.ws)
    # streamed
    ws2 = c.plan.new_workspace()
    grads, mean = c.plan.new_replicas(), c.plan.new_state()
    params = c.plan.new_replicas()
    st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    comm, producer = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    tr = dps.Tracker(c.plan, dps.DP_TRACK_REDUCE_SCATTER, ws2, grads, mean, stream=comm)
    tr.begin()
    keep = produce(c, g, grads, tr, producer, wl.P)
    tr.wait(10000)
    dps.dp_clip_coef(c.plan, ws2, a.max_norm, stream=comm)
    dps.dp_adamw_all_gather(c.plan, ws2, mean, *st, params, cfg, use_clip_coef=True, stream=comm)
    n2 = dps.dp_read_norm(c.plan, ws2, stream=comm)
    assert n2 == n_ref and n_ref[1] < 1.0
    assert torch.equal(params, p_ref)
    for x, y in zip(st, s_ref):
        assert torch.equal(x, y)
    del keep
    # and the oracle agrees
    z = np.zeros_like(master0)
    import oracle
    p_o, m_o, _, _, _, sto = orc.zero_step(c.sizes, c.decay, wl.bucket_bytes, wl.P, g, master0, z,
                                           z, oracle.adamw_cfg(a, 1))
    assert sto.coef == n2[1]
    assert np.array_equal(c.from_replicas(params), p_o)
    assert np.array_equal(c.from_flat(st[0]).view(np.uint32), m_o.view(np.uint32))


@pytest.mark.parametrize("short_ctas", [False, True], ids=["persistent", "short-ctas"])
@pytest.mark.parametrize("mode", [dps.DP_TRACK_ALLREDUCE, dps.DP_TRACK_REDUCE_SCATTER])
def test_streamed_last_micro_batch_equals_fused_single_launch(mode, short_ctas):
    """Accumulation: grads holds the earlier micro-batches' sum; the last micro-batch's
    gradients arrive tensor by tensor in backward order into `micro`, and each bucket
    fires the fused add + sync (persistent grids, or short-lived CTAs).  Equal, bit for
    bit, to one fused launch."""
    P = 8
    wl = small_workload([3, 1000, 65536, 13107, 26214, 4097, 27910, 9000], P, 32 * 1024, seed=91)
    c = Case(wl)
    acc0 = c.to_replicas(c.host_grads(1))
    g_last = c.host_grads(2)
    # reference: one fused launch over all buckets
    ref = acc0.clone()
    mean_ref = c.plan.new_state()
    if mode == dps.DP_TRACK_ALLREDUCE:
        dps.dp_allreduce_mean_accum(c.plan, c.ws, ref, c.to_replicas(g_last))
    else:
        dps.dp_reduce_scatter_mean_accum(c.plan, c.ws, ref, c.to_replicas(g_last), mean_ref,
                                         want_sumsq=True)
        dps.dp_clip_coef(c.plan, c.ws, 1.0)
    n_ref = dps.dp_read_norm(c.plan, c.ws)
    # streamed
    ws2 = c.plan.new_workspace()
    acc = acc0.clone()
    micro = c.plan.new_replicas()
    mean = c.plan.new_state()
    comm, producer = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    tr = dps.Tracker(c.plan, mode, ws2, acc, mean if mode == dps.DP_TRACK_REDUCE_SCATTER else None,
                     stream=comm, short_ctas=short_ctas)
    tr.set_micro(micro)
    tr.begin()
    keep = produce(c, g_last, micro, tr, producer, P)
    tr.wait(10000)
    if mode == dps.DP_TRACK_REDUCE_SCATTER:
        dps.dp_clip_coef(c.plan, ws2, 1.0, stream=comm)
    n2 = dps.dp_read_norm(c.plan, ws2, stream=comm)
    torch.cuda.synchronize()
    if mode == dps.DP_TRACK_ALLREDUCE:
        assert torch.equal(acc, ref)
    else:
        assert torch.equal(mean.view(torch.int32), mean_ref.view(torch.int32)) and n2 == n_ref
    del keep


@pytest.mark.parametrize("P,mesh,max_ctas", [(8, None, 0), (5, None, 16), (8, (2, 4), 0)])
def test_streamed_whole_zero_step_per_bucket_matches_oracle(orc, P, mesh, max_ctas):
    """DP_TRACK_ZERO_STEP: each bucket's whole unclipped ZeRO step (reduce-scatter,
    AdamW on the owners' shards, all-gather) fires as soon as the bucket is ready,
    while the producer is still writing earlier tensors.  Three steps through one
    tracker (the AdamW settings change with t); master/m/v and every replica equal
    the oracle's ZeRO step bit for bit."""
    import oracle as oracle_mod
    wl = small_workload([3, 1000, 65536, 13107, 26214, 4097, 27910, 9000], P, 32 * 1024,
                        sigma=0.05, seed=90 + P)
    c = Case(wl)
    if mesh:
        c.plan = dps.Plan(wl.sizes, wl.bucket_bytes, P, c.decay, mesh=mesh)
        c.off, c.ws = c.plan.tensor_offsets(), c.plan.new_workspace()
    assert c.plan.n_buckets >= 3
    adamw = configs.AdamW(max_norm=0.0)
    master = c.host_master()
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    grads, params = c.plan.new_replicas(), c.plan.new_replicas()
    st = [c.to_flat(master), c.plan.new_state(), c.plan.new_state()]
    comm, producer = torch.cuda.Stream(), torch.cuda.Stream()
    tr = dps.Tracker(c.plan, dps.DP_TRACK_ZERO_STEP, c.ws, grads, stream=comm, max_ctas=max_ctas)
    for step in (1, 2, 3):
        g = c.host_grads(step)
        ocfg = oracle_mod.adamw_cfg(adamw, step)
        if mesh:
            p_o, master, m, v, _ = orc.mesh_zero_step(c.sizes, c.decay, wl.bucket_bytes, *mesh, g,
                                                      master, m, v, ocfg)
        else:
            p_o, master, m, v, _, _ = orc.zero_step(c.sizes, c.decay, wl.bucket_bytes, P, g,
                                                    master, m, v, ocfg)
        cfg = dps.adamw_cfg(adamw.lr, adamw.beta1, adamw.beta2, adamw.eps, adamw.weight_decay,
                            0.0, step)
        grads.zero_()
        torch.cuda.synchronize()
        tr.set_zero_step(params, *st, cfg)
        tr.begin()
        keep = produce(c, g, grads, tr, producer, P)
        tr.wait(10000)
        assert tr.fired() == list(range(c.plan.n_buckets))
        torch.cuda.synchronize()
        assert np.array_equal(c.from_replicas(params), p_o)
        assert_replicas_equal(params, c.plan.L)
        for dev, ref in zip(st, (master, m, v)):
            assert np.array_equal(c.from_flat(dev).view(np.uint32), ref.view(np.uint32))
        del keep


def priority_streams():
    """The communication stream at the lowest priority, the producer at the highest
    (out-of-range priorities are clamped to the device's range)."""
    return torch.cuda.Stream(priority=0), torch.cuda.Stream(priority=-16)


@pytest.mark.parametrize("mode,mesh,marks", [
    ("allreduce", None, "tensor"), ("allreduce", None, "range"), ("allreduce", (2, 4), "tensor"),
    ("reduce_scatter", None, "tensor"), ("reduce_scatter", None, "range"),
    ("zero_step", None, "range"), ("zero_step", (2, 4), "tensor")])
def test_short_ctas_results_equal_the_oracle(orc, mode, mesh, marks):
    """DP_TRACK_SHORT_CTAS: every bucket is its own launch of short-lived CTAs (one
    per piece of a tile), the communication stream at the lowest priority and the
    producer above it.  The results equal the oracle bit for bit (the norm to
    1e-10), and range marks that complete several buckets at once still launch
    once per bucket."""
    import oracle as oracle_mod
    P = 8
    sizes = [3, 1000, 65536, 13107, 26214, 4097, 27910, 9000, 700, 12000, 5, 31000]
    wl = small_workload(sizes, P, 16 * 1024, seed=92, sigma=0.05)
    c = Case(wl)
    if mesh:
        c.plan = dps.Plan(wl.sizes, wl.bucket_bytes, P, c.decay, mesh=mesh)
        c.off, c.ws = c.plan.tensor_offsets(), c.plan.new_workspace()
    nb = c.plan.n_buckets
    g = c.host_grads(1)
    src = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).cuda()
    base = wdev.tensor_bases(c.sizes)
    grads, mean = c.plan.new_replicas(), c.plan.new_state()
    comm, producer = priority_streams()
    kinds = {"allreduce": dps.DP_TRACK_ALLREDUCE, "reduce_scatter": dps.DP_TRACK_REDUCE_SCATTER,
             "zero_step": dps.DP_TRACK_ZERO_STEP}
    tr = dps.Tracker(c.plan, kinds[mode], c.ws, grads, mean, stream=comm, max_ctas=4,
                     short_ctas=True)
    adamw = configs.AdamW(max_norm=0.0)
    master0 = c.host_master()
    if mode == "zero_step":
        params = c.plan.new_replicas()
        st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
        tr.set_zero_step(params, *st, dps.adamw_cfg(adamw.lr, adamw.beta1, adamw.beta2, adamw.eps,
                                                    adamw.weight_decay, 0.0, 1))
    groups = ([(t, t + 1) for t in range(len(sizes))] if marks == "tensor" else
              [(t0, min(t0 + 3, len(sizes))) for t0 in range(0, len(sizes), 3)])
    tr.begin()
    events = []
    with torch.cuda.stream(producer):
        for t0, t1 in reversed(groups):
            for t in reversed(range(t0, t1)):
                o, n = c.off[t], c.sizes[t]
                grads[:, o:o + n].copy_(src[:, base[t]:base[t] + n])
            ev = torch.cuda.Event()
            ev.record(producer)
            events.append(ev)
            tr.mark_ready_range(t0, t1, ev)
    tr.wait(10000)
    assert tr.fired() == list(range(nb))
    assert tr.stats()[0] == nb                       # one launch per bucket
    comm.synchronize()
    if mode == "allreduce":
        if mesh:
            want = orc.mesh_allreduce_mean(c.sizes, wl.bucket_bytes, *mesh, g)
            want = want[0] if isinstance(want, tuple) else want
        else:
            want, _, _ = orc.allreduce_mean(c.sizes, wl.bucket_bytes, P, g)
        assert np.array_equal(c.from_replicas(grads), want)
        assert_replicas_equal(grads, c.plan.L)
    elif mode == "reduce_scatter":
        _, want_mean, _ = orc.allreduce_mean(c.sizes, wl.bucket_bytes, P, g)
        assert np.array_equal(c.from_flat(mean).view(np.uint32), want_mean.view(np.uint32))
        dps.dp_clip_coef(c.plan, c.ws, 1.0, stream=comm)
        norm, _, status = dps.dp_read_norm(c.plan, c.ws, stream=comm)
        _, onorm = orc.clip_coef(orc.bucket_sumsq(c.sizes, wl.bucket_bytes, P, g), 1.0)
        assert status == 0 and abs(norm - onorm) <= 1e-10 * onorm
    else:
        z = np.zeros_like(master0)
        ocfg = oracle_mod.adamw_cfg(adamw, 1)
        if mesh:
            p_ref, m_ref, mm_ref, v_ref, _ = orc.mesh_zero_step(c.sizes, c.decay, wl.bucket_bytes,
                                                                *mesh, g, master0, z, z, ocfg)
        else:
            p_ref, m_ref, mm_ref, v_ref, _, _ = orc.zero_step(c.sizes, c.decay, wl.bucket_bytes, P,
                                                              g, master0, z, z, ocfg)
        assert np.array_equal(c.from_replicas(params), p_ref)
        for dev, ref in zip(st, (m_ref, mm_ref, v_ref)):
            assert np.array_equal(c.from_flat(dev).view(np.uint32), ref.view(np.uint32))
    del events


def test_short_ctas_bucket_larger_than_the_gpu_holds_at_once(orc):
    """A bucket whose short CTAs (64 threads, eight per 16384-element tile) are more
    than twice what the GPU can hold at once (32 CTAs per SM at most): the
    all-reduce and the reduce-scatter with its norm partials still equal the oracle
    bit for bit."""
    P = 8
    sizes = [3, 24_000_003, 70000]
    wl = small_workload(sizes, P, 32 << 20, seed=93, sigma=0.05)
    c = Case(wl)
    big = max(range(c.plan.n_buckets), key=lambda b: c.plan.bucket(b)[1])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert c.plan.bucket(big)[1] // 16384 * 8 > 2 * 32 * sms
    g = c.host_grads(1)
    want, want_mean, _ = orc.allreduce_mean(c.sizes, wl.bucket_bytes, P, g)
    for kind in (dps.DP_TRACK_REDUCE_SCATTER, dps.DP_TRACK_ALLREDUCE):
        grads, mean = c.to_replicas(g), c.plan.new_state()
        comm, _ = priority_streams()
        torch.cuda.synchronize()
        tr = dps.Tracker(c.plan, kind, c.ws, grads, mean, stream=comm, short_ctas=True)
        tr.begin()
        tr.mark_ready_range(0, len(sizes))
        tr.wait(10000)
        comm.synchronize()
        if kind == dps.DP_TRACK_ALLREDUCE:
            assert np.array_equal(c.from_replicas(grads), want)
        else:
            assert np.array_equal(c.from_flat(mean).view(np.uint32), want_mean.view(np.uint32))
            dps.dp_clip_coef(c.plan, c.ws, 1.0, stream=comm)
            norm, _, status = dps.dp_read_norm(c.plan, c.ws, stream=comm)
            _, onorm = orc.clip_coef(orc.bucket_sumsq(c.sizes, wl.bucket_bytes, P, g), 1.0)
            assert status == 0 and abs(norm - onorm) <= 1e-10 * onorm
        del tr

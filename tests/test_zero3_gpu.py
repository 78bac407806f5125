"""ZeRO-3 / FULL_SHARD unit flow on the GPU against the oracle: forward all-gather
of every unit, backward all-gather, reduce-scatter of the unit's gradients, then the
shard update — bit for bit, for a flat plan and a hybrid mesh's flat sibling."""
import numpy as np
import pytest
import torch

import gradient_sync_zero_gb300 as dps
import oracle as oracle_mod
from harness import Case, small_workload, u16
from workloads import configs, device as wdev

pytestmark = pytest.mark.gpu


def zero3_flow(c, grads, shards, mean, st, cfg, unit_buf, coef_dev=None, ws_max_norm=None,
               unit_buf2=None):
    """coef_dev: the update multiplies by the caller's own coefficient instead of
    the workspace's (which dp_clip_coef still forms, at ws_max_norm).  unit_buf2:
    the backward runs as dp_unit_backward launches, each gathering the next unit
    into the other buffer while the current unit's gradients reduce-scatter."""
    plan = c.plan
    nb = plan.n_buckets
    gathered = []
    for b in reversed(range(nb)):                           # forward
        dps.dp_unit_all_gather(plan, c.ws, shards, b, unit_buf)
        o, ln, _ = plan.bucket(b)
        gathered.append((b, unit_buf[:, :ln].clone()))
    if unit_buf2 is not None:                               # backward, fused launches
        bufs = [unit_buf, unit_buf2]
        dps.dp_unit_all_gather(plan, c.ws, shards, 0, bufs[0])
        for b in range(nb):
            o, ln, _ = plan.bucket(b)
            gathered.append((b, bufs[b % 2][:, :ln].clone()))   # unit b's backward reads it
            nxt = b + 1 if b + 1 < nb else -1
            dps.dp_unit_backward(plan, c.ws, shards, nxt, bufs[(b + 1) % 2], grads[:, o:o + ln], b,
                                 mean, want_sumsq=True)
    for b in range(nb if unit_buf2 is None else 0):         # backward
        dps.dp_unit_all_gather(plan, c.ws, shards, b, unit_buf)
        o, ln, _ = plan.bucket(b)
        dps.dp_unit_reduce_scatter(plan, c.ws, grads[:, o:o + ln], b, mean, want_sumsq=True)
    dps.dp_clip_coef(plan, c.ws, cfg.max_norm if ws_max_norm is None else ws_max_norm)
    dps.dp_shard_adamw_step(plan, c.ws, mean, *st, shards, cfg, use_clip_coef=True,
                            coef_dev=coef_dev)
    return gathered


@pytest.mark.parametrize("fused", [False, True], ids=["two-launches", "fused-backward"])
@pytest.mark.parametrize("P", [2, 4, 5, 8, 12, 16])
def test_zero3_flow_matches_oracle(orc, P, fused):
    wl = small_workload([3, 1000, 65536, 13107, 26214, 4097, 27910], P, 64 * 1024, sigma=0.05,
                        seed=30 + P)
    c = Case(wl)
    adamw = configs.AdamW(max_norm=1.0)
    master = c.host_master()
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    shards_h = u16(torch.from_numpy(master).to(torch.bfloat16))
    shards = c.plan.new_state().to(torch.bfloat16)
    wdev.fill_flat(shards, c.off, c.sizes, torch.from_numpy(master).to(torch.bfloat16).cuda())
    st = [c.to_flat(master), c.plan.new_state(), c.plan.new_state()]
    mean = c.plan.new_state()
    max_len = max(c.plan.bucket(b)[1] for b in range(c.plan.n_buckets))
    unit_buf = torch.zeros(P, max_len, dtype=torch.bfloat16, device="cuda")
    unit_buf2 = torch.zeros_like(unit_buf) if fused else None
    for step in (1, 2):
        g = c.host_grads(step)
        cfg = dps.adamw_cfg(adamw.lr, adamw.beta1, adamw.beta2, adamw.eps, adamw.weight_decay,
                            adamw.max_norm, step)
        before = shards.clone()
        gathered = zero3_flow(c, c.to_replicas(g), shards, mean, st, cfg, unit_buf,
                              unit_buf2=unit_buf2)
        shards_h, master, m, v, so = orc.zero3_step(c.sizes, c.decay, wl.bucket_bytes, P, g,
                                                    shards_h, master, m, v,
                                                    oracle_mod.adamw_cfg(adamw, step))
        assert so.gathered_ok == 1 and so.coef < 1.0
        norm, coef, status = dps.dp_read_norm(c.plan, c.ws)
        assert status == 0 and coef == so.coef
        torch.cuda.synchronize()
        for b, copy in gathered:                             # every rank gathered the unit
            o, ln, _ = c.plan.bucket(b)
            for r in range(P):
                assert torch.equal(copy[r], before[o:o + ln])
        assert np.array_equal(u16(wdev.gather_flat(shards, c.off, c.sizes)), shards_h)
        for dev, ref in zip(st, (master, m, v)):
            assert np.array_equal(c.from_flat(dev).view(np.uint32), ref.view(np.uint32))


def test_zero3_shard_update_with_caller_coefficient(orc):
    """dp_shard_adamw_step given the caller's coefficient (the oracle's at
    max_norm 0.3) while the workspace holds the one for max_norm 1.0: the shards
    and state equal the oracle's ZeRO-3 step at max_norm 0.3, bit for bit."""
    P = 4
    wl = small_workload([3, 1000, 65536, 13107, 26214, 4097, 27910], P, 64 * 1024, sigma=0.05,
                        seed=34)
    c = Case(wl)
    own = configs.AdamW(max_norm=0.3)
    master = c.host_master()
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    shards_h = u16(torch.from_numpy(master).to(torch.bfloat16))
    shards = c.plan.new_state().to(torch.bfloat16)
    wdev.fill_flat(shards, c.off, c.sizes, torch.from_numpy(master).to(torch.bfloat16).cuda())
    st = [c.to_flat(master), c.plan.new_state(), c.plan.new_state()]
    mean = c.plan.new_state()
    max_len = max(c.plan.bucket(b)[1] for b in range(c.plan.n_buckets))
    unit_buf = torch.zeros(P, max_len, dtype=torch.bfloat16, device="cuda")
    coef_dev = torch.empty(1, dtype=torch.float32, device="cuda")
    for step in (1, 2):
        g = c.host_grads(step)
        coef, _ = orc.clip_coef(orc.bucket_sumsq(c.sizes, wl.bucket_bytes, P, g), own.max_norm)
        coef_dev.fill_(coef)
        cfg = dps.adamw_cfg(own.lr, own.beta1, own.beta2, own.eps, own.weight_decay,
                            own.max_norm, step)
        zero3_flow(c, c.to_replicas(g), shards, mean, st, cfg, unit_buf, coef_dev=coef_dev,
                   ws_max_norm=1.0)
        shards_h, master, m, v, so = orc.zero3_step(c.sizes, c.decay, wl.bucket_bytes, P, g,
                                                    shards_h, master, m, v,
                                                    oracle_mod.adamw_cfg(own, step))
        _, ws_coef, status = dps.dp_read_norm(c.plan, c.ws)
        assert status == 0 and so.coef == coef < ws_coef < 1.0
        got = u16(wdev.gather_flat(shards, c.off, c.sizes))
        assert np.array_equal(got, shards_h)
        for name, dev, ref in (("master", st[0], master), ("m", st[1], m), ("v", st[2], v)):
            a = c.from_flat(dev)
            assert np.array_equal(a.view(np.uint32), ref.view(np.uint32)), name


@pytest.mark.parametrize("fused", [False, True], ids=["two-launches", "fused-backward"])
def test_zero3_flow_with_an_empty_unit(orc, fused):
    """A plan whose last unit is empty (zero-size tensors after an oversized one):
    the unit calls, the fused backward included, launch nothing for it and the flow
    still equals the oracle bit for bit."""
    P = 4
    sizes = [0, 0, 100, 3000]
    wl = small_workload(sizes, P, 64, sigma=0.05, seed=5)
    c = Case(wl)
    assert [c.plan.bucket(b)[1] for b in range(c.plan.n_buckets)][-1] == 0
    adamw = configs.AdamW(max_norm=1.0)
    master = c.host_master()
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    shards_h = u16(torch.from_numpy(master).to(torch.bfloat16))
    shards = c.plan.new_state().to(torch.bfloat16)
    wdev.fill_flat(shards, c.off, c.sizes, torch.from_numpy(master).to(torch.bfloat16).cuda())
    st = [c.to_flat(master), c.plan.new_state(), c.plan.new_state()]
    mean = c.plan.new_state()
    max_len = max(c.plan.bucket(b)[1] for b in range(c.plan.n_buckets))
    unit_buf = torch.zeros(P, max_len, dtype=torch.bfloat16, device="cuda")
    g = c.host_grads(1)
    cfg = dps.adamw_cfg(adamw.lr, adamw.beta1, adamw.beta2, adamw.eps, adamw.weight_decay,
                        adamw.max_norm, 1)
    zero3_flow(c, c.to_replicas(g), shards, mean, st, cfg, unit_buf,
               unit_buf2=torch.zeros_like(unit_buf) if fused else None)
    shards_h, master, m, v, so = orc.zero3_step(c.sizes, c.decay, wl.bucket_bytes, P, g, shards_h,
                                                master, m, v, oracle_mod.adamw_cfg(adamw, 1))
    norm, coef, status = dps.dp_read_norm(c.plan, c.ws)
    assert status == 0 and coef == so.coef
    assert np.array_equal(u16(wdev.gather_flat(shards, c.off, c.sizes)), shards_h)
    for dev, ref in zip(st, (master, m, v)):
        assert np.array_equal(c.from_flat(dev).view(np.uint32), ref.view(np.uint32))


def test_unit_all_gather_fills_every_rank_row():
    wl = small_workload([3, 1000, 65536, 4097], 4, 64 * 1024, seed=3)
    c = Case(wl)
    vals = torch.arange(c.plan.L, dtype=torch.float32, device="cuda").to(torch.bfloat16)
    max_len = max(c.plan.bucket(b)[1] for b in range(c.plan.n_buckets))
    buf = torch.zeros(4, max_len + 64, dtype=torch.bfloat16, device="cuda")
    for b in range(c.plan.n_buckets):
        o, ln, _ = c.plan.bucket(b)
        dps.dp_unit_all_gather(c.plan, c.ws, vals, b, buf)
        torch.cuda.synchronize()
        for r in range(4):
            assert torch.equal(buf[r, :ln], vals[o:o + ln])


def test_unit_reduce_scatter_equals_bucket_reduce_scatter():
    wl = small_workload([3, 1000, 65536, 13107, 26214], 8, 32 * 1024, seed=4)
    c = Case(wl)
    g = c.to_replicas(c.host_grads(1))
    a, b_ = c.plan.new_state(), c.plan.new_state()
    dps.dp_reduce_scatter_mean(c.plan, c.ws, g, a, want_sumsq=True)
    dps.dp_clip_coef(c.plan, c.ws, 1.0)
    n1 = dps.dp_read_norm(c.plan, c.ws)
    for b in range(c.plan.n_buckets):
        o, ln, _ = c.plan.bucket(b)
        unit = g[:, o:o + ln].contiguous()                  # a separate [P][len] buffer
        dps.dp_unit_reduce_scatter(c.plan, c.ws, unit, b, b_, want_sumsq=True)
    dps.dp_clip_coef(c.plan, c.ws, 1.0)
    n2 = dps.dp_read_norm(c.plan, c.ws)
    assert torch.equal(a, b_) and n1 == n2


def test_prefetch_schedule_on_two_streams_equals_sequential():
    """The FSDP-style prefetch schedule — the next unit's gather on one stream while
    the current unit's gradients reduce-scatter on another, two unit buffers —
    shares the workspace between concurrent launches and must give the sequential
    flow's mean, norm, state and gathered units bit for bit."""
    wl = configs.llama_1b1_zero2(layers=2, embeddings=False)
    wl.bucket_bytes = 4 << 20                                 # many units
    c = Case(wl)
    plan, nb, P = c.plan, c.plan.n_buckets, wl.P
    assert nb >= 8
    grads = plan.new_replicas()
    wdev.fill_grads(grads, c.off, wl, 1)
    master0 = torch.randn(plan.L, device="cuda") * 0.02
    cfg = dps.adamw_cfg(2e-4, 0.9, 0.95, 1e-8, 0.1, 1.0, 1)
    max_len = max(plan.bucket(b)[1] for b in range(nb))

    def run(prefetch):
        """prefetch: False (sequential), True (two streams) or "fused" (dp_unit_backward)."""
        shards = master0.to(torch.bfloat16)
        st = [master0.clone(), plan.new_state(), plan.new_state()]
        mean = plan.new_state()
        ws = plan.new_workspace()
        bufs = [torch.zeros(P, max_len, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        seen = []
        if not prefetch:
            for b in range(nb):
                o, ln, _ = plan.bucket(b)
                dps.dp_unit_all_gather(plan, ws, shards, b, bufs[0])
                seen.append(bufs[0][:, :ln].clone())
                dps.dp_unit_reduce_scatter(plan, ws, grads[:, o:o + ln], b, mean, want_sumsq=True)
        elif prefetch == "fused":
            dps.dp_unit_all_gather(plan, ws, shards, 0, bufs[0])
            for b in range(nb):
                o, ln, _ = plan.bucket(b)
                seen.append(bufs[b % 2][:, :ln].clone())
                dps.dp_unit_backward(plan, ws, shards, b + 1 if b + 1 < nb else -1, bufs[(b + 1) % 2],
                                     grads[:, o:o + ln], b, mean, want_sumsq=True)
        else:
            main = torch.cuda.current_stream()
            s_a, s_b = torch.cuda.Stream(), torch.cuda.Stream()
            s_a.wait_stream(main)
            s_b.wait_stream(main)
            released = [None, None]
            for i, b in enumerate(range(nb)):
                o, ln, _ = plan.bucket(b)
                with torch.cuda.stream(s_a):
                    if released[i % 2] is not None:
                        s_a.wait_event(released[i % 2])
                    dps.dp_unit_all_gather(plan, ws, shards, b, bufs[i % 2])
                    ev = torch.cuda.Event()
                    ev.record(s_a)
                with torch.cuda.stream(s_b):
                    s_b.wait_event(ev)
                    seen.append(bufs[i % 2][:, :ln].clone())   # the unit's "backward" reads it
                    dps.dp_unit_reduce_scatter(plan, ws, grads[:, o:o + ln], b, mean, want_sumsq=True)
                    done = torch.cuda.Event()
                    done.record(s_b)
                    released[i % 2] = done
            main.wait_stream(s_a)
            main.wait_stream(s_b)
        dps.dp_clip_coef(plan, ws, 1.0)
        dps.dp_shard_adamw_step(plan, ws, mean, *st, shards, cfg, use_clip_coef=True)
        torch.cuda.synchronize()
        return mean, dps.dp_read_norm(plan, ws), st, shards, seen

    m1, n1, st1, sh1, seen1 = run(False)
    for mode in (True, "fused"):
        m2, n2, st2, sh2, seen2 = run(mode)
        assert n1 == n2 and n1[2] == 0
        assert torch.equal(m1.view(torch.int32), m2.view(torch.int32))
        assert torch.equal(sh1, sh2)
        for a, b in zip(st1, st2):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
        assert len(seen1) == len(seen2)
        for a, b in zip(seen1, seen2):
            assert torch.equal(a, b)


def test_captured_prefetch_step_equals_eager():
    """The whole ZeRO-3 backward + update with the two-stream prefetch schedule,
    captured once as a CUDA graph (cfg=None, scalars from dp_set_adamw_cfg) and
    replayed for steps 1 and 2, equals the eager sequential flow bit for bit."""
    wl = configs.llama_1b1_zero2(layers=2, embeddings=False)
    wl.bucket_bytes = 4 << 20
    c = Case(wl)
    plan, nb, P = c.plan, c.plan.n_buckets, wl.P
    grads = plan.new_replicas()
    wdev.fill_grads(grads, c.off, wl, 1)
    master0 = torch.randn(plan.L, device="cuda") * 0.02
    max_len = max(plan.bucket(b)[1] for b in range(nb))

    def cfg(t):
        return dps.adamw_cfg(2e-4, 0.9, 0.95, 1e-8, 0.1, 1.0, t)

    # eager, sequential
    sh_e = master0.to(torch.bfloat16)
    st_e = [master0.clone(), plan.new_state(), plan.new_state()]
    mean_e, ws_e = plan.new_state(), plan.new_workspace()
    buf = torch.zeros(P, max_len, dtype=torch.bfloat16, device="cuda")
    for t in (1, 2):
        for b in range(nb):
            o, ln, _ = plan.bucket(b)
            dps.dp_unit_all_gather(plan, ws_e, sh_e, b, buf)
            dps.dp_unit_reduce_scatter(plan, ws_e, grads[:, o:o + ln], b, mean_e, want_sumsq=True)
        dps.dp_clip_coef(plan, ws_e, 1.0)
        dps.dp_shard_adamw_step(plan, ws_e, mean_e, *st_e, sh_e, cfg(t), use_clip_coef=True)
    # captured prefetch schedule
    sh_g = master0.to(torch.bfloat16)
    st_g = [master0.clone(), plan.new_state(), plan.new_state()]
    mean_g, ws_g = plan.new_state(), plan.new_workspace()
    bufs = [torch.zeros(P, max_len, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    s_a, s_b = torch.cuda.Stream(), torch.cuda.Stream()

    def body():
        cur = torch.cuda.current_stream()
        s_a.wait_stream(cur)
        s_b.wait_stream(cur)
        released = [None, None]
        for i, b in enumerate(range(nb)):
            o, ln, _ = plan.bucket(b)
            with torch.cuda.stream(s_a):
                if released[i % 2] is not None:
                    s_a.wait_event(released[i % 2])
                dps.dp_unit_all_gather(plan, ws_g, sh_g, b, bufs[i % 2])
                ev = torch.cuda.Event()
                ev.record(s_a)
            with torch.cuda.stream(s_b):
                s_b.wait_event(ev)
                dps.dp_unit_reduce_scatter(plan, ws_g, grads[:, o:o + ln], b, mean_g, want_sumsq=True)
                done = torch.cuda.Event()
                done.record(s_b)
                released[i % 2] = done
        cur.wait_stream(s_a)
        cur.wait_stream(s_b)
        dps.dp_clip_coef(plan, ws_g, 1.0)
        dps.dp_shard_adamw_step(plan, ws_g, mean_g, *st_g, sh_g, None, use_clip_coef=True)

    # launcher setup outside the capture, on scratch state
    scratch = [plan.new_state() for _ in range(4)]
    dps.dp_unit_all_gather(plan, ws_g, sh_g, 0, bufs[0])
    o0, ln0, _ = plan.bucket(0)
    dps.dp_unit_reduce_scatter(plan, ws_g, grads[:, o0:o0 + ln0], 0, scratch[0])
    dps.dp_shard_adamw_step(plan, ws_g, scratch[0], *scratch[1:], plan.new_state().to(torch.bfloat16),
                            cfg(1))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        body()
    for t in (1, 2):
        dps.dp_set_adamw_cfg(plan, ws_g, cfg(t))
        graph.replay()
    torch.cuda.synchronize()
    assert dps.dp_read_norm(plan, ws_g) == dps.dp_read_norm(plan, ws_e)
    assert torch.equal(sh_g, sh_e)
    assert torch.equal(mean_g.view(torch.int32), mean_e.view(torch.int32))
    for x, y in zip(st_g, st_e):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))


def test_captured_fused_backward_step_equals_eager():
    """The ZeRO-3 backward as dp_unit_backward launches (the next unit's gather
    beside this unit's reduce-scatter) plus the update, captured once as a CUDA
    graph and replayed for steps 1 and 2, equals the eager sequential flow bit for
    bit (mean, norm, shards, master/m/v)."""
    wl = configs.llama_1b1_zero2(layers=2, embeddings=False)
    wl.bucket_bytes = 4 << 20
    c = Case(wl)
    plan, nb, P = c.plan, c.plan.n_buckets, wl.P
    grads = plan.new_replicas()
    wdev.fill_grads(grads, c.off, wl, 1)
    master0 = torch.randn(plan.L, device="cuda") * 0.02
    max_len = max(plan.bucket(b)[1] for b in range(nb))

    def cfg(t):
        return dps.adamw_cfg(2e-4, 0.9, 0.95, 1e-8, 0.1, 1.0, t)

    sh_e = master0.to(torch.bfloat16)
    st_e = [master0.clone(), plan.new_state(), plan.new_state()]
    mean_e, ws_e = plan.new_state(), plan.new_workspace()
    buf = torch.zeros(P, max_len, dtype=torch.bfloat16, device="cuda")
    for t in (1, 2):
        for b in range(nb):
            o, ln, _ = plan.bucket(b)
            dps.dp_unit_all_gather(plan, ws_e, sh_e, b, buf)
            dps.dp_unit_reduce_scatter(plan, ws_e, grads[:, o:o + ln], b, mean_e, want_sumsq=True)
        dps.dp_clip_coef(plan, ws_e, 1.0)
        dps.dp_shard_adamw_step(plan, ws_e, mean_e, *st_e, sh_e, cfg(t), use_clip_coef=True)

    sh_g = master0.to(torch.bfloat16)
    st_g = [master0.clone(), plan.new_state(), plan.new_state()]
    mean_g, ws_g = plan.new_state(), plan.new_workspace()
    bufs = [torch.zeros(P, max_len, dtype=torch.bfloat16, device="cuda") for _ in range(2)]

    def body():
        dps.dp_unit_all_gather(plan, ws_g, sh_g, 0, bufs[0])
        for b in range(nb):
            o, ln, _ = plan.bucket(b)
            dps.dp_unit_backward(plan, ws_g, sh_g, b + 1 if b + 1 < nb else -1, bufs[(b + 1) % 2],
                                 grads[:, o:o + ln], b, mean_g, want_sumsq=True)
        dps.dp_clip_coef(plan, ws_g, 1.0)
        dps.dp_shard_adamw_step(plan, ws_g, mean_g, *st_g, sh_g, None, use_clip_coef=True)

    # launcher setup outside the capture, on scratch state
    scratch = [plan.new_state() for _ in range(4)]
    o0, ln0, _ = plan.bucket(0)
    dps.dp_unit_backward(plan, ws_g, sh_g, 1, bufs[1], grads[:, o0:o0 + ln0], 0, scratch[0])
    dps.dp_shard_adamw_step(plan, ws_g, scratch[0], *scratch[1:], plan.new_state().to(torch.bfloat16),
                            cfg(1))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        body()
    for t in (1, 2):
        dps.dp_set_adamw_cfg(plan, ws_g, cfg(t))
        graph.replay()
    torch.cuda.synchronize()
    assert dps.dp_read_norm(plan, ws_g) == dps.dp_read_norm(plan, ws_e)
    assert torch.equal(sh_g, sh_e)
    assert torch.equal(mean_g.view(torch.int32), mean_e.view(torch.int32))
    for x, y in zip(st_g, st_e):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))

"""Whole steps captured in a CUDA graph: the update kernels take AdamW's per-step
scalars from the workspace (dp_set_adamw_cfg) when called with cfg=None, so one
captured clipped ZeRO-2 step (reduce-scatter, clip coefficient, AdamW + all-gather)
replays steps 1, 2, 3 bit for bit like the eager calls."""
import pytest
import torch

import gradient_sync_zero_gb300 as dps
from harness import Case
from workloads import configs

pytestmark = pytest.mark.gpu


def cfg_of(a, t):
    return dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, t)


def test_captured_zero_step_replays_like_eager():
    wl = configs.tiny_plumbing()
    wl.adamw = configs.AdamW(max_norm=0.3)
    c = Case(wl)
    a = wl.adamw
    grads = [c.to_replicas(c.host_grads(s)) for s in (1, 2, 3)]
    master0 = c.host_master()
    # eager, cfg per call
    p_e = c.plan.new_replicas()
    st_e = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    mean_e = c.plan.new_state()
    for t in (1, 2, 3):
        dps.dp_reduce_scatter_mean(c.plan, c.ws, grads[t - 1], mean_e, want_sumsq=True)
        dps.dp_clip_coef(c.plan, c.ws, a.max_norm)
        dps.dp_adamw_all_gather(c.plan, c.ws, mean_e, *st_e, p_e, cfg_of(a, t))
    torch.cuda.synchronize()
    # graph: the step captured once with cfg=None; inputs copied into a fixed buffer
    ws = c.plan.new_workspace()
    g_in = c.plan.new_replicas()
    p_g = c.plan.new_replicas()
    st_g = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    mean_g = c.plan.new_state()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        # warm-up outside the capture (one-time host-side setup of each launcher)
        tmp = [c.plan.new_state() for _ in range(4)]
        dps.dp_reduce_scatter_mean(c.plan, ws, g_in, tmp[0], want_sumsq=True)
        dps.dp_clip_coef(c.plan, ws, a.max_norm)
        dps.dp_adamw_all_gather(c.plan, ws, *tmp, c.plan.new_replicas(), cfg_of(a, 1))
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=s):
            dps.dp_reduce_scatter_mean(c.plan, ws, g_in, mean_g, want_sumsq=True)
            dps.dp_clip_coef(c.plan, ws, a.max_norm)
            dps.dp_adamw_all_gather(c.plan, ws, mean_g, *st_g, p_g, None)
    for t in (1, 2, 3):
        g_in.copy_(grads[t - 1])
        dps.dp_set_adamw_cfg(c.plan, ws, cfg_of(a, t))
        graph.replay()
    torch.cuda.synchronize()
    norm_g = dps.dp_read_norm(c.plan, ws)
    norm_e = dps.dp_read_norm(c.plan, c.ws)
    assert norm_g == norm_e and norm_g[1] < 1.0
    assert torch.equal(p_g, p_e)
    for x, y in zip(st_g, st_e):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))


def test_update_without_scalars_is_refused_on_the_device():
    wl = configs.tiny_plumbing()
    c = Case(wl)
    st = [c.to_flat(c.host_master()), c.plan.new_state(), c.plan.new_state()]
    before = st[0].clone()
    mean, params = c.plan.new_state(), c.plan.new_replicas()
    dps.dp_adamw_all_gather(c.plan, c.ws, mean, *st, params, None, use_clip_coef=False)
    norm, coef, status = dps.dp_read_norm(c.plan, c.ws, raise_on_status=False)
    assert status & dps.DP_STATUS_NO_SCALARS
    assert torch.equal(st[0], before)                       # nothing was updated
    with pytest.raises(dps.DPError):
        dps.dp_read_norm(c.plan, c.ws)
    c.plan.upload(c.ws)                                      # a fresh image clears the status
    dps.dp_set_adamw_cfg(c.plan, c.ws, cfg_of(wl.adamw, 1))
    dps.dp_shard_adamw_step(c.plan, c.ws, mean, *st, params[0], None, use_clip_coef=False)
    assert dps.dp_read_norm(c.plan, c.ws)[2] == 0

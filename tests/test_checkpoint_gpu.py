"""Checkpoint and resume on the GPU: saving after step 2 and resuming into fresh
buffers (of the same plan, or of a plan with another bucket size) gives, at
step 3, the same bits as running straight through."""
import pytest
import torch

import gradient_sync_zero_gb300 as dps
from harness import Case
from workloads import configs

pytestmark = pytest.mark.gpu


def cfg(a, t):
    return dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, t)


def test_resume_is_bit_identical(tmp_path):
    wl = configs.tiny_plumbing()
    wl.adamw = configs.AdamW(max_norm=0.3)               # clip active
    c = Case(wl)
    grads = [c.to_replicas(c.host_grads(s)) for s in (1, 2, 3)]
    master0 = c.host_master()
    # straight through
    p_ref = c.plan.new_replicas()
    s_ref = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    for t in (1, 2, 3):
        dps.dp_fused_zero_step(c.plan, c.ws, grads[t - 1], p_ref, *s_ref, cfg(wl.adamw, t))
    # two steps, save, resume in fresh buffers
    p = c.plan.new_replicas()
    st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    for t in (1, 2):
        dps.dp_fused_zero_step(c.plan, c.ws, grads[t - 1], p, *st, cfg(wl.adamw, t))
    path = str(tmp_path / "s2.ckpt")
    dps.dp_checkpoint_save(c.plan, path, *st, step=2)
    del st, p
    fresh = [torch.full((c.plan.L,), float("nan"), device="cuda") for _ in range(3)]
    t0 = dps.dp_checkpoint_load(c.plan, path, *fresh)
    assert t0 == 2
    p2 = c.plan.new_replicas()
    ws2 = c.plan.new_workspace()
    dps.dp_fused_zero_step(c.plan, ws2, grads[2], p2, *fresh, cfg(wl.adamw, t0 + 1))
    torch.cuda.synchronize()
    assert torch.equal(p2, p_ref)
    for a, b in zip(fresh, s_ref):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_device_and_host_files_agree(tmp_path):
    """A save from device memory writes the same file as a save of the same
    arrays from host memory; a device load equals a host load."""
    wl = configs.tiny_plumbing()
    c = Case(wl)
    st = [c.to_flat(c.host_master()), c.plan.new_state(), c.plan.new_state()]
    st[1].normal_()
    st[2].uniform_()
    st[1][c.padding_mask().cuda()] = 0
    st[2][c.padding_mask().cuda()] = 0
    dev, host = str(tmp_path / "dev.ckpt"), str(tmp_path / "host.ckpt")
    dps.dp_checkpoint_save(c.plan, dev, *st, step=5)
    dps.dp_checkpoint_save(c.plan, host, *[x.cpu() for x in st], step=5)
    assert open(dev, "rb").read() == open(host, "rb").read()
    other = dps.Plan(c.sizes, 64 * 1024, 8)                 # another bucket size and P
    got = [torch.zeros(other.L, device="cuda") for _ in range(3)]
    assert dps.dp_checkpoint_load(other, dev, *got) == 5
    got_h = [torch.zeros(other.L) for _ in range(3)]
    dps.dp_checkpoint_load(other, host, *got_h)
    for a, b in zip(got, got_h):
        assert torch.equal(a.cpu(), b)


def test_resume_into_a_mesh_plan_continues_like_the_mesh_run(tmp_path):
    """Elastic restart onto another layout: state saved from a flat P=8 run after
    step 1 and loaded into a 2 x 4 mesh plan continues exactly like a 2 x 4 run that
    started from the same state (the update is elementwise; only the layout moved)."""
    wl = configs.tiny_plumbing()
    wl.P = 8
    c = Case(wl)
    grads1 = c.to_replicas(c.host_grads(1))
    master0 = c.host_master()
    st = [c.to_flat(master0), c.plan.new_state(), c.plan.new_state()]
    dps.dp_fused_zero_step(c.plan, c.ws, grads1, c.plan.new_replicas(), *st, cfg(wl.adamw, 1))
    path = str(tmp_path / "flat.ckpt")
    dps.dp_checkpoint_save(c.plan, path, *st, step=1)
    mesh = dps.Plan(c.sizes, wl.bucket_bytes, 8, c.decay, mesh=(2, 4))
    ws_m = mesh.new_workspace()
    st_m = [mesh.new_state() for _ in range(3)]
    t = dps.dp_checkpoint_load(mesh, path, *st_m)
    # the same state placed directly in the mesh layout from the flat arrays
    from workloads import device as wdev
    off_f, off_m = c.plan.tensor_offsets(), mesh.tensor_offsets()
    st_ref = []
    for a in st:
        x = mesh.new_state()
        for k, n in enumerate(c.sizes):
            x[off_m[k]:off_m[k] + n] = a[off_f[k]:off_f[k] + n]
        st_ref.append(x)
    for a, b in zip(st_m, st_ref):
        assert torch.equal(a, b)
    g2 = c.host_grads(2)
    def to_mesh(g):
        buf = mesh.new_replicas()
        src = torch.from_numpy(g.view("int16")).view(torch.bfloat16).cuda()
        for r in range(8):
            wdev.fill_flat(buf[r], off_m, c.sizes, src[r])
        return buf
    p1, p2 = mesh.new_replicas(), mesh.new_replicas()
    dps.dp_fused_zero_step(mesh, ws_m, to_mesh(g2), p1, *st_m, cfg(wl.adamw, t + 1))
    ws2 = mesh.new_workspace()
    dps.dp_fused_zero_step(mesh, ws2, to_mesh(g2), p2, *st_ref, cfg(wl.adamw, t + 1))
    torch.cuda.synchronize()
    assert torch.equal(p1, p2)
    for a, b in zip(st_m, st_ref):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))

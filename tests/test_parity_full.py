"""GPU path against the oracle at the workloads' full sizes, in the launch
configuration the bench times (one dp_fused_zero_step / dp_allreduce_mean over
all buckets).

* GPT-2 small all-reduce (P=8, 124M): every element of every replica.
* Llama 1.1B and GPT 2.5B fused ZeRO-2 with clipping (P=8), and the P=16 sweep
  at 64 KiB and 256 MiB buckets, three steps each with fresh gradients: at every
  step the oracle streams every bucket's input bytes (copied back from the
  device) to form the global clip norm, then recomputes sampled buckets (first,
  middle, last, random ones, and those holding the flat indices where a 32-bit
  byte or element offset would wrap) element by element, carrying their
  master, m and v on its own from step to step.
"""
import math

import numpy as np
import pytest
import torch

import gradient_sync_zero_gb300 as dps
import oracle as oracle_mod
from harness import assert_replicas_equal, bf16_ulp_diff, rel_err, u16
from workloads import configs, device as wdev, gen

pytestmark = pytest.mark.gpu


def setup(wl):
    plan = dps.Plan(wl.sizes, wl.bucket_bytes, wl.P, wl.decay)
    off = plan.tensor_offsets()
    ws = plan.new_workspace()
    grads = plan.new_replicas()
    wdev.fill_grads(grads, off, wl, step=1)
    return plan, off, ws, grads


def host_grads(grads, off, sizes, tensors):
    parts = [grads[:, off[t]:off[t] + sizes[t]] for t in tensors if sizes[t]]
    return u16(torch.cat(parts, dim=1)) if parts else np.zeros((grads.shape[0], 0), np.uint16)


def host_flat(buf, off, sizes, tensors):
    parts = [buf[off[t]:off[t] + sizes[t]] for t in tensors if sizes[t]]
    return torch.cat(parts).cpu().numpy() if parts else np.zeros(0, np.float32)


def bucket_tensors(op, b):
    return sorted(int(t) for t in np.nonzero(op["t_bucket"] == b)[0])


def test_gpt2_small_allreduce_full(orc):
    wl = configs.gpt2_small_allreduce()
    plan, off, ws, grads = setup(wl)
    g_host = u16(wdev.gather_flat(grads[:, :plan.L], off, wl.sizes))
    dps.dp_allreduce_mean(plan, ws, grads)
    torch.cuda.synchronize()
    want, _, st = orc.allreduce_mean(wl.sizes, wl.bucket_bytes, wl.P, g_host, want_mean=False)
    del g_host
    got = u16(wdev.gather_flat(grads[:, :plan.L], off, wl.sizes))
    assert np.array_equal(got, want)
    assert st.replicas_equal == 1
    assert_replicas_equal(grads, plan.L)


def boundary_buckets(op, boundaries):
    """Buckets holding the elements just below and at each flat index in
    `boundaries` (those inside [0, L)): where 32-bit byte or element offsets
    would wrap."""
    b_off, b_len = op["b_off"], op["b_len"]
    out = set()
    for x in boundaries:
        for e in (x - 1, x):
            if 0 <= e < op["L"]:
                out.add(int(np.searchsorted(b_off, e, side="right") - 1))
    return out


# flat indices where a 32-bit offset would wrap: fp32 byte offset 2^31 and 2^32,
# bf16 byte offset 2^32 (element 2^31), and element 2^31 itself
WRAP_POINTS = (1 << 29, 1 << 30, 1 << 31)


def zero_clip_sampled(orc, wl, n_random=2, batch=16, steps=3):
    """`steps` clipped ZeRO-2 steps over the whole plan, fresh gradients from
    (seed, step, rank) every step.  The oracle carries master, m and v of the
    sampled buckets from step to step on its own (each owner's optimizer state
    persists across steps), and recomputes the global clip norm from every
    bucket's input bytes at every step."""
    plan, off, ws, grads = setup(wl)
    master = plan.new_state()
    wdev.fill_flat(master, off, wl.sizes, gen.master_values(wl, 0, wl.n_params, "cuda"))
    m, v, params = plan.new_state(), plan.new_state(), plan.new_replicas()
    op = orc.plan(wl.sizes, wl.bucket_bytes, wl.P)
    nb = op["n_buckets"]
    assert nb == plan.n_buckets
    rng = np.random.default_rng(wl.seed)
    sample = sorted(set([0, nb // 2, nb - 1] + rng.integers(0, nb, n_random).tolist())
                    | boundary_buckets(op, WRAP_POINTS))
    # the oracle's optimizer state of the sampled buckets: master from the
    # generator (copied before the first step), m = v = 0
    state = {}
    for b in sample:
        tb = bucket_tensors(op, b)
        mb = host_flat(master, off, wl.sizes, tb)
        state[b] = [mb, np.zeros_like(mb), np.zeros_like(mb)]
    a = wl.adamw
    coefs = []
    for t in range(1, steps + 1):
        if t > 1:
            wdev.fill_grads(grads, off, wl, step=t)
        keep = {b: host_grads(grads, off, wl.sizes, bucket_tensors(op, b)) for b in sample}
        # oracle's global norm: every bucket's input bytes, streamed in batches
        sums = []
        for b0 in range(0, nb, batch):
            tb = sorted(x for b in range(b0, min(nb, b0 + batch)) for x in bucket_tensors(op, b))
            sub = [wl.sizes[x] for x in tb]
            sums.extend(orc.bucket_sumsq(sub, wl.bucket_bytes, wl.P,
                                         host_grads(grads, off, wl.sizes, tb)).tolist())
        assert len(sums) == nb
        coef_ref, norm_ref = orc.clip_coef(sums, a.max_norm)
        total = orc.sum(sums)
        dps.dp_fused_zero_step(plan, ws, grads, params, master, m, v,
                               dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay,
                                             a.max_norm, t))
        norm, coef, status = dps.dp_read_norm(plan, ws)
        assert status == 0
        assert math.isclose(norm, norm_ref, rel_tol=1e-10), (t, norm, norm_ref)
        assert coef == coef_ref, (t, coef, coef_ref)
        coefs.append(coef)
        cfg = oracle_mod.adamw_cfg(a, t)
        for b in sample:
            tb = bucket_tensors(op, b)
            sub = [wl.sizes[x] for x in tb]
            dec = [wl.decay[x] for x in tb]
            p_ref, m_ref, mm_ref, v_ref, _, st = orc.zero_step(sub, dec, wl.bucket_bytes, wl.P,
                                                               keep[b], *state[b], cfg,
                                                               sumsq_total=total)
            assert st.n_buckets == 1 and st.replicas_equal == 1
            for name, dev, ref in (("master", master, m_ref), ("m", m, mm_ref), ("v", v, v_ref)):
                got = host_flat(dev, off, wl.sizes, tb)
                e = rel_err(got, ref)
                assert np.all(e <= 1e-5), f"step {t} bucket {b} {name}: max rel err {e.max():.3g}"
                assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), \
                    f"step {t} bucket {b} {name} bits"
            got_p = host_grads(params, off, wl.sizes, tb)
            assert np.all(bf16_ulp_diff(got_p, p_ref) <= 1), f"step {t} bucket {b} params"
            assert np.array_equal(got_p, p_ref), f"step {t} bucket {b} params bits"
            state[b] = [m_ref, mm_ref, v_ref]     # the oracle's own state, carried on
        assert_replicas_equal(params, plan.L)
    return coefs


def test_llama_1b1_zero2_clip_sampled(orc):
    coefs = zero_clip_sampled(orc, configs.llama_1b1_zero2())
    assert all(c < 1.0 for c in coefs)          # ||mean|| ~ 5.9: the clip is active


def test_gpt_2b5_zero2_clip_sampled(orc):
    wl = configs.gpt_2b5_clip()
    assert wl.n_params > (1 << 31)              # buckets beyond element 2^31 are sampled
    coefs = zero_clip_sampled(orc, wl, batch=8)
    assert all(0.2 < c < 0.3 for c in coefs)    # ||mean|| ~ 4


@pytest.mark.parametrize("cap", [64 * 1024, 256 << 20])
def test_sweep_p16_zero2_clip_sampled(orc, cap):
    wl = configs.sweep_small_tensors(cap, "zero")
    zero_clip_sampled(orc, wl, n_random=8, batch=64 if cap < (1 << 20) else 2)


@pytest.mark.parametrize("cap", [64 * 1024, 25 << 20])
def test_sweep_p16_allreduce_sampled(orc, cap):
    wl = configs.sweep_small_tensors(cap, "allreduce")
    plan, off, ws, grads = setup(wl)
    op = orc.plan(wl.sizes, wl.bucket_bytes, wl.P)
    nb = op["n_buckets"]
    rng = np.random.default_rng(5)
    sample = sorted(set([0, nb - 1] + rng.integers(0, nb, 10).tolist()))
    keep = {b: (bucket_tensors(op, b), host_grads(grads, off, wl.sizes, bucket_tensors(op, b)))
            for b in sample}
    dps.dp_allreduce_mean(plan, ws, grads)
    torch.cuda.synchronize()
    for b in sample:
        tb, g_b = keep[b]
        want, _, _ = orc.allreduce_mean([wl.sizes[t] for t in tb], wl.bucket_bytes, wl.P, g_b)
        assert np.array_equal(host_grads(grads, off, wl.sizes, tb), want), f"bucket {b}"
    assert_replicas_equal(grads, plan.L)


def test_llama_1b1_zero3_fused_backward_sampled(orc):
    """The ZeRO-3 unit flow at the 1.1B workload's full size, its backward as
    dp_unit_backward launches (the next unit's gather beside this unit's
    reduce-scatter), two clipped steps: the global norm and coefficient equal the
    oracle's; for sampled units (first, middle, last, random, and those holding
    flat indices 2^29 and 2^30) the gathered rows equal the parameter shards, and
    the mean, master/m/v and updated shards equal the oracle's step bit for bit
    (the oracle pins that the ZeRO-3 update equals the ZeRO-2 step's on the same
    mean, so its ZeRO-2 step on the sampled buckets is the reference)."""
    wl = configs.llama_1b1_zero2()
    plan, off, ws, grads = setup(wl)
    master = plan.new_state()
    wdev.fill_flat(master, off, wl.sizes, gen.master_values(wl, 0, wl.n_params, "cuda"))
    m, v, mean = plan.new_state(), plan.new_state(), plan.new_state()
    shards = master.to(torch.bfloat16)
    op = orc.plan(wl.sizes, wl.bucket_bytes, wl.P)
    nb, P = op["n_buckets"], wl.P
    rng = np.random.default_rng(wl.seed + 3)
    sample = sorted(set([0, nb // 2, nb - 1] + rng.integers(0, nb, 2).tolist())
                    | boundary_buckets(op, WRAP_POINTS))
    buckets = [plan.bucket(b) for b in range(nb)]
    max_len = max(ln for _, ln, _ in buckets)
    bufs = [torch.zeros(P, max_len, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    state = {}
    for b in sample:
        mb = host_flat(master, off, wl.sizes, bucket_tensors(op, b))
        state[b] = [mb, np.zeros_like(mb), np.zeros_like(mb)]
    a = wl.adamw
    for t in (1, 2):
        if t > 1:
            wdev.fill_grads(grads, off, wl, step=t)
        keep = {b: host_grads(grads, off, wl.sizes, bucket_tensors(op, b)) for b in sample}
        before = {b: shards[buckets[b][0]:buckets[b][0] + buckets[b][1]].clone() for b in sample}
        sums = []
        for b0 in range(0, nb, 16):
            tb = sorted(x for b in range(b0, min(nb, b0 + 16)) for x in bucket_tensors(op, b))
            sums.extend(orc.bucket_sumsq([wl.sizes[x] for x in tb], wl.bucket_bytes, P,
                                         host_grads(grads, off, wl.sizes, tb)).tolist())
        coef_ref, norm_ref = orc.clip_coef(sums, a.max_norm)
        total = orc.sum(sums)
        gathered = {}
        dps.dp_unit_all_gather(plan, ws, shards, 0, bufs[0])
        for b in range(nb):
            o, ln, _ = buckets[b]
            if b in sample:
                gathered[b] = bufs[b % 2][:, :ln].clone()       # unit b's backward reads it
            dps.dp_unit_backward(plan, ws, shards, b + 1 if b + 1 < nb else -1, bufs[(b + 1) % 2],
                                 grads[:, o:o + ln], b, mean, want_sumsq=True)
        dps.dp_clip_coef(plan, ws, a.max_norm)
        dps.dp_shard_adamw_step(plan, ws, mean, master, m, v, shards,
                                dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay,
                                              a.max_norm, t), use_clip_coef=True)
        norm, coef, status = dps.dp_read_norm(plan, ws)
        assert status == 0
        assert math.isclose(norm, norm_ref, rel_tol=1e-10), (t, norm, norm_ref)
        assert coef == coef_ref < 1.0
        cfg = oracle_mod.adamw_cfg(a, t)
        for b in sample:
            tb = bucket_tensors(op, b)
            for r in range(P):
                assert torch.equal(gathered[b][r], before[b]), f"step {t} unit {b} row {r}"
            p_ref, m_ref, mm_ref, v_ref, mean_ref, _ = orc.zero_step(
                [wl.sizes[x] for x in tb], [wl.decay[x] for x in tb], wl.bucket_bytes, P, keep[b],
                *state[b], cfg, sumsq_total=total)
            got_mean = host_flat(mean, off, wl.sizes, tb)
            assert np.array_equal(got_mean.view(np.uint32), mean_ref.view(np.uint32)), f"{t} {b} mean"
            for name, dev, ref in (("master", master, m_ref), ("m", m, mm_ref), ("v", v, v_ref)):
                got = host_flat(dev, off, wl.sizes, tb)
                assert np.all(rel_err(got, ref) <= 1e-5), f"step {t} unit {b} {name}"
                assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"{t} {b} {name}"
            got_sh = u16(torch.cat([shards[off[x]:off[x] + wl.sizes[x]] for x in tb if wl.sizes[x]]))
            assert np.array_equal(got_sh, p_ref[0]), f"step {t} unit {b} shards"
            state[b] = [m_ref, mm_ref, v_ref]

"""GPU path against the oracle at the workloads' full sizes, in the launch
configuration the bench times (one dp_fused_zero_step / dp_allreduce_mean over
all buckets).

* GPT-2 small all-reduce (P=8, 124M): every element of every replica.
* Llama 1.1B and GPT 2.5B fused ZeRO-2 with clipping (P=8), and the P=16 sweep
  at 64 KiB and 256 MiB buckets: the oracle streams every bucket's input bytes
  (copied back from the device before the step) to form the global clip norm,
  then recomputes sampled buckets (first, middle, last, plus random ones)
  element by element.
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


def zero_clip_sampled(orc, wl, n_random=2, batch=16):
    plan, off, ws, grads = setup(wl)
    master = plan.new_state()
    wdev.fill_flat(master, off, wl.sizes, gen.master_values(wl, 0, wl.n_params, "cuda"))
    m, v, params = plan.new_state(), plan.new_state(), plan.new_replicas()
    op = orc.plan(wl.sizes, wl.bucket_bytes, wl.P)
    nb = op["n_buckets"]
    assert nb == plan.n_buckets
    rng = np.random.default_rng(wl.seed)
    sample = sorted(set([0, nb // 2, nb - 1] + rng.integers(0, nb, n_random).tolist()))
    # inputs of the sampled buckets, copied before the step
    keep = {}
    for b in sample:
        tb = bucket_tensors(op, b)
        keep[b] = (tb, host_grads(grads, off, wl.sizes, tb), host_flat(master, off, wl.sizes, tb))
    # oracle's global norm: every bucket's input bytes, streamed in batches
    sums = []
    for b0 in range(0, nb, batch):
        tb = sorted(t for b in range(b0, min(nb, b0 + batch)) for t in bucket_tensors(op, b))
        sub = [wl.sizes[t] for t in tb]
        sums.extend(orc.bucket_sumsq(sub, wl.bucket_bytes, wl.P,
                                     host_grads(grads, off, wl.sizes, tb)).tolist())
    assert len(sums) == nb
    coef_ref, norm_ref = orc.clip_coef(sums, wl.adamw.max_norm)
    total = orc.sum(sums)
    a = wl.adamw
    dps.dp_fused_zero_step(plan, ws, grads, params, master, m, v,
                           dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay,
                                         a.max_norm, 1))
    norm, coef, status = dps.dp_read_norm(plan, ws)
    assert status == 0
    assert math.isclose(norm, norm_ref, rel_tol=1e-10), (norm, norm_ref)
    assert coef == coef_ref, (coef, coef_ref)
    cfg = oracle_mod.adamw_cfg(a, 1)
    for b in sample:
        tb, g_b, m_b = keep[b]
        sub = [wl.sizes[t] for t in tb]
        dec = [wl.decay[t] for t in tb]
        z = np.zeros_like(m_b)
        p_ref, m_ref, mm_ref, v_ref, _, st = orc.zero_step(sub, dec, wl.bucket_bytes, wl.P, g_b,
                                                           m_b, z, z, cfg, sumsq_total=total)
        assert st.n_buckets == 1 and st.replicas_equal == 1
        for name, dev, ref in (("master", master, m_ref), ("m", m, mm_ref), ("v", v, v_ref)):
            got = host_flat(dev, off, wl.sizes, tb)
            e = rel_err(got, ref)
            assert np.all(e <= 1e-5), f"bucket {b} {name}: max rel err {e.max():.3g}"
            assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"{b} {name} bits"
        got_p = host_grads(params, off, wl.sizes, tb)
        assert np.all(bf16_ulp_diff(got_p, p_ref) <= 1), f"bucket {b} params"
        assert np.array_equal(got_p, p_ref), f"bucket {b} params bits"
    assert_replicas_equal(params, plan.L)
    return coef


def test_llama_1b1_zero2_clip_sampled(orc):
    coef = zero_clip_sampled(orc, configs.llama_1b1_zero2())
    assert coef < 1.0          # ||mean|| ~ 5.9: the clip is active


def test_gpt_2b5_zero2_clip_sampled(orc):
    coef = zero_clip_sampled(orc, configs.gpt_2b5_clip(), batch=8)
    assert 0.2 < coef < 0.3    # ||mean|| ~ 4


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

"""dp_clip_coef_noalloc: the reduce-scatter mean and clip coefficient for callers
that cannot allocate device memory (they are handed buffers by a host that owns
the memory pool, or their allocator must account for every byte, or a
cudaMalloc/cudaFree that may synchronise the device is not acceptable).  The call
keeps its scratch in a library-owned static device array instead of a
workspace.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test; it also passes alone in a fresh
process.  It calls the new entry point through the C ABI and checks it against
the workspace path (dp_reduce_scatter_mean + dp_clip_coef + dp_read_norm) on two
calls in a row, with the parity tests' tolerances (mean <= 1e-6 relative,
norm/coef <= 1e-6 relative), where bit equality is expected as well; on the
small cases also against the oracle directly (its ring mean, its per-bucket sums
of squares and its clip coefficient); and once on a plan that fills the static
array almost to its limit.
"""
import ctypes as C
import math

import numpy as np
import pytest
import torch

import gradient_sync_zero_gb300 as dps
from harness import Case, rel_err, small_workload
from workloads import device as wdev

pytestmark = pytest.mark.gpu


def _noalloc(plan, grads, mean, max_norm, coef_out, norm_out):
    """Direct C-ABI call (no binding-side checks)."""
    lib = dps.lib()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.dp_clip_coef_noalloc(plan.handle, C.c_void_p(grads.data_ptr()),
                                    C.c_void_p(mean.data_ptr()), C.c_double(max_norm),
                                    C.c_void_p(coef_out.data_ptr()),
                                    C.c_void_p(norm_out.data_ptr()), stream)


def _reference(c, grads, max_norm):
    mean = c.plan.new_state()
    dps.dp_reduce_scatter_mean(c.plan, c.ws, grads, mean, want_sumsq=True)
    dps.dp_clip_coef(c.plan, c.ws, max_norm)
    norm, coef, status = dps.dp_read_norm(c.plan, c.ws)
    assert status == 0
    return mean, norm, coef


def test_noalloc_matches_workspace_path_on_two_calls(orc):
    cases = [
        (small_workload([3, 1000, 65536, 13107, 26214, 4097, 27910], 8, 64 * 1024, sigma=0.05,
                        seed=11), 1, 1.0),
        (small_workload([70000, 12, 130000, 5], 5, 32 * 1024, sigma=1e-3, seed=12), 2, 0.25),
    ]
    coef_out = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    norm_out = torch.full((1,), -1.0, dtype=torch.float64, device="cuda")
    for wl, step, max_norm in cases:                      # two calls in a row
        c = Case(wl)
        g_host = c.host_grads(step)
        grads = c.to_replicas(g_host)
        want_mean, want_norm, want_coef = _reference(c, grads, max_norm)
        mean = torch.full((c.plan.L,), float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc(c.plan, grads, mean, max_norm, coef_out, norm_out)
        assert rc == dps.DP_OK, dps.lib().dp_last_error().decode()
        torch.cuda.synchronize()
        got_mean = mean.cpu().numpy()
        ref_mean = want_mean.cpu().numpy()
        assert np.all(rel_err(got_mean, ref_mean) <= 1e-6)
        assert np.array_equal(got_mean.view(np.uint32), ref_mean.view(np.uint32))
        norm, coef = float(norm_out.item()), float(coef_out.item())
        assert math.isclose(norm, want_norm, rel_tol=1e-6) and math.isclose(coef, want_coef,
                                                                            rel_tol=1e-6)
        assert norm == want_norm and coef == want_coef
        if max_norm == 1.0:
            assert coef < 1.0                             # the clip acts in the first case
        # the oracle itself: the literal ring's mean, bit for bit; its compensated
        # norm within the parity tests' 1e-10 and the same fp32 coefficient
        _, orc_mean, _ = orc.allreduce_mean(c.sizes, wl.bucket_bytes, wl.P, g_host)
        got_t = c.from_flat(mean)
        assert np.array_equal(got_t.view(np.uint32), orc_mean.view(np.uint32))
        orc_coef, orc_norm = orc.clip_coef(orc.bucket_sumsq(c.sizes, wl.bucket_bytes, wl.P, g_host),
                                           max_norm)
        assert math.isclose(norm, orc_norm, rel_tol=1e-10)
        assert coef == orc_coef


def _largest_fitting_plan(limit=32 << 20, tile=8192, P=2):
    """One tensor, as many 8192-element tiles as the static array's tables and
    norm partials still fit (host planning only)."""
    def need(pl):
        return pl.info.workspace_bytes - (-(-4 * pl.L // 256) * 256)
    lo, hi = 1, 1 << 20
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if need(dps.Plan([mid * tile], 1 << 40, P)) <= limit:
            lo = mid
        else:
            hi = mid
    plan = dps.Plan([lo * tile], 1 << 40, P)
    assert need(plan) <= limit < need(dps.Plan([hi * tile], 1 << 40, P))
    return plan


def test_noalloc_near_the_size_limit():
    """A plan that uses all but the last tile's worth of the static array
    (1.2e9 parameters, P = 2): the call equals the workspace path bit for bit on
    every element, twice in a row."""
    plan = _largest_fitting_plan()
    wl = small_workload(plan.sizes, plan.P, 1 << 40, sigma=1e-3, seed=13)
    c = Case(wl)
    assert c.plan.L == plan.L
    grads = c.plan.new_replicas()
    wdev.fill_grads(grads, c.off, wl, step=1)
    want_mean, want_norm, want_coef = _reference(c, grads, 1.0)
    coef_out = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    norm_out = torch.full((1,), -1.0, dtype=torch.float64, device="cuda")
    for _ in range(2):
        mean = torch.full((c.plan.L,), float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc(c.plan, grads, mean, 1.0, coef_out, norm_out)
        assert rc == dps.DP_OK, dps.lib().dp_last_error().decode()
        torch.cuda.synchronize()
        assert torch.equal(mean.view(torch.int32), want_mean.view(torch.int32))
        assert float(norm_out.item()) == want_norm and float(coef_out.item()) == want_coef
        del mean


def test_noalloc_refuses_plans_beyond_its_array():
    sizes = [1 << 30, 1 << 30]                            # 2.1e9 parameters > the static array
    plan = dps.Plan(sizes, 25 << 20, 8)
    t = torch.zeros(8, dtype=torch.float32, device="cuda")
    d = torch.zeros(1, dtype=torch.float64, device="cuda")
    rc = dps.lib().dp_clip_coef_noalloc(plan.handle, C.c_void_p(t.data_ptr()),
                                        C.c_void_p(t.data_ptr()), C.c_double(1.0),
                                        C.c_void_p(t.data_ptr()), C.c_void_p(d.data_ptr()), None)
    assert rc == dps.DP_EINVAL
    assert "static array" in dps.lib().dp_last_error().decode()

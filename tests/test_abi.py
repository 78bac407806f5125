"""The C ABI on the CPU: the library loads, exports every entry point the
header declares, its host planner agrees with the oracle's planner bit for bit,
and bad arguments are rejected before any device work."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import gradient_sync_zero_gb300 as dps
from gradient_sync_zero_gb300 import build as dbuild
from oracle_pins import check_plan_invariants
from workloads import configs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    dbuild.build()


def header_symbols():
    with open(os.path.join(ROOT, "include", "dpsync.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dp_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    syms = header_symbols()
    assert len(syms) >= 18
    lib = C.CDLL(dps.LIB_PATH)
    missing = [s for s in syms if not hasattr(lib, s)]
    assert not missing, missing
    assert dps.dp_version() == 2


def test_declared_entry_points_are_bound():
    lib = dps.lib()
    for s in header_symbols():
        assert getattr(lib, s).restype is not None or s in ("dp_plan_free", "dp_tracker_free")


def _compare(sizes, cap, P, orc, decay=None):
    p = dps.Plan(sizes, cap, P, decay=decay)
    o = orc.plan(sizes, cap, P)
    assert p.n_buckets == o["n_buckets"]
    assert p.L == o["L"]
    assert [p.tensor(t) for t in range(len(sizes))] == list(zip(o["t_bucket"].tolist(),
                                                                 o["t_off"].tolist()))
    for b in range(p.n_buckets):
        off, ln, sh = p.bucket(b)
        assert (off, ln) == (o["b_off"][b], o["b_len"][b])
        assert sh * P == ln
    assert p.stride >= p.L and p.stride % 128 == 0
    assert p.info.n_params == sum(sizes)
    return p


@pytest.mark.parametrize("wl", [configs.tiny_plumbing(), configs.gpt2_small_allreduce(),
                                configs.llama_1b1_zero2(), configs.gpt_2b5_clip()],
                         ids=lambda w: w.name)
def test_planner_matches_oracle_on_workloads(wl, orc):
    p = _compare(wl.sizes, wl.bucket_bytes, wl.P, orc, wl.decay)
    tiles = -(-np.array([p.bucket(b)[1] for b in range(p.n_buckets)]) // p.info.tile_elems)
    assert p.info.n_tiles == int(tiles.sum())


@pytest.mark.parametrize("cap", configs.SWEEP_BUCKETS)
def test_planner_matches_oracle_on_sweep(cap, orc):
    wl = configs.sweep_small_tensors(cap)
    _compare(wl.sizes, cap, wl.P, orc)


def test_planner_matches_oracle_random(orc):
    rng = np.random.default_rng(17)
    for _ in range(200):
        n = int(rng.integers(0, 40))
        sizes = rng.integers(0, 3000, size=n).tolist()
        if n and rng.random() < 0.3:
            sizes[int(rng.integers(0, n))] = int(rng.integers(10000, 50000))
        P = int(rng.integers(1, 65))
        cap = int(rng.choice([2, 16, 100, 4096, 65536]))
        p = _compare(sizes, cap, P, orc)
        check_plan_invariants(sizes, cap, P, orc.plan(sizes, cap, P))
        assert p.L % (16 * P) == 0


def test_tiny_plan_golden():
    import json
    with open(os.path.join(ROOT, "tests", "golden", "plan_tiny_P4_1MiB.json")) as f:
        g = json.load(f)
    p = dps.Plan(g["sizes"], g["bucket_bytes"], g["P"])
    assert [p.tensor(t)[1] for t in range(7)] == g["t_off"]
    assert [p.bucket(b)[:2] for b in range(3)] == list(zip(g["b_off"], g["b_len"]))


def test_empty_and_degenerate_plans():
    p = dps.Plan([], 1024, 4)
    assert (p.n_buckets, p.L, p.info.n_tiles) == (0, 0, 0)
    p = dps.Plan([0, 0], 1024, 4)
    assert (p.n_buckets, p.L) == (1, 0)
    p = dps.Plan([1], 2, 1)
    assert (p.n_buckets, p.L) == (1, 16)
    p = dps.Plan([100], 2, 64)
    assert p.L == 1024 and p.bucket(0)[2] == 16


def test_explicit_stride():
    p = dps.Plan([1000, 24], 1 << 20, 4, replica_stride=4096)
    assert p.stride == 4096
    with pytest.raises(dps.DPError) as e:
        dps.Plan([1000, 24], 1 << 20, 4, replica_stride=1000)
    assert e.value.code == dps.DP_EINVAL


@pytest.mark.parametrize("sizes,cap,P", [([4], 1024, 0), ([4], 1024, 65), ([-1], 1024, 2),
                                         ([4], 1, 2)])
def test_planner_rejects_bad_arguments(sizes, cap, P):
    with pytest.raises(dps.DPError) as e:
        dps.Plan(sizes, cap, P)
    assert e.value.code == dps.DP_EINVAL
    assert dps.lib().dp_last_error().decode()


def test_query_ranges():
    p = dps.Plan([10, 20], 1024, 2)
    with pytest.raises(dps.DPError):
        p.tensor(2)
    with pytest.raises(dps.DPError):
        p.bucket(1)


def test_compute_calls_validate_before_any_device_work():
    """Bad ranges, NULL and misaligned pointers are refused on the host, so no
    kernel is launched (these calls run without a GPU)."""
    lib = dps.lib()
    p = dps.Plan([1000, 24], 1 << 20, 4)
    nb = p.n_buckets
    ws, ok, odd = C.c_void_p(1 << 20), C.c_void_p(1 << 21), C.c_void_p((1 << 21) + 16)
    assert lib.dp_allreduce_mean(p.handle, ws, ok, 0, nb + 1, None) == dps.DP_EINVAL
    assert lib.dp_allreduce_mean(p.handle, ws, ok, 1, 0, None) == dps.DP_EINVAL
    assert lib.dp_allreduce_mean(p.handle, ws, odd, 0, nb, None) == dps.DP_EALIGN
    assert lib.dp_allreduce_mean(None, ws, ok, 0, nb, None) == dps.DP_EINVAL
    assert lib.dp_all_gather(p.handle, None, ok, 0, nb, None) == dps.DP_EINVAL
    assert lib.dp_broadcast(p.handle, ws, ok, 4, 0, nb, None) == dps.DP_EINVAL
    assert lib.dp_reduce_scatter_mean(p.handle, ws, ok, None, 0, nb, 0, None) == dps.DP_EINVAL
    cfg = dps.adamw_cfg(step=0)
    assert lib.dp_fused_zero_step(p.handle, ws, ok, ok, ok, ok, ok, C.byref(cfg), None,
                                  None) == dps.DP_EINVAL
    cfg = dps.adamw_cfg(beta1=1.0)
    assert lib.dp_sharded_adamw_step(p.handle, ws, ok, ok, ok, ok, ok, C.byref(cfg), 0, None, 0,
                                     nb, None) == dps.DP_EINVAL
    assert "range" in lib.dp_last_error().decode() or lib.dp_last_error()
    # a caller-given clip coefficient: only with use_clip_coef, 4-byte aligned
    cfg = dps.adamw_cfg()
    coef, coef_odd = C.c_void_p(1 << 22), C.c_void_p((1 << 22) + 2)
    assert lib.dp_sharded_adamw_step(p.handle, ws, ok, ok, ok, ok, ok, C.byref(cfg), 0, coef, 0,
                                     nb, None) == dps.DP_EINVAL
    assert "use_clip_coef" in lib.dp_last_error().decode()
    assert lib.dp_adamw_all_gather(p.handle, ws, ok, ok, ok, ok, ok, C.byref(cfg), 1, coef_odd,
                                   None) == dps.DP_EALIGN
    assert lib.dp_shard_adamw_step(p.handle, ws, ok, ok, ok, ok, ok, C.byref(cfg), 0, coef,
                                   None) == dps.DP_EINVAL


def test_unit_backward_validates_before_any_device_work():
    """dp_unit_backward refuses units out of range, short strides and a gather
    buffer that overlaps the gradients or the mean, on the host."""
    lib = dps.lib()
    p = dps.Plan([1000, 4096, 333], 8192, 4)
    nb = p.n_buckets
    ws, sh = C.c_void_p(1 << 20), C.c_void_p(1 << 22)
    gb, ug, mean = C.c_void_p(1 << 30), C.c_void_p(1 << 31), C.c_void_p(1 << 32)
    st = 4096
    assert lib.dp_unit_backward(p.handle, ws, sh, nb, gb, st, ug, st, 0, mean, 1, None) == dps.DP_EINVAL
    assert lib.dp_unit_backward(p.handle, ws, sh, 0, gb, st, ug, st, -2, mean, 1, None) == dps.DP_EINVAL
    assert lib.dp_unit_backward(p.handle, ws, sh, 1, gb, 16, ug, st, 0, mean, 1, None) == dps.DP_EINVAL
    assert lib.dp_unit_backward(p.handle, ws, sh, 1, ug, st, ug, st, 0, mean, 1, None) == dps.DP_EINVAL
    assert "overlaps" in lib.dp_last_error().decode()
    assert lib.dp_unit_backward(p.handle, ws, sh, 1, gb, st, ug, st, 0, C.c_void_p((1 << 30) + 64), 1,
                                None) == dps.DP_EINVAL
    assert lib.dp_unit_backward(p.handle, ws, sh, -1, gb, st, ug, st, -1, mean, 1, None) == dps.DP_OK
    assert lib.dp_unit_backward(None, ws, sh, 0, gb, st, ug, st, 1, mean, 1, None) == dps.DP_EINVAL


def test_launch_counts():
    assert dps.dp_fused_zero_step_launches(dps.adamw_cfg(max_norm=0.0)) == 1
    assert dps.dp_fused_zero_step_launches(dps.adamw_cfg(max_norm=1.0)) == 3


def test_empty_plan_accepts_null_pointers():
    """An empty plan touches no memory: NULL device pointers are accepted and no
    kernel is launched."""
    lib = dps.lib()
    p = dps.Plan([], 1024, 4)
    ws = C.c_void_p(1 << 20)
    assert lib.dp_allreduce_mean(p.handle, ws, None, 0, 0, None) == dps.DP_OK
    assert lib.dp_all_gather(p.handle, ws, None, 0, 0, None) == dps.DP_OK


NOALLOC_BYTES = 32 << 20


def noalloc_need(plan):
    """Bytes of the no-alloc call's static array a plan uses: the workspace
    without its fp32 stage [L] (device tables and per-tile norm partials)."""
    return plan.info.workspace_bytes - (-(-4 * plan.L // 256) * 256)


def test_noalloc_refuses_oversized_plans_on_the_host():
    """dp_clip_coef_noalloc checks the static array's size before any device work."""
    lib = dps.lib()
    plan = dps.Plan([1 << 30, 1 << 30], 25 << 20, 8)
    ok = C.c_void_p(1 << 21)
    rc = lib.dp_clip_coef_noalloc(plan.handle, ok, ok, C.c_double(1.0), ok, ok, None)
    assert rc == dps.DP_EINVAL
    msg = lib.dp_last_error().decode()
    assert "static array holds 33554432 bytes" in msg
    assert f"the plan needs {noalloc_need(plan)} bytes" in msg
    assert lib.dp_clip_coef_noalloc(plan.handle, ok, ok, C.c_double(1.0), None, ok,
                                    None) == dps.DP_EINVAL


def test_noalloc_size_limit_at_the_boundary():
    """The bench's 1.1B-parameter plan fits the static array, the 2.65B plan does
    not, and a one-tensor plan one tile past the largest that fits is refused
    (the calls that would pass the check are not made: they would launch)."""
    lib = dps.lib()
    ok = C.c_void_p(1 << 21)
    llama = configs.llama_1b1_zero2()
    assert noalloc_need(dps.Plan(llama.sizes, llama.bucket_bytes, llama.P)) <= NOALLOC_BYTES
    big = configs.gpt_2b5_clip()
    p_big = dps.Plan(big.sizes, big.bucket_bytes, big.P)
    assert noalloc_need(p_big) > NOALLOC_BYTES
    assert lib.dp_clip_coef_noalloc(p_big.handle, ok, ok, C.c_double(1.0), ok, ok,
                                    None) == dps.DP_EINVAL
    tile = 8192
    lo, hi = 1, 1 << 20                   # in tiles of one tensor
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if noalloc_need(dps.Plan([mid * tile], 1 << 40, 2)) <= NOALLOC_BYTES:
            lo = mid
        else:
            hi = mid
    fits, over = dps.Plan([lo * tile], 1 << 40, 2), dps.Plan([hi * tile], 1 << 40, 2)
    assert noalloc_need(fits) <= NOALLOC_BYTES < noalloc_need(over)
    assert 1.15e9 < lo * tile < 1.3e9                      # "about 1.2e9 parameters"
    assert lib.dp_clip_coef_noalloc(over.handle, ok, ok, C.c_double(1.0), ok, ok,
                                    None) == dps.DP_EINVAL
    assert f"the plan needs {noalloc_need(over)} bytes" in lib.dp_last_error().decode()


@pytest.mark.parametrize("R,S", [(2, 4), (4, 2), (8, 1), (1, 8), (3, 2)])
def test_mesh_plan_layout(orc, R, S):
    """A mesh plan has the flat P = R*S layout; its shards are len/S."""
    wl = configs.tiny_plumbing()
    P = R * S
    p = dps.Plan(wl.sizes, wl.bucket_bytes, P, mesh=(R, S))
    q = dps.Plan(wl.sizes, wl.bucket_bytes, P)
    assert (p.info.R, p.info.S, p.P) == (R, S, P) and (q.info.R, q.info.S) == (1, P)
    assert p.tensor_offsets() == q.tensor_offsets() and p.L == q.L
    for b in range(p.n_buckets):
        off, ln, sh = p.bucket(b)
        assert sh * S == ln and (ln // S) % (16 * R) == 0 or R == 1


def test_mesh_plan_rejects_bad_shapes():
    with pytest.raises(ValueError):
        dps.Plan([10], 1024, 8, mesh=(3, 2))
    with pytest.raises(dps.DPError):
        dps.Plan([10], 1024, 128, mesh=(16, 8))


def test_binding_rejects_wrong_buffers_before_any_call():
    """The binding checks dtype, device, contiguity and size of every buffer and
    raises before the library is called (no GPU needed to see it)."""
    import torch
    plan = dps.Plan([1000, 70000], 64 * 1024, 4)
    ws = torch.zeros(plan.info.workspace_bytes, dtype=torch.uint8)
    g = torch.zeros(plan.P, plan.stride, dtype=torch.bfloat16)          # host tensor
    with pytest.raises(ValueError, match="CUDA tensor"):
        dps.dp_allreduce_mean(plan, ws, g)
    with pytest.raises(TypeError, match="must be a torch.Tensor"):
        dps.dp_allreduce_mean(plan, ws, g.float().numpy())
    with pytest.raises(ValueError, match="does not multiply"):
        dps.Plan([1000], 1 << 20, 8, mesh=(3, 2))
    with pytest.raises(dps.DPError) as e:
        dps.Plan([1000], 1 << 20, 65)
    assert e.value.code == dps.DP_EINVAL


def test_stream_launch_shape_registry():
    """dp_stream_set_launch / dp_stream_get_launch keep a shape per stream handle on
    the host (no device work): set, read back, reset, other handles untouched, NULL
    (the legacy default stream) allowed, unknown shapes refused."""
    lib = dps.lib()
    a, b = C.c_void_p(0x5000), C.c_void_p(0x6000)
    out = C.c_int32(-1)

    def get(h):
        assert lib.dp_stream_get_launch(h, C.byref(out)) == 0
        return out.value

    assert get(a) == dps.DP_LAUNCH_DEFAULT and get(None) == dps.DP_LAUNCH_DEFAULT
    assert lib.dp_stream_set_launch(a, dps.DP_LAUNCH_SHORT_CTAS) == 0
    assert get(a) == dps.DP_LAUNCH_SHORT_CTAS and get(b) == dps.DP_LAUNCH_DEFAULT
    assert lib.dp_stream_set_launch(None, dps.DP_LAUNCH_SHORT_CTAS) == 0
    assert get(None) == dps.DP_LAUNCH_SHORT_CTAS
    for bad in (2, -1, 7):
        assert lib.dp_stream_set_launch(a, bad) == dps.DP_EINVAL
        assert b"unknown launch shape" in lib.dp_last_error()
    assert get(a) == dps.DP_LAUNCH_SHORT_CTAS          # a refused call changes nothing
    assert lib.dp_stream_get_launch(a, None) == dps.DP_EINVAL
    assert lib.dp_stream_set_launch(a, dps.DP_LAUNCH_DEFAULT) == 0
    assert lib.dp_stream_set_launch(None, dps.DP_LAUNCH_DEFAULT) == 0
    assert get(a) == dps.DP_LAUNCH_DEFAULT and get(None) == dps.DP_LAUNCH_DEFAULT
    assert dps.DP_LAUNCH_PERSISTENT == dps.DP_LAUNCH_DEFAULT == 0   # the older name
    assert dps.stream_launch(0x5000) is False
    dps.set_stream_launch(0x5000, True)
    assert dps.stream_launch(0x5000) is True
    dps.set_stream_launch(0x5000, False)
    assert dps.stream_launch(0x5000) is False

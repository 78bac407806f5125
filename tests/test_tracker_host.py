"""Bucket readiness tracker, host logic (dry run: no launches, no GPU).

DDP fires a bucket's collective once every gradient in it is ready, buckets in
the same order every step; a gradient that never becomes ready hangs DDP — the
tracker reports it instead ("4.1 Data parallelism in depth", sec. 4.2)."""
import random
import threading

import pytest

import gradient_sync_zero_gb300 as dps
from gradient_sync_zero_gb300 import build as dbuild
from workloads import configs


@pytest.fixture(scope="module", autouse=True)
def built():
    dbuild.build()


def dry(sizes, cap, P):
    plan = dps.Plan(sizes, cap, P)
    return plan, dps.Tracker(plan, dps.DP_TRACK_ALLREDUCE, dry_run=True)


def test_backward_order_fires_every_bucket_in_plan_order():
    wl = configs.gpt2_small_allreduce()
    plan, tr = dry(wl.sizes, wl.bucket_bytes, wl.P)
    tr.begin()
    for t in reversed(range(len(wl.sizes))):          # backward: last layer first
        tr.mark_ready(t)
    tr.wait(1000)
    assert tr.fired() == list(range(plan.n_buckets))


def test_bucket_fires_exactly_when_complete():
    sizes = [1000, 1000, 1000, 1000]                   # reverse packing: buckets {3,2}, {1,0}
    plan, tr = dry(sizes, 4000, 2)
    assert plan.n_buckets == 2 and [plan.tensor(t)[0] for t in range(4)] == [1, 1, 0, 0]
    tr.begin()
    tr.mark_ready(3)
    assert tr.fired() == []
    tr.mark_ready(2)
    assert tr.fired() == [0]
    tr.mark_ready(0)
    assert tr.fired() == [0]
    tr.mark_ready(1)
    assert tr.fired() == [0, 1]


def test_later_bucket_waits_for_earlier_ones():
    """A later bucket that completes first is held until the buckets before it
    have fired, so the launch order is the same every step."""
    sizes = [1000, 1000, 1000, 1000]
    plan, tr = dry(sizes, 4000, 2)
    tr.begin()
    tr.mark_ready(0)
    tr.mark_ready(1)                                   # bucket 1 complete, bucket 0 not
    assert tr.fired() == []
    tr.mark_ready(3)
    tr.mark_ready(2)
    assert tr.fired() == [0, 1]


def test_missing_gradient_times_out_with_its_name():
    sizes = [10, 20, 30, 40]
    plan, tr = dry(sizes, 64, 1)
    tr.begin()
    for t in (3, 2, 0):
        tr.mark_ready(t)
    with pytest.raises(dps.DPError) as e:
        tr.wait(50)
    assert e.value.code == dps.DP_ETIMEOUT
    msg = str(e.value)
    assert "1 tensor(s) never marked ready: 1" in msg


def test_double_mark_and_range_are_rejected_and_begin_resets():
    plan, tr = dry([10, 20], 1 << 20, 2)
    tr.begin()
    tr.mark_ready(1)
    with pytest.raises(dps.DPError) as e:
        tr.mark_ready(1)
    assert e.value.code == dps.DP_EINVAL
    with pytest.raises(dps.DPError):
        tr.mark_ready(2)
    tr.mark_ready(0)
    tr.wait(100)
    assert tr.fired() == [0]
    tr.begin()
    assert tr.fired() == []
    tr.mark_ready(0)
    tr.mark_ready(1)
    tr.wait(100)
    assert tr.fired() == [0]


def test_concurrent_marking_from_many_threads():
    wl = configs.sweep_small_tensors(64 * 1024)
    plan, tr = dry(wl.sizes, wl.bucket_bytes, wl.P)
    order = list(range(len(wl.sizes)))
    random.Random(3).shuffle(order)
    chunks = [order[i::8] for i in range(8)]
    errors = []

    def work(ts):
        try:
            for t in ts:
                tr.mark_ready(t)
        except Exception as e:  # noqa: BLE001
            errors.append(e)

    for step in range(2):
        tr.begin()
        th = [threading.Thread(target=work, args=(c,)) for c in chunks]
        for x in th:
            x.start()
        for x in th:
            x.join()
        assert not errors
        tr.wait(5000)
        assert tr.fired() == list(range(plan.n_buckets))


def test_create_validates_buffers():
    plan = dps.Plan([1000], 1 << 20, 4)
    lib = dps.lib()
    import ctypes as C
    h = C.c_void_p()
    assert lib.dp_tracker_create(plan.handle, 0, None, None, None, None, 0, 0,
                                 C.byref(h)) == dps.DP_EINVAL
    ok, odd = C.c_void_p(1 << 20), C.c_void_p((1 << 20) + 8)
    assert lib.dp_tracker_create(plan.handle, 0, ok, odd, None, None, 0, 0,
                                 C.byref(h)) == dps.DP_EALIGN
    assert lib.dp_tracker_create(plan.handle, 1, ok, ok, None, None, 0, 0,
                                 C.byref(h)) == dps.DP_EINVAL    # reduce-scatter needs `mean`
    assert lib.dp_tracker_create(plan.handle, 7, ok, ok, ok, None, 0, 0,
                                 C.byref(h)) == dps.DP_EINVAL
    for bad_flags in (4, 8, -1):                      # bits other than DRY_RUN | SHORT_CTAS
        assert lib.dp_tracker_create(plan.handle, 0, None, None, None, None, 0,
                                     dps.DP_TRACK_DRY_RUN | bad_flags, C.byref(h)) == dps.DP_EINVAL
        assert b"unknown flags" in lib.dp_last_error()
    assert lib.dp_tracker_create(plan.handle, 0, None, None, None, None, 0,
                                 dps.DP_TRACK_DRY_RUN | dps.DP_TRACK_SHORT_CTAS, C.byref(h)) == 0
    lib.dp_tracker_free(h)


def test_set_micro_rules():
    """Accumulation mode: flat plans only, 32-byte aligned, and not in the middle
    of a step (some but not all buckets fired)."""
    import ctypes as C
    sizes = [1000, 1000, 1000, 1000]
    plan, tr = dry(sizes, 4000, 2)
    lib = dps.lib()
    assert lib.dp_tracker_set_micro(tr._h, C.c_void_p(1 << 20)) == dps.DP_OK
    assert lib.dp_tracker_set_micro(tr._h, C.c_void_p((1 << 20) + 16)) == dps.DP_EALIGN
    tr.begin()
    tr.mark_ready(3)
    tr.mark_ready(2)                                   # bucket 0 fired, bucket 1 not
    assert tr.fired() == [0]
    assert lib.dp_tracker_set_micro(tr._h, None) == dps.DP_EINVAL
    tr.mark_ready(1)
    tr.mark_ready(0)
    assert lib.dp_tracker_set_micro(tr._h, None) == dps.DP_OK   # step complete
    mesh = dps.Plan(sizes, 4000, 4, mesh=(2, 2))
    trm = dps.Tracker(mesh, dps.DP_TRACK_ALLREDUCE, dry_run=True)
    assert lib.dp_tracker_set_micro(trm._h, C.c_void_p(1 << 20)) == dps.DP_EINVAL


def test_unused_parameters_marked_after_forward_let_the_bucket_fire():
    """find_unused_parameters: a tensor the step did not use is marked ready up
    front (its gradient slots zeroed by the caller); its bucket then fires as soon
    as the used tensors are ready, instead of timing out."""
    sizes = [1000, 1000, 1000, 1000]
    plan, tr = dry(sizes, 4000, 2)                      # buckets {3,2}, {1,0}
    tr.begin()
    tr.mark_ready(2)                                   # tensor 2 unused this step
    tr.mark_ready(3)
    assert tr.fired() == [0]
    tr.mark_ready(1)
    tr.mark_ready(0)
    tr.wait(100)
    assert tr.fired() == [0, 1]


def test_set_zero_step_rules():
    """DP_TRACK_ZERO_STEP: the targets and AdamW settings of each bucket's whole
    step.  Refused in another mode, with clipping (the global norm must precede
    every update), with NULL or misaligned pointers, with a micro-batch buffer,
    and in the middle of a step; `mean` is not needed to create the tracker."""
    import ctypes as C
    sizes = [1000, 1000, 1000, 1000]
    plan = dps.Plan(sizes, 4000, 2)
    lib = dps.lib()
    ok, odd = C.c_void_p(1 << 20), C.c_void_p((1 << 20) + 8)
    h = C.c_void_p()
    assert lib.dp_tracker_create(plan.handle, dps.DP_TRACK_ZERO_STEP, ok, ok, None, None, 0, 0,
                                 C.byref(h)) == dps.DP_OK
    lib.dp_tracker_free(h)
    cfg = dps.adamw_cfg(max_norm=0.0, step=1)
    clipped = dps.adamw_cfg(max_norm=1.0, step=1)
    _, ar = dry(sizes, 4000, 2)
    assert lib.dp_tracker_set_zero_step(ar._h, ok, ok, ok, ok, C.byref(cfg)) == dps.DP_EINVAL
    tr = dps.Tracker(plan, dps.DP_TRACK_ZERO_STEP, dry_run=True)
    assert lib.dp_tracker_set_zero_step(tr._h, ok, ok, ok, ok, C.byref(clipped)) == dps.DP_EINVAL
    assert lib.dp_tracker_set_zero_step(tr._h, ok, ok, ok, ok, None) == dps.DP_EINVAL
    assert lib.dp_tracker_set_zero_step(tr._h, ok, None, ok, ok, C.byref(cfg)) == dps.DP_EINVAL
    assert lib.dp_tracker_set_zero_step(tr._h, ok, ok, odd, ok, C.byref(cfg)) == dps.DP_EALIGN
    assert lib.dp_tracker_set_zero_step(tr._h, ok, ok, ok, ok, C.byref(cfg)) == dps.DP_OK
    assert lib.dp_tracker_set_micro(tr._h, ok) == dps.DP_EINVAL       # no accumulation here
    tr.begin()
    tr.mark_ready(3)
    tr.mark_ready(2)                                   # bucket 0 fired, bucket 1 not
    assert tr.fired() == [0]
    step2 = dps.adamw_cfg(max_norm=0.0, step=2)
    assert lib.dp_tracker_set_zero_step(tr._h, ok, ok, ok, ok, C.byref(step2)) == dps.DP_EINVAL
    tr.mark_ready(1)
    tr.mark_ready(0)
    assert lib.dp_tracker_set_zero_step(tr._h, ok, ok, ok, ok, C.byref(step2)) == dps.DP_OK


class _Ev:
    """Stands in for a torch.cuda.Event in dry runs (only its handle is passed)."""

    def __init__(self, handle):
        self.cuda_event = handle


def test_range_mark_fires_completed_buckets_as_one_launch():
    """One mark that completes several buckets fires them together, in plan order,
    as one launch; its stream waits once per distinct event."""
    sizes = [1000] * 8                                  # reverse packing: 4 buckets of 2
    plan, tr = dry(sizes, 4000, 2)
    assert plan.n_buckets == 4
    tr.begin()
    tr.mark_ready_range(4, 8, _Ev(0x1000))              # buckets 0 and 1 complete
    assert tr.fired() == [0, 1]
    assert tr.stats() == (1, 1)
    tr.mark_ready_range(2, 4, _Ev(0x2000))              # bucket 2
    assert tr.stats() == (2, 2)
    tr.mark_ready(1, _Ev(0x3000))
    tr.mark_ready(0, _Ev(0x4000))                       # bucket 3: two events, two waits
    tr.wait(1000)
    assert tr.fired() == [0, 1, 2, 3]
    assert tr.stats() == (3, 4)
    tr.begin()
    assert tr.stats() == (0, 0)


def test_short_ctas_launch_every_bucket_on_its_own():
    """DP_TRACK_SHORT_CTAS: a mark that completes several buckets still waits once
    per distinct event, but launches each bucket separately, in plan order."""
    sizes = [1000] * 8
    plan = dps.Plan(sizes, 4000, 2)
    tr = dps.Tracker(plan, dps.DP_TRACK_ALLREDUCE, dry_run=True, short_ctas=True)
    tr.begin()
    tr.mark_ready_range(4, 8, _Ev(0x1000))              # buckets 0 and 1: one wait, two launches
    assert tr.fired() == [0, 1] and tr.stats() == (2, 1)
    tr.mark_ready_range(0, 4)                           # buckets 2 and 3, no event
    tr.wait(1000)
    assert tr.fired() == [0, 1, 2, 3] and tr.stats() == (4, 1)


def test_range_mark_held_back_and_released_together():
    """Buckets completed out of order are held, then fire in one launch when the
    first of them completes."""
    sizes = [1000] * 8
    plan, tr = dry(sizes, 4000, 2)
    tr.begin()
    tr.mark_ready_range(0, 6)                           # buckets 1, 2, 3 complete; 0 is not
    assert tr.fired() == [] and tr.stats() == (0, 0)
    tr.mark_ready_range(6, 8)
    assert tr.fired() == [0, 1, 2, 3] and tr.stats() == (1, 0)


def test_range_mark_rejections_leave_nothing_marked():
    sizes = [1000] * 8
    plan, tr = dry(sizes, 4000, 2)
    tr.begin()
    tr.mark_ready(5)
    with pytest.raises(dps.DPError) as e:
        tr.mark_ready_range(4, 8)                       # tensor 5 already marked
    assert e.value.code == dps.DP_EINVAL and "tensor 5" in str(e.value)
    with pytest.raises(dps.DPError):
        tr.mark_ready_range(6, 9)                       # outside [0, 8)
    with pytest.raises(dps.DPError):
        tr.mark_ready_range(3, 2)
    tr.mark_ready_range(6, 8)                           # 4 and 7 were not marked by the refusals
    tr.mark_ready(4)
    assert tr.fired() == [0, 1]


def test_batch_mark_keeps_per_tensor_events_apart():
    """dp_tracker_mark_ready_batch: one call, each tensor its own event.  A bucket
    whose tensors carry different events goes out alone (it must not wait for a
    later bucket's readiness); buckets whose tensors share one event go out
    together."""
    sizes = [1000] * 8                                  # 4 buckets: {7,6} {5,4} {3,2} {1,0}
    plan, tr = dry(sizes, 4000, 2)
    tr.begin()
    evs = [_Ev(0x100 * (t + 1)) for t in range(8)]
    tr.mark_ready_batch([7, 6, 5, 4], [evs[t] for t in (7, 6, 5, 4)])
    assert tr.fired() == [0, 1]
    assert tr.stats() == (2, 4)                          # two launches, one wait per event
    shared = _Ev(0x9000)
    tr.mark_ready_batch([3, 2, 1, 0], [shared] * 4)     # both buckets: one event
    assert tr.fired() == [0, 1, 2, 3]
    assert tr.stats() == (3, 5)
    tr.wait(1000)


def test_batch_mark_rejections_leave_nothing_marked():
    sizes = [1000] * 8
    plan, tr = dry(sizes, 4000, 2)
    tr.begin()
    tr.mark_ready(2)
    for bad in ([7, 6, 7], [7, 2], [7, 8], [-1]):
        with pytest.raises(dps.DPError) as e:
            tr.mark_ready_batch(bad)
        assert e.value.code == dps.DP_EINVAL
    tr.mark_ready_batch([7, 6])                         # none of them was left marked
    assert tr.fired() == [0]
    with pytest.raises(ValueError):
        tr.mark_ready_batch([5, 4], [_Ev(1)])
    tr.mark_ready_batch([5, 4, 3, 1, 0])
    tr.wait(1000)
    assert tr.fired() == [0, 1, 2, 3]


def test_batch_refusal_messages():
    sizes = [1000] * 4
    plan, tr = dry(sizes, 4000, 2)
    tr.begin()
    with pytest.raises(dps.DPError, match="listed twice"):
        tr.mark_ready_batch([1, 1])
    tr.mark_ready(3)
    with pytest.raises(dps.DPError, match="already marked"):
        tr.mark_ready_batch([2, 3])
    with pytest.raises(dps.DPError, match="outside"):
        tr.mark_ready_batch([4])


def test_side_stream_rules_in_a_dry_run():
    """A side stream changes where buckets run, not the firing order; it cannot be
    changed while a step has fired some but not all buckets."""
    sizes = [1000] * 8
    plan, tr = dry(sizes, 4000, 2)
    tr.set_side_stream(0x1234, 16)           # dry run: nothing is launched on it
    tr.begin()
    tr.mark_ready_range(4, 8)
    with pytest.raises(dps.DPError, match="in progress"):
        tr.set_side_stream(None)
    with pytest.raises(dps.DPError):
        tr.set_side_stream(0x1234, -1)
    tr.mark_ready_range(0, 4)
    tr.wait(1000)
    assert tr.fired() == [0, 1, 2, 3]
    tr.set_side_stream(None)

"""Index checks and the bounded wait on the GPU.

The library built with -DDPSYNC_CHECKED runs the GPU parity suites (in a child
process with DPSYNC_VARIANT=checked, where every test must end with no failed
check); a workspace whose last tile descriptor runs one 32-byte block past the
plan is caught and skipped by that build; the bounded mbarrier wait times out into
a status the host reads, with the context still usable."""
import os
import subprocess
import sys

import pytest
import torch

import gradient_sync_zero_gb300 as dps

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CHECKED = os.environ.get("DPSYNC_VARIANT") == "checked"


@pytest.mark.skipif(CHECKED, reason="this test starts the checked run")
def test_parity_suites_under_index_checks():
    from gradient_sync_zero_gb300 import build as dbuild
    dbuild.build(checked=True)
    env = dict(os.environ, DPSYNC_VARIANT="checked")
    suites = ["tests/test_parity_gpu.py", "tests/test_parity_mesh.py", "tests/test_zero3_gpu.py",
              "tests/test_accum_gpu.py", "tests/test_tracker_gpu.py", "tests/test_graph_gpu.py",
              "tests/test_fuzz_gpu.py", "tests/test_staged_owner_rows_gpu.py", "tests/test_checked_gpu.py"]
    r = subprocess.run([sys.executable, "-m", "pytest", "-m", "gpu", "-x", "-q",
                        "-p", "no:cacheprovider", *suites],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    import re
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and int(m.group(1)) >= 150 and " failed" not in r.stdout, r.stdout[-2000:]


@pytest.mark.plants_bad_descriptor
@pytest.mark.skipif(not CHECKED, reason="only the checked build guards a bad descriptor")
def test_descriptor_past_the_plan_is_caught():
    """The last tile is made one block longer than the plan.  Even unchecked, that
    block lies inside the replica stride's slack (at least 128 elements past L),
    so no access could leave the buffer; the checked build counts and skips it."""
    assert dps.dp_bounds_violations(reset=True) == 0
    plan = dps.Plan([1000, 4096, 333], 8192, 4)
    assert plan.stride - plan.L >= 128
    ws = plan.new_workspace()
    g = plan.new_replicas()
    g.normal_()
    ref = g.clone()
    hdr = ws[:192].cpu()
    off_tiles = int(hdr[48:56].view(torch.int64))
    n_tiles = int(hdr[24:32].view(torch.int64))
    last = off_tiles + 32 * (n_tiles - 1)
    nvec = int(ws[last + 16:last + 20].cpu().view(torch.int32))
    ws[last + 16:last + 20].copy_(torch.tensor([nvec + 2], dtype=torch.int32).view(torch.uint8))
    dps.dp_allreduce_mean(plan, ws, g)
    torch.cuda.synchronize()
    assert dps.dp_bounds_violations(reset=True) >= 1
    # the bad tile was skipped whole: its elements still hold the inputs
    v0 = int(ws[last:last + 8].cpu().view(torch.int64))
    assert torch.equal(g[:, 8 * v0:plan.L], ref[:, 8 * v0:plan.L])
    assert torch.equal(g[:, plan.L:], ref[:, plan.L:])


def test_bounded_wait_times_out_into_a_status():
    st, ms = dps.dp_selftest_bounded_wait(limit_ns=20_000_000)      # 20 ms
    assert st == dps.DP_STATUS_TIMEOUT
    assert 20 <= ms < 2000
    x = torch.arange(1024, device="cuda", dtype=torch.float32)       # the context still works
    assert float(x.sum()) == 1023 * 1024 / 2
    with pytest.raises(dps.DPError):
        dps.dp_selftest_bounded_wait(limit_ns=10)

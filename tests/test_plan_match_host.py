"""Cross-process plan check on the CPU: every rank must build the same buckets in
the same order ("4.1 Data parallelism in depth", sec. 4.2; "Data Parallelism:
DDP, ZeRO and FSDP", "DDP, and why it works"), or the ranks' collectives stop
lining up.  dp_plan_fingerprint / dp_plan_check_match turn a mismatch into
DP_EPLAN; here they are checked against a Python restatement of the documented
fingerprint format, for sensitivity to every layout field, and across two gloo
ranks of which one built a different plan."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

import gradient_sync_zero_gb300 as dps

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SIZES = [3, 1000, 65536, 131071, 262144, 262144, 279105]   # the 7-tensor plumbing case
CAP = 1 << 20


def _fnv_words(words):
    """64-bit FNV-1a over 8-byte little-endian words (the header's format)."""
    h = 0xcbf29ce484222325
    for w in words:
        for byte in (int(w) & (2**64 - 1)).to_bytes(8, "little"):
            h ^= byte
            h = (h * 0x100000001b3) & (2**64 - 1)
    return h


def _expected(plan, decay):
    info = plan.info
    words = [0x31544e4946504c44, info.P, info.R, info.S, plan.L, len(plan.sizes)]
    for t, size in enumerate(plan.sizes):
        b, off = plan.tensor(t)
        words += [size, 1 if decay[t] else 0, off, b]
    words.append(plan.n_buckets)
    for b in range(plan.n_buckets):
        off, n, _ = plan.bucket(b)
        words += [off, n]
    return _fnv_words(words)


@pytest.mark.parametrize("P,mesh", [(4, None), (8, None), (8, (2, 4)), (16, (4, 4))])
def test_fingerprint_follows_the_documented_format(P, mesh):
    decay = [t % 3 != 0 for t in range(len(SIZES))]
    plan = dps.Plan(SIZES, CAP, P, decay=decay, mesh=mesh)
    assert plan.fingerprint == _expected(plan, decay)


def test_equal_layouts_give_equal_fingerprints():
    a = dps.Plan(SIZES, CAP, 4)
    assert dps.Plan(SIZES, CAP, 4).fingerprint == a.fingerprint
    # the replica stride is each process's own
    assert dps.Plan(SIZES, CAP, 4, replica_stride=a.stride + 4096).fingerprint == a.fingerprint
    # two caps that both hold the whole model give the same single bucket
    big = dps.Plan(SIZES, 64 << 20, 4)
    assert big.n_buckets == 1
    assert dps.Plan(SIZES, 128 << 20, 4).fingerprint == big.fingerprint


def test_every_layout_change_changes_the_fingerprint():
    base = dps.Plan(SIZES, CAP, 8)
    variants = {
        "one size": dps.Plan(SIZES[:-1] + [SIZES[-1] + 1], CAP, 8),
        "one decay flag": dps.Plan(SIZES, CAP, 8, decay=[1] * 6 + [0]),
        "rank count": dps.Plan(SIZES, CAP, 4),
        "mesh": dps.Plan(SIZES, CAP, 8, mesh=(2, 4)),
        "bucket cap": dps.Plan(SIZES, CAP // 2, 8),
        "tensor order": dps.Plan(SIZES[1:] + SIZES[:1], CAP, 8),
        "one tensor fewer": dps.Plan(SIZES[:-1], CAP, 8),
    }
    seen = {base.fingerprint}
    for name, plan in variants.items():
        assert plan.fingerprint not in seen, name
        seen.add(plan.fingerprint)


def test_check_match_names_the_rank_and_rejects_bad_lists():
    a, b = dps.Plan(SIZES, CAP, 4), dps.Plan(SIZES, CAP // 2, 4)
    a.check_match([])
    a.check_match([a.fingerprint] * 3)
    with pytest.raises(dps.DPError) as e:
        a.check_match([a.fingerprint, a.fingerprint, b.fingerprint])
    assert e.value.code == dps.DP_EPLAN and "rank 2" in str(e.value)
    lib = dps.lib()
    assert lib.dp_plan_check_match(a.handle, None, 2) == dps.DP_EINVAL
    assert lib.dp_plan_check_match(a.handle, None, -1) == dps.DP_EINVAL
    assert lib.dp_plan_check_match(None, None, 0) == dps.DP_EINVAL
    assert lib.dp_plan_fingerprint(a.handle, None) == dps.DP_EINVAL


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, differ, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import gradient_sync_zero_gb300 as lib
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sizes = list(SIZES)
    if differ and rank == 1:
        sizes[2] += 8                     # rank 1 built its plan from another model
    plan = lib.Plan(sizes, CAP, 4)
    try:
        lib.check_plans_match(plan)
        out[rank] = "ok"
    except lib.DPError as e:
        out[rank] = f"code {e.code}"
    dist.destroy_process_group()


@pytest.mark.parametrize("differ", [False, True])
def test_two_gloo_ranks_agree_or_both_refuse(differ):
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, differ, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    want = f"code {dps.DP_EPLAN}" if differ else "ok"
    assert dict(out) == {0: want, 1: want}

"""Host logic of bench.py on the CPU: max-over-ranks timing with two gloo ranks,
the reference (CPU oracle) arm, and the clock-sample parser."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    got = bench.max_over_ranks(10.0 + rank * 5.0, world)
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def _run_bench(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_json_line():
    r = _run_bench(["--impl", "reference", "--steps", "2", "--warmup", "1",
                    "--workload", "tiny-P4-1M"])
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "params/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0",
                    "--workload", "tiny-P4-1M"], {"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_clock_summary_parser():
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(0)
    c.lines = ["0, 1950, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Active",
               "0, 1980, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 2000, 2070, 990.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    s = c.summary()
    assert s["sm_mhz"] == 1980 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    assert bench.ClockSampler(0).summary()["reasons"] == ["unsampled"]


def test_workload_names_resolve():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.workload_by_name("llama-1.1B-P8-zero2").P == 8
    with pytest.raises(SystemExit):
        bench.workload_by_name("nope")


def test_reference_arm_times_the_allreduce_for_allreduce_workloads(monkeypatch):
    """An all-reduce workload's reference arm times the oracle's mean all-reduce and
    names the all-reduce metric (the plumbing shapes, switched to all-reduce mode)."""
    import argparse
    import dataclasses
    sys.path.insert(0, ROOT)
    import bench
    from workloads import configs
    wl = dataclasses.replace(configs.tiny_plumbing(), name="tiny-P4-1M-allreduce", mode="allreduce")
    monkeypatch.setattr(bench, "workload_by_name", lambda name: wl)
    calls = []
    import oracle
    orc = oracle.default()
    real = orc.allreduce_mean
    monkeypatch.setattr(orc, "allreduce_mean", lambda *a, **k: calls.append(1) or real(*a, **k))
    monkeypatch.setattr(orc, "zero_step", lambda *a, **k: pytest.fail("zero step timed"))
    monkeypatch.setattr(oracle, "default", lambda: orc)
    d = bench.run_reference(argparse.Namespace(steps=2, warmup=1, workload=wl.name), 0, 1)
    assert len(calls) == 3
    assert d["metric"] == "bucketed mean all-reduce params/s" and d["value"] > 0
    assert "all-reduce" in d["cpu_baseline"]["sample"]
    json.dumps(d)


def test_oracle_allreduce_rate_on_host_buffers():
    """The all-reduce CPU baseline gathers the tensors out of the padded replica
    layout and times whole passes of the oracle's ring, at least one and at most
    max_passes."""
    import dataclasses
    sys.path.insert(0, ROOT)
    import bench
    import gradient_sync_zero_gb300 as dps
    from workloads import configs
    wl = dataclasses.replace(configs.tiny_plumbing(), name="tiny-P4-1M-allreduce", mode="allreduce")
    plan = dps.Plan(wl.sizes, wl.bucket_bytes, wl.P)
    grads = plan.new_replicas(device="cpu")
    grads.normal_(0.0, 1e-3)
    rate, n, secs, thr, desc = bench.oracle_allreduce_rate(wl, plan.tensor_offsets(), grads,
                                                           budget_s=0.0, max_passes=2)
    assert n == wl.n_params and secs > 0 and rate == n / secs and thr >= 1
    assert desc.startswith("1 pass(es)")
    _, _, _, _, desc2 = bench.oracle_allreduce_rate(wl, plan.tensor_offsets(), grads,
                                                    budget_s=1e9, max_passes=2)
    assert desc2.startswith("2 pass(es)")


def test_layer_groups_cover_every_tensor_once():
    """--streamed --mark layer: one mark per layer, tensors in order, none lost."""
    import bench
    from workloads import configs
    for wl, n_groups in ((configs.gpt2_small_allreduce(), 16), (configs.llama_1b1_zero2(), 25)):
        g = bench.layer_groups(wl.names)
        assert len(g) == n_groups
        assert g[0][0] == 0 and g[-1][1] == len(wl.names)
        assert all(a[1] == b[0] for a, b in zip(g, g[1:]))
        for g0, g1 in g:
            keys = {".".join(n.split(".")[:2]) for n in wl.names[g0:g1]}
            assert len(keys) == 1


def test_traffic_record_from_an_ncu_csv(tmp_path):
    """--traffic-record: per kernel the mean read + write bytes of its launches,
    scaled by parameters from the captured workload, with the current kernel hash;
    bench.py's roofline reads it back."""
    import json as js
    import bench
    hdr = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
           '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
           '"Metric Value"')
    rows = []
    for i, (name, rd, wr) in enumerate([("void k_reduce_scatter<8, 0, 0, 0, 256>(KCommon)", 1000, 200),
                                        ("k_norm_finalize(KCommon, double)", 5, 0),
                                        ("void k_adamw_all_gather<0, 2048, 2>(KCommon)", 3000, 5000),
                                        ("void k_reduce_scatter<8, 0, 0, 0, 256>(KCommon)", 1002, 198)]):
        for metric, unit, v in (("dram__bytes_read.sum", "Mbyte", rd), ("dram__bytes_write.sum", "Mbyte", wr),
                                ("gpu__time_duration.sum", "ns", 100)):
            rows.append(f'"{i}","1","python","h","{name}","1","7","(256, 1, 1)","(456, 1, 1)","0",'
                        f'"10.3","Command line profiler metrics","{metric}","{unit}","{v}"')
    csv_path = tmp_path / "dram.csv"
    csv_path.write_text("==PROF== noise\n" + hdr + "\n" + "\n".join(rows) + "\n")
    out = bench.traffic_record(str(csv_path), "llama-1.1B-P8-zero2", "llama-2L-P8-zero2",
                               ["ncu ..."], out_dir=str(tmp_path))
    text = open(out).read()
    rec = js.loads(text[text.index("{"):])
    scale = 1_100_048_384 / 88_090_624
    rs = rec["llama-1.1B-P8-zero2:reduce_scatter"]
    ag = rec["llama-1.1B-P8-zero2:adamw_all_gather"]
    assert abs(rs["bytes_per_launch"] - 1200e6 * scale) < 1.0
    assert abs(ag["bytes_per_launch"] - 8000e6 * scale) < 1.0
    assert rs["kernel_src_sha"] == bench.kernel_source_hash()
    assert "# ncu ..." in text.replace("#   ", "# ")


def test_kernel_key_maps_ncu_names_of_every_variant():
    """The traffic record and the roofline key ncu's kernel names by what the bench
    times: persistent, small-CTA (the _small suffix or a template flag) and
    bulk-copy variants of one kernel share a key; other kernels have none."""
    import bench
    cases = {
        "void k_adamw_all_gather_small<0, 0>(KCommon, const float *, unsigned char *)": "adamw_all_gather",
        "void k_adamw_all_gather<0, 2048, 2>(KCommon, const float *)": "adamw_all_gather",
        "void k_reduce_scatter<8, 0, 0, 1, 64, 1>(KCommon, const unsigned char *)": "reduce_scatter",
        "void k_reduce_scatter<8, 0, 0, 0, 256>(KCommon)": "reduce_scatter",
        "void k_allreduce<8, 0, 1, 0>(KCommon, unsigned char *)": "allreduce",
        "void k_zero_fused<8, 0, 1, 1>(KCommon)": "zero_fused",
        "k_norm_finalize(KCommon, double)": None,
        "void k_allreduce_accum<8, 1, 0>(KCommon)": None,
        "void k_allreduce_bf16wire<8, 1, 1>(KCommon)": None,
        "void k_replicate_small<1>(KCommon, RepArgs)": None,
    }
    for name, key in cases.items():
        assert bench.kernel_key(name) == key, name

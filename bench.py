"""Throughput bench of the fused ZeRO-2 synchronisation step on GB300.

Default workload: P = 8 virtual ranks, Llama-style 1.1B tensor list (201
tensors, 1,100,048,384 parameters), 25 MiB buckets, bf16 gradients
N(0, 5e-4), AdamW (lr 2e-4, betas 0.9/0.95, eps 1e-8, wd 0.1) with global
gradient-norm clipping at 1.0.  One step = dp_fused_zero_step over all buckets:
reduce-scatter-mean (+ norm partials), clip coefficient, AdamW fused with the
all-gather of bf16 parameters into all 8 replicas.

Prints ONE JSON line (rank 0).  `value` is parameters synchronised per second
over all GPUs (inputs resident in HBM, CUDA events, max over ranks); `e2e`
repeats the step through the same call with the gradients copied in from
pinned host memory and the norm read back every step; `roofline` reports the
dominant kernel (AdamW + all-gather) against the measured HBM copy bandwidth;
`cpu_baseline` times the CPU oracle on a bounded sample on this host's cores.

`--impl reference` times only the CPU oracle (the reference implementation of
the method for this build) on the same workload, sample by sample.

Multi-GPU (torchrun): every rank runs an independent replica of the workload on
its own GPU (the method has no inter-GPU exchange here); value = all ranks'
parameters / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import configs, device as wdev, gen  # noqa: E402

KERNEL_BYTES_PER_PARAM = {
    # algorithmic bytes per parameter of each launch (reads + writes)
    "reduce_scatter": lambda P: 2 * P + 4,
    "adamw_all_gather": lambda P: 4 + 12 + 12 + 2 * P,
    "zero_fused": lambda P: 2 * P + 12 + 12 + 2 * P,
    "allreduce": lambda P: 4 * P,
}


def kernel_key(name):
    """KERNEL_BYTES_PER_PARAM's key of an ncu kernel name (k_<key>, with the _small
    suffix of a small-CTA variant or without, then its template or argument
    list), or None."""
    for k in KERNEL_BYTES_PER_PARAM:
        if re.search(rf"\bk_{k}(_small)?[<(]", name):
            return k
    return None


def workload_by_name(name):
    table = {w.name: w for w in (configs.tiny_plumbing(), configs.gpt2_small_allreduce(),
                                 configs.llama_1b1_zero2(), configs.gpt_2b5_clip(),
                                 configs.llama_1b1_zero2(layers=2, embeddings=False))}
    for cap in configs.SWEEP_BUCKETS:
        for mode in ("zero", "allreduce"):
            w = configs.sweep_small_tensors(cap, mode)
            table[w.name] = w
    if name not in table:
        raise SystemExit(f"unknown workload {name}; known: {sorted(table)}")
    return table[name]


# --------------------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- peaks
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# --------------------------------------------------------------------------- ncu traffic
KERNEL_SOURCES = ["kernels.cuh", "kernels_reduce.cu", "kernels_update.cu", "launch.cuh"]


def kernel_source_hash():
    """Hash of the kernel sources' code: comments and whitespace are removed first,
    so an edit to a comment does not retire a DRAM-traffic record."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "gradient_sync_zero_gb300", "csrc", name)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)   # block comments
        src = re.sub(r"//[^\n]*", " ", src)                 # line comments
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def stored_traffic(workload, kernel):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from the
    profiles' DRAM-traffic record of this workload, only if it was taken on the
    current kernel sources."""
    tf = os.path.join(ROOT, "profiles", f"dram_traffic_{workload}.txt")
    if not os.path.exists(tf):
        return None, "no ncu capture recorded for this workload"
    with open(tf) as f:
        text = f.read()
    tdb = json.loads(text[text.index("{"):])     # comment lines, then the JSON record
    rec = tdb.get(f"{workload}:{kernel}")
    if rec is None:
        return None, "no ncu capture for this workload and kernel"
    if rec.get("kernel_src_sha") != kernel_source_hash():
        return None, "kernel changed since the ncu capture"
    return rec["bytes_per_launch"], rec.get("how", "")


_BYTE_UNITS = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12}


def traffic_record(csv_path, target, captured, commands, out_dir=None):
    """Write profiles/dram_traffic_<target>.txt from an ncu CSV of
    dram__bytes_read.sum / dram__bytes_write.sum per launch taken on workload
    `captured`: per kernel, the mean read + write bytes of its launches, scaled by
    parameters from `captured` to `target` (every kernel streams each parameter's
    bytes once, so its traffic grows in proportion).  `commands`: the ncu command
    lines, recorded in the file's header."""
    import csv
    rows = list(csv.reader(open(csv_path)))
    hi = next(i for i, r in enumerate(rows) if r and r[0] == "ID")
    h = rows[hi]
    col = {k: h.index(k) for k in ("ID", "Kernel Name", "Metric Name", "Metric Unit", "Metric Value")}
    launches = {}
    for r in rows[hi + 1:]:
        if len(r) < len(h):
            continue
        name = r[col["Kernel Name"]]
        key = kernel_key(name)
        if key is None or r[col["Metric Name"]] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        v = float(r[col["Metric Value"]].replace(",", "")) * _BYTE_UNITS[r[col["Metric Unit"]]]
        launches.setdefault(key, {}).setdefault(r[col["ID"]], []).append(v)
    wt, wc = workload_by_name(target), workload_by_name(captured)
    scale = wt.n_params / wc.n_params
    sha = kernel_source_hash()
    lines = [f"# DRAM traffic per launch on {target} ({wt.n_params:,} params), the `traffic` field",
             "# of bench.py's roofline (read only while kernel_src_sha matches the kernel sources'",
             "# code, comments and whitespace removed).  Made on a GB300 by, after the same bench",
             "# command exited 0 without ncu:"]
    lines += [f"#   {c}" for c in commands]
    rec = {}
    for key, per in sorted(launches.items()):
        vals = [sum(v) for v in per.values()]
        mean = sum(vals) / len(vals)
        alg = KERNEL_BYTES_PER_PARAM[key](wc.P) * wc.n_params
        lines.append(f"# {key}: {len(vals)} launch(es) on {captured}, read + write "
                     f"{mean / 1e9:.4f} GB (algorithmic {alg / 1e9:.4f} GB)"
                     + (f", x {scale:.4f} (parameters) = {mean * scale / 1e9:.4f} GB" if scale != 1 else ""))
        how = "ncu dram__bytes_read.sum + dram__bytes_write.sum" + (
            f" on {captured} ({wc.n_params:,} params), scaled by parameters to {wt.n_params:,}"
            if scale != 1 else f" on the full workload, mean of {len(vals)} launch(es)")
        rec[f"{target}:{key}"] = {"bytes_per_launch": mean * scale, "kernel_src_sha": sha, "how": how}
    out = os.path.join(out_dir or os.path.join(ROOT, "profiles"), f"dram_traffic_{target}.txt")
    with open(out, "w") as f:
        f.write("\n".join(lines) + "\n" + json.dumps(rec, indent=1) + "\n")
    return out


# --------------------------------------------------------------------------- CPU oracle
def oracle_sample_rate(wl, plan_sizes_offsets, grads_dev, master_dev, budget_s=15.0,
                       max_passes=3, step=1):
    """Time the CPU oracle's fused step on consecutive batches of buckets
    (skipping the first, a single oversized head matrix), one batch of as many
    buckets as host threads per call, until ~budget_s of work (at most
    max_passes passes over the workload).
    Returns (params/s, params, seconds, threads, description)."""
    import numpy as np
    import oracle
    orc = oracle.default()
    sizes = wl.sizes
    op = orc.plan(sizes, wl.bucket_bytes, wl.P)
    nb = op["n_buckets"]
    threads = os.cpu_count() or 1
    done_params, done_s, b = 0, 0.0, min(1, nb - 1)
    used = []
    offsets = plan_sizes_offsets
    cfg = oracle.adamw_cfg(wl.adamw, step)
    passes = 0
    while done_s < budget_s and passes < max_passes:
        if b >= nb:                      # wrap around for another pass over the workload
            b, passes = min(1, nb - 1), passes + 1
            if passes >= max_passes:
                break
        batch = list(range(b, min(nb, b + threads)))
        tens = [t for t in range(len(sizes)) if op["t_bucket"][t] in batch]
        tens.sort()
        sub = [sizes[t] for t in tens]
        dec = [wl.decay[t] for t in tens]
        g = torch.cat([grads_dev[:, offsets[t]:offsets[t] + sizes[t]] for t in tens], dim=1)
        g = g.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        mst = torch.cat([master_dev[offsets[t]:offsets[t] + sizes[t]] for t in tens]).cpu().numpy()
        z = np.zeros_like(mst)
        t0 = time.perf_counter()
        orc.zero_step(sub, dec, wl.bucket_bytes, wl.P, g, mst, z, z, cfg, n_threads=threads)
        done_s += time.perf_counter() - t0
        done_params += sum(sub)
        used += batch
        b = batch[-1] + 1
    desc = (f"{len(used)} bucket calls over buckets {min(used)}..{max(used)} of {nb} "
            f"({done_params} params in total, {done_params / wl.n_params:.2f}x the workload), "
            f"oracle fused ZeRO step in batches of {threads} buckets, each with its own clip "
            f"norm, inputs copied from the GPU run")
    return done_params / done_s, done_params, done_s, threads, desc


def oracle_allreduce_rate(wl, offsets, grads_dev, budget_s=15.0, max_passes=40):
    """Time the CPU oracle's mean all-reduce (the literal ring over P host buffers,
    every bucket of the plan) on the whole workload: passes until ~budget_s of work,
    at least one and at most max_passes.
    Returns (params/s, params, seconds, threads, description)."""
    import numpy as np
    import oracle
    orc = oracle.default()
    threads = os.cpu_count() or 1
    g = torch.cat([grads_dev[:, offsets[t]:offsets[t] + wl.sizes[t]]
                   for t in range(len(wl.sizes))], dim=1)
    g = g.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    done_params, done_s, passes = 0, 0.0, 0
    while passes < max_passes and (passes == 0 or done_s < budget_s):
        t0 = time.perf_counter()
        orc.allreduce_mean(wl.sizes, wl.bucket_bytes, wl.P, g, want_mean=False, n_threads=threads)
        done_s += time.perf_counter() - t0
        done_params += wl.n_params
        passes += 1
    desc = (f"{passes} pass(es) over the whole workload ({wl.n_params} params each), oracle "
            f"mean all-reduce over all {orc.plan(wl.sizes, wl.bucket_bytes, wl.P)['n_buckets']} "
            f"buckets with {threads} threads, inputs copied from the GPU run")
    return done_params / done_s, done_params, done_s, threads, desc


# --------------------------------------------------------------------------- GPU bench
def run_gpu(args, rank, local, world):
    import gradient_sync_zero_gb300 as dps

    torch.cuda.set_device(local)
    wl = workload_by_name(args.workload)
    if args.max_norm is not None:
        wl.adamw = dataclasses.replace(wl.adamw, max_norm=args.max_norm)
    mesh = tuple(int(x) for x in args.mesh.split(",")) if args.mesh else None
    plan = dps.Plan(wl.sizes, wl.bucket_bytes, wl.P, wl.decay, mesh=mesh)
    if world > 1:
        dps.check_plans_match(plan)      # every process built the same buckets (else DP_EPLAN)
    P, L, stride = plan.P, plan.L, plan.stride
    off = plan.tensor_offsets()
    ws = plan.new_workspace()
    grads = plan.new_replicas()
    wdev.fill_grads(grads, off, wl, step=1)
    zero = wl.mode == "zero"
    if zero:
        params = plan.new_replicas()
        master = plan.new_state()
        wdev.fill_flat(master, off, wl.sizes, gen.master_values(wl, 0, wl.n_params, "cuda"))
        m, v = plan.new_state(), plan.new_state()
        clip = wl.adamw.max_norm > 0
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def cfg(step):
        a = wl.adamw
        return dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, step)

    n_ev = dps.dp_fused_zero_step_launches(cfg(1)) + 1 if zero else 2

    def new_events():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
        for e in evs:
            e.record(stream)
        return evs

    def step_fn(step, evs=None):
        if zero:
            dps.dp_fused_zero_step(plan, ws, grads, params, master, m, v, cfg(step), events=evs)
        else:
            if evs:
                evs[0].record(stream)
            dps.dp_allreduce_mean(plan, ws, grads)
            if evs:
                evs[1].record(stream)

    step = 0
    for _ in range(args.warmup):
        step += 1
        step_fn(step)
    torch.cuda.synchronize()
    ev_sets = [new_events() for _ in range(args.steps)]
    torch.cuda.synchronize()
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    def timed_region():
        nonlocal step
        with ClockSampler(local) as clocks:
            time.sleep(0.3)
            t_begin.record(stream)
            for k in range(args.steps):
                step += 1
                step_fn(step, ev_sets[k])
            t_end.record(stream)
            torch.cuda.synchronize()
        return clocks

    clocks = timed_region()
    # a run that saw hardware or thermal slowdown is measured once more; which
    # run the line reports, and what the first one saw, are in "clocks"
    first_reasons = None
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad & set(clocks.summary()["reasons"]):
        first_reasons = clocks.summary()["reasons"]
        barrier(world)
        clocks = timed_region()
    barrier(world)
    ms_total = t_begin.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / args.steps
    stage_ms = [[ev[i].elapsed_time(ev[i + 1]) for i in range(n_ev - 1)] for ev in ev_sets]
    stage_avg = [sum(s[i] for s in stage_ms) / len(stage_ms) for i in range(n_ev - 1)]
    norm = None
    if zero and clip:
        norm, coef, _ = dps.dp_read_norm(plan, ws)

    # dominant kernel: the longest stage
    if zero:
        names = ["reduce_scatter", "norm_finalize", "adamw_all_gather"] if clip else ["zero_fused"]
    else:
        names = ["allreduce"]
    dom = max(range(len(stage_avg)), key=lambda i: stage_avg[i])
    dom_name = names[dom]
    n_params = wl.n_params
    dom_bytes = KERNEL_BYTES_PER_PARAM[dom_name](P) * n_params
    peak, peak_src = measured_peaks()
    achieved = dom_bytes / (stage_avg[dom] * 1e-3) / 1e9
    step_bytes_pp = (KERNEL_BYTES_PER_PARAM["reduce_scatter"](P)
                     + KERNEL_BYTES_PER_PARAM["adamw_all_gather"](P)) if (zero and clip) else \
        KERNEL_BYTES_PER_PARAM[names[0]](P)
    step_gbs = step_bytes_pp * n_params / (ms_step * 1e-3) / 1e9

    traffic, traffic_src = stored_traffic(wl.name, dom_name)

    result = {
        "metric": "fused ZeRO-2 step params/s and achieved HBM GB/s vs GB300 peak (P=8, 1 GPU)"
        if zero else "bucketed mean all-reduce params/s",
        "value": n_params * world / (ms_step * 1e-3),
        "unit": "params/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "storage": "bf16 gradient and parameter replicas, fp32 master/m/v",
        "data": "synthetic (seeded counter-based N(0, sigma) gradients, N(0, 0.02) master)",
        "config": {
            "workload": wl.name,
            "P": P,
            "n_params": n_params,
            "padded_len": L,
            "replica_stride": stride,
            "n_tensors": len(wl.sizes),
            "n_buckets": plan.n_buckets,
            "bucket_bytes": wl.bucket_bytes,
            "clip_max_norm": wl.adamw.max_norm if zero else None,
            "parallelism": f"{P} virtual ranks per GPU x {world} GPU(s), independent replicas",
            "mesh": f"{plan.info.R}x{plan.info.S} (replicate x shard)",
            "l2": "inputs larger than L2 (no flush): "
                  f"{step_bytes_pp * n_params / 1e9:.1f} GB moved per step vs 0.13 GB L2",
        },
        "step_gbs": step_gbs,
        "stage_ms": dict(zip(names, stage_avg)),
        "roofline": {
            "kernel": dom_name,
            "bound": "hbm",
            "achieved": achieved,
            "peak": peak,
            "peak_source": f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)" if peak_src == "measured"
            else "fallback 6.8 TB/s",
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": traffic,
            "traffic_source": traffic_src,
            "bytes_per_param": KERNEL_BYTES_PER_PARAM[dom_name](P),
        },
        "gpu_launches": (n_ev - 1) * args.steps,
        "clocks": dict(clocks.summary(), **({"remeasured_after": first_reasons}
                                            if first_reasons else {})),
    }
    if norm is not None:
        result["grad_norm"] = norm
        result["clip_coef"] = coef

    # ---- end to end through the public call, host buffers ----
    if not args.no_e2e:
        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        host_buf = PinnedHost(tuple(grads.shape), grads.dtype)
        host = host_buf.t
        host.copy_(grads)
        torch.cuda.synchronize()
        for _ in range(1):                  # untimed: first transfer from fresh pinned pages
            step += 1
            grads.copy_(host, non_blocking=True)
            step_fn(step)
        torch.cuda.synchronize()
        # the host link's own rate on this buffer, for reading the e2e number
        h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h0.record(stream)
        grads.copy_(host, non_blocking=True)
        h1.record(stream)
        torch.cuda.synchronize()
        h2d_gbs = host.numel() * host.element_size() / (h0.elapsed_time(h1) * 1e-3) / 1e9
        # Pipelined: the host-to-device copy runs on its own stream in bucket groups
        # of about equal size; each group's reduction starts as soon as its bytes
        # have arrived.  Across steps, step t+1's copy starts as soon as step t's
        # reductions have consumed the gradient buffer, so it overlaps step t's
        # update pass; each step's result (the workspace's norm and status fields) is
        # read back asynchronously into its own pinned buffer
        # and checked after the loop (flat plans; a mesh plan runs copy-then-step).
        pipelined = mesh is None
        copy_stream = torch.cuda.Stream()
        nb = plan.n_buckets
        groups, lo_b, acc_len = [], 0, 0
        target = plan.L / 16
        for b in range(nb):
            acc_len += plan.bucket(b)[1]
            if acc_len >= target or b == nb - 1:
                groups.append((lo_b, b + 1))
                lo_b, acc_len = b + 1, 0
        if pipelined and zero:
            mean_buf = plan.new_state()
        consumed = [None]                    # event: the last reduction of the previous step
        # --e2e-readback: every step also reads one updated replica back to pinned
        # host memory (the parameters; the mean gradients for an all-reduce), on its
        # own stream, so it runs on the link's other direction beside the next
        # step's host-to-device copy.  The next writer of that replica waits for it.
        readback = args.e2e_readback and pipelined
        if readback:
            d2h_stream = torch.cuda.Stream()
            out_rep = params if zero else grads
            host_out_buf = PinnedHost((L,), torch.bfloat16)
            host_out = host_out_buf.t
        read_done = [None]                   # event: the last step's read-back finished

        def grouped_copies_ms():
            # the copies alone, in the step's bucket groups (for reading the e2e number)
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            for b0, b1 in groups:
                o = plan.bucket(b0)[0]
                e = plan.bucket(b1 - 1)[0] + plan.bucket(b1 - 1)[1]
                for r in range(P):
                    grads[r, o:e].copy_(host[r, o:e], non_blocking=True)
            c1.record(stream)
            torch.cuda.synchronize()
            return c0.elapsed_time(c1)

        copy_before_ms = grouped_copies_ms()

        def e2e_step(step):
            if not pipelined:
                grads.copy_(host, non_blocking=True)
                step_fn(step)
                return
            evs = []
            if consumed[0] is None:
                copy_stream.wait_stream(stream)
            else:
                copy_stream.wait_event(consumed[0])
            if readback and not zero and read_done[0] is not None:
                copy_stream.wait_event(read_done[0])     # the mean is read before it is overwritten
            with torch.cuda.stream(copy_stream):
                for b0, b1 in groups:
                    o = plan.bucket(b0)[0]
                    e = plan.bucket(b1 - 1)[0] + plan.bucket(b1 - 1)[1]
                    for r in range(P):
                        grads[r, o:e].copy_(host[r, o:e], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(copy_stream)
                    evs.append(ev)
            for (b0, b1), ev in zip(groups, evs):
                stream.wait_event(ev)
                if zero:
                    dps.dp_reduce_scatter_mean(plan, ws, grads, mean_buf, b0, b1, want_sumsq=clip)
                else:
                    dps.dp_allreduce_mean(plan, ws, grads, b0, b1)
            consumed[0] = torch.cuda.Event()
            consumed[0].record(stream)
            if zero:
                if clip:
                    dps.dp_clip_coef(plan, ws, wl.adamw.max_norm)
                if readback and read_done[0] is not None:
                    stream.wait_event(read_done[0])      # last step's parameters are out
                dps.dp_adamw_all_gather(plan, ws, mean_buf, master, m, v, params, cfg(step),
                                        use_clip_coef=clip)
            if readback:
                ready = torch.cuda.Event()
                ready.record(stream)
                d2h_stream.wait_event(ready)
                with torch.cuda.stream(d2h_stream):
                    host_out.copy_(out_rep[0, :L], non_blocking=True)
                read_done[0] = torch.cuda.Event()
                read_done[0].record(d2h_stream)

        e2e_step(step + 1)                  # untimed: the pipelined path once
        step += 1
        torch.cuda.synchronize()
        consumed[0] = None
        # the step's result: the workspace's result fields (norm, coef, status), at the
        # offsets the library reports
        off_n2, off_norm, off_coef, off_status = dps.workspace_result_offsets()
        res_bytes = off_status + 4
        results = [torch.empty(res_bytes, dtype=torch.uint8, pin_memory=True)
                   for _ in range(e2e_steps)]
        done = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps + 1)]
        barrier(world)
        t0 = time.perf_counter()
        done[0].record(stream)
        for k in range(e2e_steps):
            step += 1
            e2e_step(step)
            if zero:
                results[k].copy_(ws[:res_bytes], non_blocking=True)   # this step's result, D2H
            else:
                torch.cuda.synchronize()
            done[k + 1].record(stream)
        torch.cuda.synchronize()
        e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, world)
        step_ms = [done[k].elapsed_time(done[k + 1]) for k in range(e2e_steps)]
        if readback and not torch.equal(host_out, out_rep[0, :L].cpu()):
            raise RuntimeError("e2e: the replica read back differs from the device's")
        if zero:
            norms = [float(r[off_norm:off_norm + 8].view(torch.float64)) for r in results]
            status = [int(r[off_status:off_status + 4].view(torch.int32)) for r in results]
            if any(st != 0 for st in status) or norms[-1] != dps.dp_read_norm(plan, ws)[0]:
                raise RuntimeError(f"e2e: unexpected step results {norms} {status}")
        copy_only_ms = grouped_copies_ms()
        result["e2e"] = {"value": n_params * world / e2e_s, "unit": "params/s",
                         "h2d_bytes_per_step": host.numel() * host.element_size(),
                         "d2h_bytes_per_step": (res_bytes if zero else 0) + (2 * L if readback else 0),
                         "steps": e2e_steps, "h2d_gbs_alone": h2d_gbs,
                         "step_ms": [round(x, 2) for x in step_ms],
                         "grouped_copies_alone_ms": round(copy_only_ms, 2),
                         "grouped_copies_before_ms": round(copy_before_ms, 2),
                         "copy": (f"pipelined: {len(groups)} bucket groups, each group's reduction "
                                  "overlapped with the copy, the next step's copy with this step's "
                                  "update; results read back asynchronously"
                                  + ("; one updated replica read back to pinned host memory every "
                                     "step, beside the next step's copy" if readback else "")
                                  if pipelined else "copy, then the step")}
        result["e2e"]["host_memory"] = ("cudaHostAlloc, exact size" if host_buf.exact
                                        else "torch pinned memory")
        if pipelined and zero:
            del mean_buf
        del host
        host_buf.release()
        if readback:
            del host_out
            host_out_buf.release()

    # ---- CPU oracle baseline (rank 0, N=1 only) ----
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if zero:
            rate, npar, secs, thr, desc = oracle_sample_rate(wl, off, grads, master,
                                                             budget_s=args.cpu_budget)
        else:
            wdev.fill_grads(grads, off, wl, step=1)      # fresh inputs, not the last mean
            rate, npar, secs, thr, desc = oracle_allreduce_rate(wl, off, grads,
                                                                budget_s=args.cpu_budget)
        result["cpu_baseline"] = {"value": rate, "unit": "params/s", "cores": thr, "kind": "oracle",
                                  "sample": desc, "seconds": secs}
    return result


class PinnedHost:
    """A page-locked host tensor of exactly its size.  torch's pinned allocator rounds
    each request up to a power of two (32 GB for the 17.6 GB of gradient replicas), so
    large buffers come from cudaHostAlloc directly, through the CUDA runtime torch
    loaded; torch's own pinned memory is the fallback."""

    def __init__(self, shape, dtype):
        self.ptr, self.rt = None, None
        nbytes = int(math.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        try:
            path = next(ln.split()[-1] for ln in open("/proc/self/maps") if "libcudart.so" in ln)
            self.rt = ctypes.CDLL(path)
        except (OSError, StopIteration):
            self.rt = None
        p = ctypes.c_void_p()
        if self.rt is not None and nbytes and \
                self.rt.cudaHostAlloc(ctypes.byref(p), ctypes.c_size_t(nbytes), 0) == 0:
            self.ptr = p.value
            raw = (ctypes.c_uint8 * nbytes).from_address(self.ptr)
            self.t = torch.frombuffer(raw, dtype=torch.uint8).view(dtype).view(shape)
        else:
            if self.rt is not None:
                self.rt.cudaGetLastError()        # a refused allocation's error, read off
            self.t = torch.empty(shape, dtype=dtype, pin_memory=True)

    @property
    def exact(self):
        return self.ptr is not None

    def release(self):
        self.t = None
        if self.ptr is not None:
            torch.cuda.synchronize()
            self.rt.cudaFreeHost(ctypes.c_void_p(self.ptr))
            self.ptr = None


def layer_groups(names):
    """Runs of consecutive tensors of one layer ("<block>.<i>.<rest>"), others
    alone: [(t0, t1), ...] in tensor order."""
    def key(n):
        parts = n.split(".")
        return ".".join(parts[:2]) if len(parts) > 2 and parts[1].isdigit() else n
    out = []
    for t, n in enumerate(names):
        if out and key(names[out[-1][0]]) == key(n):
            out[-1] = (out[-1][0], t + 1)
        else:
            out.append((t, t + 1))
    return out


def run_streamed(args):
    """DDP's overlap, measured: a synthetic backward (one bf16 GEMM per weight
    tensor, dW = dY^T X with `--tokens` rows, last tensor first) on a compute
    stream marks each tensor ready; the tracker fires every complete bucket's
    reduction on a communication stream: by default as short-lived CTAs on a
    stream of the lowest priority, the backward's stream at the highest, so the
    GEMM waves take the SMs first (`--launch persistent`: a persistent grid capped
    at --comm-ctas).  Compared with the backward alone and with backward-then-sync
    on one stream.
    ZeRO without clipping (--max-norm 0) fires each bucket's whole step
    (DP_TRACK_ZERO_STEP); with clipping the tracker reduce-scatters per bucket and
    the clip and the AdamW + all-gather pass follow the backward.  The GEMMs only
    model the backward's time; the gradients are the workload's synthetic ones,
    already resident."""
    import gradient_sync_zero_gb300 as dps

    torch.cuda.set_device(0)
    wl = workload_by_name(args.workload)
    if args.max_norm is not None:
        wl.adamw = dataclasses.replace(wl.adamw, max_norm=args.max_norm)
    plan = dps.Plan(wl.sizes, wl.bucket_bytes, wl.P, wl.decay)
    off = plan.tensor_offsets()
    ws = plan.new_workspace()
    grads = plan.new_replicas()
    wdev.fill_grads(grads, off, wl, step=1)
    zero = wl.mode == "zero"
    a = wl.adamw
    whole = zero and not (a.max_norm > 0)    # each bucket's whole step fires on readiness
    cfg = dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, 1)
    if zero:
        mean, params = plan.new_state(), plan.new_replicas()
        master, m, v = plan.new_state(), plan.new_state(), plan.new_state()
    T = args.tokens
    mats = []
    for shape in wl.shapes:
        if len(shape) >= 2:
            rows, cols = shape[0], int(math.prod(shape[1:]))
            mats.append((torch.randn(T, rows, dtype=torch.bfloat16, device="cuda") * 0.01,
                         torch.randn(T, cols, dtype=torch.bfloat16, device="cuda") * 0.01,
                         torch.empty(rows, cols, dtype=torch.bfloat16, device="cuda")))
        else:
            mats.append(None)
    compute = torch.cuda.Stream(priority=args.compute_priority)
    comm = torch.cuda.Stream(priority=args.comm_priority)
    mode = (dps.DP_TRACK_ZERO_STEP if whole else
            dps.DP_TRACK_REDUCE_SCATTER if zero else dps.DP_TRACK_ALLREDUCE)
    tr = dps.Tracker(plan, mode, ws, grads, mean if zero else None, stream=comm,
                     max_ctas=args.comm_ctas, short_ctas=args.launch == "short")
    side = None
    producer = compute
    if args.side_sms:
        # the GPU split in two SM partitions: the streamed step's backward on the
        # larger, every bucket but the last on the smaller; the last bucket on comm
        side = dps.SmStreams(args.side_sms, priority=args.comm_priority, with_rest=True)
        tr.set_side_stream(side.part, args.side_ctas or 3 * side.n_part)
        producer = side.rest

    events = [torch.cuda.Event() for _ in wl.sizes]
    # marking: "tensor" = an event and a mark call per tensor; "batch" = an event
    # per tensor, one mark call per layer (the tensors "<block>.<i>.*" of one
    # layer; others alone); "layer" = one event and one call per layer
    groups = [(t, t + 1) for t in range(len(wl.sizes))] if args.mark == "tensor" else \
        layer_groups(wl.names)
    host_mark_s = [0.0]
    dry_tr = dps.Tracker(plan, mode, dry_run=True)

    def backward(stream, mark, tracker=None):
        tracker = tracker or tr
        with torch.cuda.stream(stream):
            for g0, g1 in reversed(groups):
                for t in reversed(range(g0, g1)):
                    if mats[t] is not None:
                        dy, x, dw = mats[t]
                        torch.matmul(dy.t(), x, out=dw)
                    if mark and args.mark == "batch":
                        h0 = time.perf_counter()
                        events[t].record(stream)
                        host_mark_s[0] += time.perf_counter() - h0
                if mark:
                    h0 = time.perf_counter()
                    if args.mark == "batch":
                        ts = list(range(g1 - 1, g0 - 1, -1))
                        tracker.mark_ready_batch(ts, [events[t] for t in ts])
                    else:
                        events[g0].record(stream)
                        if g1 - g0 == 1:
                            tracker.mark_ready(g0, events[g0])
                        else:
                            tracker.mark_ready_range(g0, g1, events[g0])
                    host_mark_s[0] += time.perf_counter() - h0

    def finish(stream):
        if zero and not whole:
            dps.dp_clip_coef(plan, ws, a.max_norm, stream=stream)
            dps.dp_adamw_all_gather(plan, ws, mean, master, m, v, params, cfg, stream=stream)

    def sync_all(stream):
        if whole:
            dps.dp_fused_zero_step(plan, ws, grads, params, master, m, v, cfg, stream=stream)
            return
        if zero:
            dps.dp_reduce_scatter_mean(plan, ws, grads, mean, want_sumsq=True, stream=stream)
        else:
            dps.dp_allreduce_mean(plan, ws, grads, stream=stream)
        finish(stream)

    def timed(fn, reps):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps * 1e3

    def only_backward():
        backward(compute, False)

    def sequential():
        backward(compute, False)
        sync_all(compute)

    def streamed():
        if whole:
            tr.set_zero_step(params, master, m, v, cfg)
        tr.begin()
        producer.wait_stream(torch.cuda.current_stream())
        backward(producer, True)
        tr.wait(60000)
        finish(comm)
        # the next step follows this one on the GPU, not after a host sync (the
        # other variants do not sync either; the next step's events are recorded
        # after this step's waits were enqueued)
        torch.cuda.current_stream().wait_stream(comm)
        torch.cuda.current_stream().wait_stream(producer)

    def backward_on_producer():
        producer.wait_stream(torch.cuda.current_stream())
        backward(producer, False)

    def only_sync():
        sync_all(compute)

    def concurrent():
        # the sync of every bucket on the comm stream beside the backward, with no
        # readiness waits (the result is not a valid step): what SM and HBM
        # contention alone cost
        comm.wait_stream(compute)
        backward(compute, False)
        if whole:
            dps.dp_fused_zero_step(plan, ws, grads, params, master, m, v, cfg, stream=comm)
        elif zero:
            dps.dp_reduce_scatter_mean(plan, ws, grads, mean, want_sumsq=True, stream=comm)
            finish(comm)
        else:
            dps.dp_allreduce_mean(plan, ws, grads, stream=comm)
        compute.wait_stream(comm)

    def marks_only():
        # the backward with its event records and marks on a dry-run tracker
        # (no waits, no launches): what marking costs the backward
        dry_tr.begin()
        backward(compute, True, dry_tr)

    def host_ms(fn, reps):
        torch.cuda.synchronize()
        host_mark_s[0] = 0.0
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        t1 = time.perf_counter()
        torch.cuda.synchronize()
        return (t1 - t0) / reps * 1e3, host_mark_s[0] / reps * 1e3

    reps = max(3, args.steps // 5)
    t_bp = timed(backward_on_producer, reps) if side is not None else None
    t_b = timed(only_backward, reps)
    t_s = timed(only_sync, reps)
    t_seq = timed(sequential, reps)
    t_str = timed(streamed, reps)
    t_con = timed(concurrent, reps)
    t_mrk = timed(marks_only, reps)
    hb, _ = host_ms(only_backward, reps)
    hm, hmark = host_ms(marks_only, reps)
    n_launch, n_wait = tr.stats()                 # the last streamed step
    hidden = (t_seq - t_str) / max(t_seq - t_b, 1e-9)
    return {
        "metric": "streamed per-bucket sync: share of sync time hidden under a synthetic backward",
        "value": hidden, "unit": "fraction", "higher_is_better": True,
        "ms": {"backward": t_b, "sync": t_s, "backward_then_sync": t_seq, "streamed": t_str,
               "backward_beside_sync_no_waits": t_con, "backward_with_marks_dry": t_mrk,
               **({"backward_on_the_larger_partition": t_bp} if t_bp is not None else {})},
        "host_ms": {"backward_issue": hb, "backward_issue_with_marks": hm,
                    "in_record_and_mark_calls": hmark},
        "per_step": {"marks": len(groups), "launches": n_launch, "stream_waits": n_wait},
        "config": {"workload": wl.name, "tokens": T,
                   "launch": ("short-lived CTAs, one launch per bucket" if args.launch == "short"
                              else f"persistent grid of at most {args.comm_ctas} CTAs"),
                   "mark": args.mark,
                   "partitions": (f"backward on {side.n_rest} SMs, buckets but the last on "
                                  f"{side.n_part} SMs ({args.side_ctas or 3 * side.n_part} CTAs)"
                                  if side is not None else None),
                   "n_buckets": plan.n_buckets, "mode": wl.mode, "clip_max_norm": a.max_norm,
                   "comm_priority": args.comm_priority,
                   "compute_priority": args.compute_priority,
                   "tracker_mode": ("whole zero step per bucket" if whole else
                                    "reduce-scatter per bucket" if zero else
                                    "all-reduce per bucket")},
    }


def run_zero3_overlap(args):
    """FSDP's overlap, measured (--zero3 --overlap): the ZeRO-3 unit flow beside a
    synthetic forward and backward ("Data Parallelism: DDP, ZeRO and FSDP", "How
    FSDP actually runs").  Forward, first layers first: unit u's GEMMs (Y = X W^T
    per weight tensor, W read from the unit's gathered buffer) wait for u's
    all-gather, which a gather stream issues one unit ahead.  Backward, last layers
    first: the gather stream gathers the unit ahead while the current unit's GEMMs
    (dX = dY W and dW = dY^T X per weight tensor) run; each unit's reduce-scatter
    follows its GEMMs on a reduce-scatter stream.  A buffer is gathered into again
    only after the GEMMs that read it are done.  Then the clip coefficient and the
    shard update.  The gradients reduce-scattered are the workload's synthetic
    replicas (the GEMM outputs only model the compute's time).  Compared with the
    GEMMs alone, the flow alone, and both on one stream in the same order.  The
    collectives run as short-lived CTAs on low-priority streams beside the compute
    stream at the highest priority (--launch persistent: persistent grids on
    high-priority streams)."""
    import gradient_sync_zero_gb300 as dps

    torch.cuda.set_device(0)
    wl = workload_by_name(args.workload)
    plan = dps.Plan(wl.sizes, wl.bucket_bytes, wl.P, wl.decay)
    off = plan.tensor_offsets()
    ws = plan.new_workspace()
    grads = plan.new_replicas()
    wdev.fill_grads(grads, off, wl, step=1)
    master = plan.new_state()
    wdev.fill_flat(master, off, wl.sizes, gen.master_values(wl, 0, wl.n_params, "cuda"))
    shards = master.to(torch.bfloat16)
    m, v, mean = plan.new_state(), plan.new_state(), plan.new_state()
    nb, P, T = plan.n_buckets, plan.P, args.tokens
    buckets = [plan.bucket(b) for b in range(nb)]
    depth = max(1, args.prefetch_depth)
    bufs = [torch.zeros(P, max(ln for _, ln, _ in buckets), dtype=torch.bfloat16, device="cuda")
            for _ in range(depth + 1)]
    short = args.launch == "short"
    compute = torch.cuda.Stream(priority=args.compute_priority if short else 0)
    s_gather = torch.cuda.Stream(priority=args.comm_priority if short else -1)
    s_rs = torch.cuda.Stream(priority=args.comm_priority if short else -1)
    a = wl.adamw
    # weight tensors of each unit (views into a unit buffer's row 0) and GEMM operands
    # shared by shape
    unit_w = [[] for _ in range(nb)]
    ops = {}
    for t, shape in enumerate(wl.shapes):
        if len(shape) < 2:
            continue
        rows, cols = shape[0], int(math.prod(shape[1:]))
        b = plan.tensor(t)[0]
        unit_w[b].append((off[t] - buckets[b][0], rows, cols))
        if (rows, cols) not in ops:
            ops[(rows, cols)] = dict(
                x=torch.randn(T, cols, dtype=torch.bfloat16, device="cuda") * 0.01,
                dy=torch.randn(T, rows, dtype=torch.bfloat16, device="cuda") * 0.01,
                y=torch.empty(T, rows, dtype=torch.bfloat16, device="cuda"),
                dx=torch.empty(T, cols, dtype=torch.bfloat16, device="cuda"),
                dw=torch.empty(rows, cols, dtype=torch.bfloat16, device="cuda"))

    def gemms(b, buf, backward):
        for o, rows, cols in unit_w[b]:
            w = buf[0, o:o + rows * cols].view(rows, cols)
            op = ops[(rows, cols)]
            if backward:
                torch.matmul(op["dy"], w, out=op["dx"])
                torch.matmul(op["dy"].t(), op["x"], out=op["dw"])
            else:
                torch.matmul(op["x"], w.t(), out=op["y"])

    def update(stream):
        dps.dp_clip_coef(plan, ws, a.max_norm, stream=stream)
        dps.dp_shard_adamw_step(plan, ws, mean, master, m, v, shards, cfg, use_clip_coef=True,
                                stream=stream)

    cfg = dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, 1)
    fwd, bwd = list(reversed(range(nb))), list(range(nb))

    def rs(b, stream):
        o, ln, _ = buckets[b]
        dps.dp_unit_reduce_scatter(plan, ws, grads[:, o:o + ln], b, mean, want_sumsq=True,
                                   stream=stream)

    def one_stream(with_gemms, with_flow):
        with torch.cuda.stream(compute):
            for i, b in enumerate(fwd):
                if with_flow:
                    dps.dp_unit_all_gather(plan, ws, shards, b, bufs[i % 2])
                if with_gemms:
                    gemms(b, bufs[i % 2], False)
            for i, b in enumerate(bwd):
                if with_flow:
                    dps.dp_unit_all_gather(plan, ws, shards, b, bufs[i % 2])
                if with_gemms:
                    gemms(b, bufs[i % 2], True)
                if with_flow:
                    rs(b, compute)
            if with_flow:
                update(compute)

    def overlapped():
        cur = torch.cuda.current_stream()
        for s_ in (compute, s_gather, s_rs):
            s_.wait_stream(cur)
        nbuf = len(bufs)
        released = [None] * nbuf

        def gather(i, order):
            with torch.cuda.stream(s_gather):
                if released[i % nbuf] is not None:
                    s_gather.wait_event(released[i % nbuf])
                dps.dp_unit_all_gather(plan, ws, shards, order[i], bufs[i % nbuf], stream=s_gather)
                ev = torch.cuda.Event()
                ev.record(s_gather)
            return ev

        for order, backward in ((fwd, False), (bwd, True)):
            ready = {}
            for i in range(min(depth, len(order))):          # `depth` units ahead
                ready[i] = gather(i, order)
            for i, b in enumerate(order):
                if i + depth < len(order):
                    ready[i + depth] = gather(i + depth, order)
                compute.wait_event(ready.pop(i))
                with torch.cuda.stream(compute):
                    gemms(b, bufs[i % nbuf], backward)
                    done = torch.cuda.Event()
                    done.record(compute)
                released[i % nbuf] = done
                if backward:
                    s_rs.wait_event(done)
                    rs(b, s_rs)
        compute.wait_stream(s_rs)
        compute.wait_stream(s_gather)
        update(compute)
        cur.wait_stream(compute)

    def timed(fn, reps):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps * 1e3

    def flow_on(stream):
        cur = torch.cuda.current_stream()
        stream.wait_stream(cur)
        with torch.cuda.stream(stream):
            for i, b in enumerate(fwd):
                dps.dp_unit_all_gather(plan, ws, shards, b, bufs[i % 2])
            for i, b in enumerate(bwd):
                dps.dp_unit_all_gather(plan, ws, shards, b, bufs[i % 2])
                rs(b, stream)
            update(stream)
        cur.wait_stream(stream)

    if short:
        for s_ in (s_gather, s_rs):
            dps.set_stream_launch(s_, True)
    try:
        reps = max(3, args.steps // 5)
        t_c = timed(lambda: one_stream(True, False), reps)
        t_f = timed(lambda: one_stream(False, True), reps)
        t_seq = timed(lambda: one_stream(True, True), reps)
        t_ov = timed(overlapped, reps)
        t_part = None
        if args.side_sms:
            # the flow alone on a partition of the SMs the GEMMs leave idle: what the
            # collectives can do beside the GEMMs without taking SMs from them
            part = dps.SmStreams(args.side_sms)
            try:
                t_part = timed(lambda: flow_on(part.part), reps)
            finally:
                part.close()
    finally:
        for s_ in (s_gather, s_rs):
            dps.set_stream_launch(s_, False)
    n_gemm = sum(len(u) for u in unit_w)
    return {
        "metric": "ZeRO-3 unit flow beside a synthetic forward + backward: share of the flow's "
                  "time hidden",
        "value": (t_seq - t_ov) / max(t_seq - t_c, 1e-9), "unit": "fraction",
        "higher_is_better": True,
        "ms": {"gemms": t_c, "flow": t_f, "gemms_then_flow_one_stream": t_seq,
               "overlapped": t_ov,
               **({f"flow_alone_on_{part.n_part}_sms": t_part} if t_part is not None else {})},
        "config": {"workload": wl.name, "P": P, "n_units": nb, "tokens": T,
                   "prefetch_depth": depth, "gemms_per_step": 3 * n_gemm,
                   "gemm_tflops_per_step": 6 * T * sum(r * c for u in unit_w for _, r, c in u) / 1e12,
                   "launch": ("short-lived CTAs on low-priority gather and reduce-scatter streams, "
                              "compute at the highest priority" if short else
                              "persistent grids on high-priority gather and reduce-scatter streams"),
                   "data": "synthetic gradients resident; GEMM operands random, W from the "
                           "gathered unit buffer"},
    }


def run_zero3(args):
    """ZeRO-3 unit flow on the bench workload: per step, every unit's forward
    all-gather (last bucket first), its backward all-gather and gradient
    reduce-scatter (first bucket first), the clip coefficient and the shard
    update.  Persistent state 18 B/param over all ranks; one [P][max unit]
    transient buffer (two with --prefetch).  --prefetch: the next unit is
    gathered on a second stream while the current one reduce-scatters (FSDP's
    prefetch; the reduce-scatter waits for its unit's gather, which stands in for
    the backward compute that needs those parameters, and a buffer is reused only
    after the unit that last held it is done).  --graph: the whole step is
    captured once with cfg=None and replayed, the step's AdamW scalars written
    into the workspace before each replay."""
    import gradient_sync_zero_gb300 as dps

    torch.cuda.set_device(0)
    wl = workload_by_name(args.workload)
    mesh = tuple(int(x) for x in args.mesh.split(",")) if args.mesh else None
    plan = dps.Plan(wl.sizes, wl.bucket_bytes, wl.P, wl.decay, mesh=mesh)
    off = plan.tensor_offsets()
    ws = plan.new_workspace()
    grads = plan.new_replicas()
    wdev.fill_grads(grads, off, wl, step=1)
    master = plan.new_state()
    wdev.fill_flat(master, off, wl.sizes, gen.master_values(wl, 0, wl.n_params, "cuda"))
    shards = master.to(torch.bfloat16)
    m, v, mean = plan.new_state(), plan.new_state(), plan.new_state()
    nb, P = plan.n_buckets, plan.P
    buckets = [plan.bucket(b) for b in range(nb)]
    unit_buf = torch.empty(P, max(ln for _, ln, _ in buckets), dtype=torch.bfloat16, device="cuda")
    unit_bufs = [unit_buf, torch.empty_like(unit_buf)] if (args.prefetch or args.fused_backward) \
        else [unit_buf]
    s_a, s_b = torch.cuda.Stream(), torch.cuda.Stream()
    a = wl.adamw
    stream = torch.cuda.current_stream()

    def cfg_of(t):
        return dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, t)

    def forward():
        if not args.prefetch:
            for b in reversed(range(nb)):
                dps.dp_unit_all_gather(plan, ws, shards, b, unit_buf)
            return
        cur = torch.cuda.current_stream()
        s_a.wait_stream(cur)
        s_b.wait_stream(cur)
        for i, b in enumerate(reversed(range(nb))):
            with torch.cuda.stream(s_a if i % 2 == 0 else s_b):
                dps.dp_unit_all_gather(plan, ws, shards, b, unit_bufs[i % 2])
        cur.wait_stream(s_a)
        cur.wait_stream(s_b)

    def backward():
        if args.fused_backward:
            # one launch per unit: the next unit's gather beside this unit's reduce-scatter
            dps.dp_unit_all_gather(plan, ws, shards, 0, unit_bufs[0])
            for b in range(nb):
                o, ln, _ = buckets[b]
                dps.dp_unit_backward(plan, ws, shards, b + 1 if b + 1 < nb else -1,
                                     unit_bufs[(b + 1) % 2], grads[:, o:o + ln], b, mean,
                                     want_sumsq=True)
            return
        if not args.prefetch:
            for b in range(nb):
                o, ln, _ = buckets[b]
                dps.dp_unit_all_gather(plan, ws, shards, b, unit_buf)
                dps.dp_unit_reduce_scatter(plan, ws, grads[:, o:o + ln], b, mean, want_sumsq=True)
            return
        cur = torch.cuda.current_stream()
        s_a.wait_stream(cur)
        s_b.wait_stream(cur)
        released = [None, None]
        for i, b in enumerate(range(nb)):
            o, ln, _ = buckets[b]
            with torch.cuda.stream(s_a):
                if released[i % 2] is not None:
                    s_a.wait_event(released[i % 2])
                dps.dp_unit_all_gather(plan, ws, shards, b, unit_bufs[i % 2])
                gathered = torch.cuda.Event()
                gathered.record(s_a)
            with torch.cuda.stream(s_b):
                s_b.wait_event(gathered)
                dps.dp_unit_reduce_scatter(plan, ws, grads[:, o:o + ln], b, mean, want_sumsq=True)
                done = torch.cuda.Event()
                done.record(s_b)
                released[i % 2] = done
        cur.wait_stream(s_a)
        cur.wait_stream(s_b)

    def update(cfg):
        dps.dp_clip_coef(plan, ws, a.max_norm)
        dps.dp_shard_adamw_step(plan, ws, mean, master, m, v, shards, cfg, use_clip_coef=True)

    graph = None
    if args.graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            dps.dp_set_adamw_cfg(plan, ws, cfg_of(1))
            forward()                       # one eager step first: launcher setup off capture
            backward()
            update(None)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            forward()
            backward()
            update(None)

    def step(t, evs=None):
        def mark(i):
            if evs:
                evs[i].record(stream)
        mark(0)
        if graph is not None:
            dps.dp_set_adamw_cfg(plan, ws, cfg_of(t))
            mark(1)
            mark(2)
            graph.replay()
            mark(3)
            return
        forward()
        mark(1)
        backward()
        mark(2)
        update(cfg_of(t))
        mark(3)

    for t in range(1, args.warmup + 1):
        step(t)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for k in range(args.steps):
        step(args.warmup + 1 + k, evs[k])
    torch.cuda.synchronize()
    parts = [sum(e[i].elapsed_time(e[i + 1]) for e in evs) / args.steps for i in range(3)]
    ms = sum(parts)
    n = wl.n_params
    bytes_pp = 2 * (2 + 2 * P) + (2 * P + 4) + 30          # 2 all-gathers, reduce-scatter, update
    return {
        "metric": "ZeRO-3 unit flow (2 all-gathers + reduce-scatter + shard update) params/s",
        "value": n / (ms * 1e-3), "unit": "params/s", "higher_is_better": True,
        "ms_per_step": ms,
        "stage_ms": {"forward_all_gather": parts[0], "backward_all_gather_reduce_scatter": parts[1],
                     "clip_and_update": parts[2]},
        "gbs": bytes_pp * n / (ms * 1e-3) / 1e9, "bytes_per_param": bytes_pp,
        "resident_bytes_per_param_all_ranks": 2 + 4 + 12,
        "transient_bytes": sum(x.numel() * 2 for x in unit_bufs),
        "config": {"workload": wl.name, "P": P, "n_units": nb,
                   "mesh": f"{plan.info.R}x{plan.info.S} (replicate x shard)",
                   "launch": ("CUDA graph of the whole step" if graph is not None else "host launches")
                   + (", prefetch on two streams" if args.prefetch and not args.fused_backward else "")
                   + (", backward as one launch per unit (next unit's gather beside this unit's "
                      "reduce-scatter)" if args.fused_backward else "")},
    }


def run_accum(args):
    """Gradient accumulation over k micro-batches, then the mean all-reduce: the
    local accumulations (k-1 passes of acc = bf16(acc + g)) and the last
    micro-batch fused with the sync, timed against the unfused last step
    (accumulate, then all-reduce).  Also the all-reduce with bf16 partial sums on
    the ring against the fp32 ring: time and error against an fp64 mean."""
    import gradient_sync_zero_gb300 as dps

    torch.cuda.set_device(0)
    wl = workload_by_name(args.workload)
    plan = dps.Plan(wl.sizes, wl.bucket_bytes, wl.P, wl.decay)
    off = plan.tensor_offsets()
    ws = plan.new_workspace()
    k = max(2, args.accum)
    micro = [plan.new_replicas() for _ in range(2)]
    wdev.fill_grads(micro[0], off, wl, step=1)
    wdev.fill_grads(micro[1], off, wl, step=2)
    acc = plan.new_replicas()
    stream = torch.cuda.current_stream()
    P, n = plan.P, wl.n_params

    def timed(fn, reps):
        for _ in range(args.warmup):
            fn()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * reps)]
        torch.cuda.synchronize()
        for i in range(reps):
            ev[2 * i].record(stream)
            fn()
            ev[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        return sum(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(reps)) / reps

    def accumulate_only():
        dps.dp_accumulate(plan, ws, acc, micro[1])

    def fused_last():
        dps.dp_allreduce_mean_accum(plan, ws, acc, micro[1])

    def unfused_last():
        dps.dp_accumulate(plan, ws, acc, micro[1])
        dps.dp_allreduce_mean(plan, ws, acc)

    def ar_fp32():
        dps.dp_allreduce_mean(plan, ws, acc)

    def ar_bf16():
        dps.dp_allreduce_mean_bf16wire(plan, ws, acc)

    acc.copy_(micro[0])
    t_acc = timed(accumulate_only, args.steps)
    t_fused = timed(fused_last, args.steps)
    t_unfused = timed(unfused_last, args.steps)
    t_ar = timed(ar_fp32, args.steps)
    t_wire = timed(ar_bf16, args.steps)
    step_fused = (k - 1) * t_acc + t_fused          # micro 1 is written in place, k-1 adds
    step_unfused = k * t_acc + t_ar
    # precision of the two rings against the fp64 mean, on the first micro-batch
    L = plan.L
    exact = micro[0][:, :L].double().mean(0)
    res = {}
    for name, fn in (("fp32_ring", dps.dp_allreduce_mean), ("bf16_wire", dps.dp_allreduce_mean_bf16wire)):
        buf = micro[0].clone()
        fn(plan, ws, buf)
        err = (buf[0, :L].double() - exact).abs()
        scale = micro[0][:, :L].double().abs().mean(0)
        rel = err / scale.clamp_min(1e-30)
        res[name] = {"max_err_over_mean_abs_g": float(rel.max()), "mean_err_over_mean_abs_g": float(rel.mean())}
        del buf
    torch.cuda.synchronize()
    b_acc, b_fused, b_ar = 6 * P, 6 * P, 4 * P
    return {
        "metric": f"gradient accumulation ({k} micro-batches) + mean all-reduce, params/s",
        "value": n / (step_fused * 1e-3), "unit": "params/s", "higher_is_better": True,
        "ms_per_step": step_fused, "ms_per_step_unfused": step_unfused,
        "kernel_ms": {"accumulate": t_acc, "fused_last_micro_batch": t_fused,
                      "accumulate_then_allreduce": t_unfused, "allreduce_fp32_ring": t_ar,
                      "allreduce_bf16_wire": t_wire},
        "kernel_gbs": {"accumulate": b_acc * n / (t_acc * 1e-3) / 1e9,
                       "fused_last_micro_batch": b_fused * n / (t_fused * 1e-3) / 1e9,
                       "allreduce_fp32_ring": b_ar * n / (t_ar * 1e-3) / 1e9,
                       "allreduce_bf16_wire": b_ar * n / (t_wire * 1e-3) / 1e9},
        "bytes_per_param": {"accumulate": b_acc, "fused_last_micro_batch": b_fused, "allreduce": b_ar},
        "precision_vs_fp64_mean": res,
        "config": {"workload": wl.name, "P": P, "micro_batches": k, "l2": "inputs > L2"},
    }


def run_sweep(args):
    """Bucket-size sweep on the 6024-tensor P=16 case (24 matrices of 1024x4096 and
    6000 log-uniform 4K-64K vectors): per bucket cap and mode, the bucket and launch
    counts, the padding fraction, and the step time with one launch over the whole
    tile table, with one launch per bucket (DDP's granularity) issued from the host,
    and with those per-bucket launches replayed from a CUDA graph, as one chain and as
    --sweep-chains independent chains (the buckets touch disjoint memory)."""
    import gradient_sync_zero_gb300 as dps

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    rows = []

    def timed(fn, reps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(reps):
            fn()
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / reps

    caps = [int(c) for c in args.sweep_caps.split(",")] if args.sweep_caps else configs.SWEEP_BUCKETS
    modes = args.sweep_modes.split(",")
    for cap in caps:
        for mode in modes:
            wl = configs.sweep_small_tensors(cap, mode, args.sweep_groups)
            plan = dps.Plan(wl.sizes, wl.bucket_bytes, wl.P, wl.decay)
            off = plan.tensor_offsets()
            ws = plan.new_workspace()
            grads = plan.new_replicas()
            wdev.fill_grads(grads, off, wl, step=1)
            nb, P, n = plan.n_buckets, plan.P, wl.n_params
            a = wl.adamw
            cfg = dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, a.max_norm, 1)
            if mode == "zero":
                params = plan.new_replicas()
                master = plan.new_state()
                wdev.fill_flat(master, off, wl.sizes, gen.master_values(wl, 0, wl.n_params, "cuda"))
                m, v, mean = plan.new_state(), plan.new_state(), plan.new_state()

                def single():
                    dps.dp_fused_zero_step(plan, ws, grads, params, master, m, v, cfg)

                def one_bucket(b):
                    dps.dp_reduce_scatter_mean(plan, ws, grads, mean, b, b + 1, want_sumsq=True)

                def buckets():
                    for b in range(nb):
                        one_bucket(b)

                def tail():
                    dps.dp_clip_coef(plan, ws, a.max_norm)
                    dps.dp_adamw_all_gather(plan, ws, mean, master, m, v, params, cfg)

                launches_single = dps.dp_fused_zero_step_launches(cfg)
                launches_bucket = nb + 2
                bpp = 4 * P + 32
            else:
                def single():
                    dps.dp_allreduce_mean(plan, ws, grads)

                def one_bucket(b):
                    dps.dp_allreduce_mean(plan, ws, grads, b, b + 1)

                def buckets():
                    for b in range(nb):
                        one_bucket(b)

                def tail():
                    pass

                launches_single, launches_bucket, bpp = 1, nb, 4 * P
            reps = max(3, args.steps // 5)
            t_single = timed(single, reps)

            def per_bucket():
                buckets()
                tail()

            t_bucket = timed(per_bucket, reps)
            graph_ms, chains_ms, graph_note = None, None, ""
            try:
                g = torch.cuda.CUDAGraph()
                side = torch.cuda.Stream()
                side.wait_stream(stream)
                with torch.cuda.stream(side):
                    buckets()                      # warm the host-side caches off capture
                torch.cuda.synchronize()
                with torch.cuda.graph(g):
                    buckets()

                def graphed():
                    g.replay()
                    tail()

                graph_ms = timed(graphed, reps)
                del g
                # the same launches as independent chains: the buckets touch disjoint
                # memory, so bucket b goes to chain b mod K, forked from and joined
                # to the capture stream (K graph branches instead of one chain)
                chains = [torch.cuda.Stream() for _ in range(args.sweep_chains)]

                def branched():
                    cur = torch.cuda.current_stream()
                    for s_ in chains:
                        s_.wait_stream(cur)
                    for b in range(nb):
                        with torch.cuda.stream(chains[b % len(chains)]):
                            one_bucket(b)
                    for s_ in chains:
                        cur.wait_stream(s_)

                g2 = torch.cuda.CUDAGraph()
                with torch.cuda.stream(side):
                    branched()
                torch.cuda.synchronize()
                with torch.cuda.graph(g2):
                    branched()

                def graphed2():
                    g2.replay()
                    tail()

                chains_ms = timed(graphed2, reps)
                del g2
            except Exception as e:  # noqa: BLE001  (reported in the line, not hidden)
                graph_note = f"graph capture failed: {e}"
            rows.append({
                "bucket_bytes": cap, "mode": mode, "n_buckets": nb, "n_tiles": plan.info.n_tiles,
                "padding_frac": (plan.L - n) / n,
                "launches": {"single": launches_single, "per_bucket": launches_bucket},
                "ms": {"single": t_single, "per_bucket_host": t_bucket, "per_bucket_graph": graph_ms,
                       f"per_bucket_graph_{args.sweep_chains}_chains": chains_ms},
                "gbs_single": bpp * n / (t_single * 1e-3) / 1e9, "bytes_per_param": bpp,
                **({"note": graph_note} if graph_note else {}),
            })
            del grads, ws
            if mode == "zero":
                del params, master, m, v, mean
            torch.cuda.empty_cache()
    return {"metric": "bucket-size sweep: ms per step, single launch vs per-bucket launches",
            "unit": "ms", "rows": rows,
            "config": {"workload": f"sweep-P16 ({len(wl.sizes)} tensors)", "P": 16,
                       "n_params": wl.n_params, "clip_max_norm": wl.adamw.max_norm,
                       "l2": f"inputs > L2 ({wl.n_params * 32 / 1e9:.1f} GB per replica set)"}}


def run_kernels(args):
    """Every entry point's kernel(s) on the workload, one after another: average
    time per launch (CUDA events on the launching stream, after warm-up) and the
    HBM rate of its algorithmic bytes against the measured copy peak.  The unit
    kernels of the ZeRO-3 flow are timed as one pass over all units."""
    import gradient_sync_zero_gb300 as dps

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    wl = workload_by_name(args.workload)
    plan = dps.Plan(wl.sizes, wl.bucket_bytes, wl.P, wl.decay)
    off = plan.tensor_offsets()
    ws = plan.new_workspace()
    P, n, nb = plan.P, wl.n_params, plan.n_buckets
    grads, params, micro = plan.new_replicas(), plan.new_replicas(), plan.new_replicas()
    wdev.fill_grads(grads, off, wl, step=1)
    wdev.fill_grads(micro, off, wl, step=2)
    master = plan.new_state()
    wdev.fill_flat(master, off, wl.sizes, gen.master_values(wl, 0, wl.n_params, "cuda"))
    m, v, mean = plan.new_state(), plan.new_state(), plan.new_state()
    shards = master.to(torch.bfloat16)
    buckets = [plan.bucket(b) for b in range(nb)]
    unit_buf = torch.empty(P, max(ln for _, ln, _ in buckets), dtype=torch.bfloat16, device="cuda")
    a = wl.adamw
    cfg = dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, 1.0, 1)
    cfg0 = dps.adamw_cfg(a.lr, a.beta1, a.beta2, a.eps, a.weight_decay, 0.0, 1)

    def unit_ag_pass():
        for b in range(nb):
            dps.dp_unit_all_gather(plan, ws, shards, b, unit_buf)

    def unit_rs_pass():
        for b in range(nb):
            dps.dp_unit_reduce_scatter(plan, ws, unit_buf[:, :buckets[b][1]], b, mean, want_sumsq=True)

    unit_bufs = [unit_buf, torch.empty_like(unit_buf)]

    def unit_bwd_pass():
        dps.dp_unit_all_gather(plan, ws, shards, 0, unit_bufs[0])
        for b in range(nb):
            o, ln, _ = buckets[b]
            dps.dp_unit_backward(plan, ws, shards, b + 1 if b + 1 < nb else -1, unit_bufs[(b + 1) % 2],
                                 grads[:, o:o + ln], b, mean, want_sumsq=True)

    table = [  # name, kernel, bytes per parameter, call
        ("dp_reduce_scatter_mean", "k_reduce_scatter (small)", 2 * P + 4,
         lambda: dps.dp_reduce_scatter_mean(plan, ws, grads, mean, want_sumsq=True)),
        ("dp_clip_coef", "k_norm_finalize", 0, lambda: dps.dp_clip_coef(plan, ws, 1.0)),
        ("dp_sharded_adamw_step", "k_adamw_all_gather_small (owner rows)", 30,
         lambda: dps.dp_sharded_adamw_step(plan, ws, mean, master, m, v, params, cfg, use_clip_coef=True)),
        ("dp_all_gather", "k_replicate_small (all-gather)", 2 * P, lambda: dps.dp_all_gather(plan, ws, params)),
        ("dp_broadcast", "k_replicate_small (broadcast)", 2 * P, lambda: dps.dp_broadcast(plan, ws, params, 0)),
        ("dp_adamw_all_gather", "k_adamw_all_gather_small", 28 + 2 * P,
         lambda: dps.dp_adamw_all_gather(plan, ws, mean, master, m, v, params, cfg)),
        ("dp_fused_zero_step (no clip)", "k_zero_fused (small)", 4 * P + 24,
         lambda: dps.dp_fused_zero_step(plan, ws, grads, params, master, m, v, cfg0)),
        ("dp_allreduce_mean", "k_allreduce (small)", 4 * P, lambda: dps.dp_allreduce_mean(plan, ws, grads)),
        ("dp_allreduce_mean_bf16wire", "k_allreduce_bf16wire", 4 * P,
         lambda: dps.dp_allreduce_mean_bf16wire(plan, ws, grads)),
        ("dp_accumulate", "k_accumulate", 6 * P, lambda: dps.dp_accumulate(plan, ws, grads, micro)),
        ("dp_allreduce_mean_accum", "k_allreduce_accum", 6 * P,
         lambda: dps.dp_allreduce_mean_accum(plan, ws, grads, micro)),
        ("dp_reduce_scatter_mean_accum", "k_reduce_scatter (accumulating)", 4 * P + 4,
         lambda: dps.dp_reduce_scatter_mean_accum(plan, ws, grads, micro, mean, want_sumsq=True)),
        ("dp_unit_all_gather (all units)", "k_replicate_small (unit)", 2 + 2 * P, unit_ag_pass),
        ("dp_unit_reduce_scatter (all units)", "k_reduce_scatter (small)", 2 * P + 4, unit_rs_pass),
        ("dp_unit_backward (all units)", "k_unit_backward_small", (2 + 2 * P) + (2 * P + 4), unit_bwd_pass),
        ("dp_shard_adamw_step", "k_adamw_all_gather_small (1 row)", 30,
         lambda: dps.dp_shard_adamw_step(plan, ws, mean, master, m, v, shards, cfg, use_clip_coef=True)),
    ]
    peak, peak_src = measured_peaks()
    rows = []
    for name, kern, bpp, fn in table:
        for _ in range(args.warmup):
            fn()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
        torch.cuda.synchronize()
        for i in range(args.steps):
            evs[2 * i].record(stream)
            fn()
            evs[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        ms = sum(evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(args.steps)) / args.steps
        gbs = bpp * n / (ms * 1e-3) / 1e9
        rows.append({"entry": name, "kernel": kern, "ms": round(ms, 4), "bytes_per_param": bpp,
                     "gbs": round(gbs, 1), "frac": round(gbs / peak, 4) if bpp else None})
    return {"metric": "per-kernel time and HBM rate of algorithmic bytes", "unit": "GB/s",
            "peak": peak, "peak_source": peak_src, "rows": rows,
            "config": {"workload": wl.name, "P": P, "n_params": n, "n_buckets": nb,
                       "l2": "inputs larger than L2"}}


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is a bounded sample."""
    import numpy as np
    import oracle
    if rank != 0:
        return None
    wl = workload_by_name(args.workload)
    orc = oracle.default()
    op = orc.plan(wl.sizes, wl.bucket_bytes, wl.P)
    threads = os.cpu_count() or 1
    nb = op["n_buckets"]
    batch = list(range(min(1, nb - 1), min(nb, min(1, nb - 1) + max(1, min(threads, 4)))))
    tens = sorted(t for t in range(len(wl.sizes)) if op["t_bucket"][t] in batch)
    sub = [wl.sizes[t] for t in tens]
    dec = [wl.decay[t] for t in tens]
    base = wdev.tensor_bases(wl.sizes)
    g = np.stack([torch.cat([gen.grad_values(wl, 1, r, base[t], wl.sizes[t]) for t in tens])
                  .view(torch.int16).numpy().view(np.uint16) for r in range(wl.P)])
    mst = torch.cat([gen.master_values(wl, base[t], wl.sizes[t]) for t in tens]).numpy()
    z = np.zeros_like(mst)
    zero = wl.mode == "zero"

    def one_step(step):
        if zero:
            orc.zero_step(sub, dec, wl.bucket_bytes, wl.P, g, mst, z, z,
                          oracle.adamw_cfg(wl.adamw, step), n_threads=threads)
        else:
            orc.allreduce_mean(sub, wl.bucket_bytes, wl.P, g, want_mean=False, n_threads=threads)

    step = 0
    for _ in range(args.warmup):
        step += 1
        one_step(step)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step += 1
        one_step(step)
    secs = (time.perf_counter() - t0) / args.steps
    value = sum(sub) / secs
    desc = (f"buckets {batch[0]}..{batch[-1]} of {nb} ({sum(sub)} params per step), " +
            ("oracle fused ZeRO step with its own clip norm over the sample" if zero else
             "oracle mean all-reduce (literal ring) over the sample"))
    return {
        "impl": "reference",
        "metric": "fused ZeRO-2 step params/s and achieved HBM GB/s vs GB300 peak (P=8, 1 GPU)"
        if zero else "bucketed mean all-reduce params/s",
        "value": value, "unit": "params/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded counter-based)",
        "config": {"workload": wl.name, "P": wl.P, "n_params": wl.n_params},
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--traffic-record", default="",
                    help="write profiles/dram_traffic_<--workload>.txt from this ncu CSV (no GPU)")
    ap.add_argument("--traffic-captured-on", default="",
                    help="--traffic-record: the workload the CSV was captured on (default: --workload)")
    ap.add_argument("--traffic-command", action="append", default=[],
                    help="--traffic-record: an ncu command line to record in the file (repeatable)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama-1.1B-P8-zero2")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-readback", action="store_true",
                    help="e2e: also read one updated replica back to the host every step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--mesh", default="",
                    help="R,S: hybrid mesh of R replicate groups x S shard ranks (R*S = P)")
    ap.add_argument("--zero3", action="store_true", help="time the ZeRO-3 unit flow")
    ap.add_argument("--comm-priority", type=int, default=0,
                    help="with --streamed: CUDA priority of the communication stream (0 lowest; "
                         "lower numbers are higher priorities)")
    ap.add_argument("--compute-priority", type=int, default=-16,
                    help="with --streamed: CUDA priority of the backward's stream (clamped to "
                         "the device's range; -16 = the highest)")
    ap.add_argument("--launch", choices=["short", "persistent"], default="short",
                    help="with --streamed: each bucket as short-lived CTAs (DP_TRACK_SHORT_CTAS) "
                         "or as a persistent grid capped at --comm-ctas")
    ap.add_argument("--max-norm", type=float, default=None,
                    help="override the workload's clip threshold (0 = no clipping: one fused pass)")
    ap.add_argument("--prefetch", action="store_true",
                    help="with --zero3: gather the next unit while the current one reduce-scatters")
    ap.add_argument("--fused-backward", action="store_true",
                    help="--zero3: the backward as dp_unit_backward launches (gather of the next "
                         "unit and reduce-scatter of this one in one launch)")
    ap.add_argument("--graph", action="store_true",
                    help="with --zero3: replay the unit passes from a CUDA graph")
    ap.add_argument("--prefetch-depth", type=int, default=1,
                    help="--zero3 --overlap: units gathered ahead of the compute (buffers = depth + 1)")
    ap.add_argument("--overlap", action="store_true",
                    help="with --zero3: the unit flow beside a synthetic forward and backward "
                         "(FSDP's overlap; --tokens GEMM rows, --launch)")
    ap.add_argument("--kernels", action="store_true",
                    help="time every entry point's kernel on the workload")
    ap.add_argument("--sweep", action="store_true",
                    help="bucket-size sweep: single launch vs per-bucket launches")
    ap.add_argument("--sweep-caps", default="",
                    help="--sweep: comma-separated bucket caps in bytes (default: the four caps)")
    ap.add_argument("--sweep-modes", default="allreduce,zero",
                    help="--sweep: allreduce, zero or both")
    ap.add_argument("--sweep-chains", type=int, default=8,
                    help="--sweep: independent graph chains the per-bucket launches are spread over")
    ap.add_argument("--sweep-groups", type=int, default=24,
                    help="--sweep: groups of (matrix + 250 vectors) in the workload (24 = full)")
    ap.add_argument("--accum", type=int, default=0,
                    help="time k-micro-batch gradient accumulation and the bf16-wire ring")
    ap.add_argument("--streamed", action="store_true",
                    help="measure the overlap of per-bucket sync with a synthetic backward")
    ap.add_argument("--tokens", type=int, default=4096, help="GEMM rows of the synthetic backward")
    ap.add_argument("--mark", choices=["batch", "layer", "tensor"], default="batch",
                    help="--streamed: an event per tensor and a mark call per layer (batch), "
                         "an event and a call per layer (layer), or per tensor (tensor)")
    ap.add_argument("--comm-ctas", type=int, default=152,
                    help="grid cap of the streamed sync kernels")
    ap.add_argument("--side-sms", type=int, default=0,
                    help="--streamed: every bucket but the last on a stream confined to this many SMs")
    ap.add_argument("--side-ctas", type=int, default=0,
                    help="--streamed: grid cap on the SM-partition stream (default 3 per SM)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("note: warm-up raised to the minimum of 3", file=sys.stderr)
        args.warmup = 3
    if args.traffic_record:
        print(traffic_record(args.traffic_record, args.workload,
                             args.traffic_captured_on or args.workload, args.traffic_command))
        return
    if args.impl == "reference":
        # the CPU oracle runs on rank 0 only; other ranks exit without work
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if args.streamed:
        print(json.dumps(run_streamed(args)), flush=True)
        return
    if args.zero3:
        print(json.dumps(run_zero3_overlap(args) if args.overlap else run_zero3(args)), flush=True)
        return
    if args.accum:
        print(json.dumps(run_accum(args)), flush=True)
        return
    if args.sweep:
        print(json.dumps(run_sweep(args)), flush=True)
        return
    if args.kernels:
        print(json.dumps(run_kernels(args)), flush=True)
        return
    rank, local, world = dist_setup()
    res = run_gpu(args, rank, local, world)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

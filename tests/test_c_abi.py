"""The boundary from C: include/dpsync.h compiles as C99 and C11 with warnings as
errors, and a C program linked against libdpsync.so plans tensors (no GPU needed)
with the same layout the Python binding reports."""
import os
import shutil
import subprocess

import pytest

import gradient_sync_zero_gb300 as dps
from gradient_sync_zero_gb300 import build as dbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INC = os.path.join(ROOT, "include")
CC = shutil.which("gcc") or shutil.which("cc")
pytestmark = pytest.mark.skipif(CC is None, reason="no C compiler")


@pytest.mark.parametrize("std", ["c99", "c11"])
def test_header_is_plain_c(std, tmp_path):
    src = tmp_path / "h.c"
    src.write_text('#include "dpsync.h"\nint main(void) { return dp_version() == 2 ? 0 : 1; }\n')
    r = subprocess.run([CC, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                        "-I", INC, str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_plans_like_the_binding(tmp_path):
    lib = dbuild.build()
    exe = tmp_path / "plan_only"
    r = subprocess.run([CC, "-std=c99", "-Wall", "-Werror", "-I", INC,
                        os.path.join(ROOT, "tests", "c", "plan_only.c"), "-o", str(exe),
                        lib, f"-Wl,-rpath,{os.path.dirname(lib)}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stderr
    lines = run.stdout.split("\n")
    plan = dps.Plan([1000, 70000, 12], 64 * 1024, 4, [1, 1, 0])
    assert int(lines[0]) == 71012 and int(lines[1]) == plan.L and int(lines[2]) == plan.n_buckets
    for t in range(3):
        b, off = (int(x) for x in lines[3 + t].split())
        assert (b, off) == plan.tensor(t)
    assert int(lines[6], 16) == plan.fingerprint
    assert lines[7] == "1 1"
    assert lines[8] == "1 1"
    # the header's result offsets are the library's (DevHeader), and the binding's
    assert lines[9] == lines[10], (lines[9], lines[10])
    assert tuple(int(x) for x in lines[10].split()) == dps.workspace_result_offsets()


def _cuda_home():
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


GPU_PROGRAMS = ["allreduce_gpu", "zero_step_gpu", "tracker_gpu"]


def _build_gpu_program(tmp_path, name="allreduce_gpu"):
    lib = dbuild.build()
    cuda = _cuda_home()
    exe = tmp_path / name
    r = subprocess.run([CC, "-std=c99", "-Wall", "-Werror", "-I", INC, "-I", os.path.join(cuda, "include"),
                        os.path.join(ROOT, "tests", "c", f"{name}.c"), "-o", str(exe), lib,
                        f"-Wl,-rpath,{os.path.dirname(lib)}", "-L", os.path.join(cuda, "lib64"),
                        "-lcudart", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"],
                       capture_output=True, text=True)
    return exe, r


@pytest.mark.parametrize("name", GPU_PROGRAMS)
def test_c_gpu_program_builds(tmp_path, name):
    """The GPU callers compile and link as C99 against the library and cudart."""
    if not os.path.exists(os.path.join(_cuda_home(), "include", "cuda_runtime.h")):
        pytest.skip("no CUDA headers")
    _, r = _build_gpu_program(tmp_path, name)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_c_program_allreduces_on_the_gpu(tmp_path):
    """A C99 process with no Python in it: plan, cudaMalloc, upload, all-reduce;
    every replica holds the exact mean."""
    exe, r = _build_gpu_program(tmp_path)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "mismatches 0" in run.stdout


@pytest.mark.gpu
def test_c_program_streams_buckets_through_the_tracker(tmp_path):
    """A C99 process with no Python in it: a high-priority producer stream uploads
    tensors last first and marks them ready; the tracker fires every bucket's
    all-reduce as short-lived CTAs on a lowest-priority stream, in plan order, one
    launch per bucket; every replica holds the exact mean, and a single
    dp_allreduce_mean on a stream set to short-lived CTAs gives the same bits."""
    exe, r = _build_gpu_program(tmp_path, "tracker_gpu")
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "order ok mismatches 0" in run.stdout


# the workload tests/c/zero_step_gpu.c runs (its sizes, decay flags, rank count,
# bucket cap, AdamW settings and step count)
C_ZERO_SIZES = [3, 70000, 4097, 12, 33000]
C_ZERO_DECAY = [1, 1, 0, 0, 1]
C_ZERO_P, C_ZERO_STEPS, C_ZERO_CAP = 4, 2, 64 * 1024


@pytest.mark.gpu
def test_c_program_runs_the_fused_zero_step(tmp_path, orc):
    """A C99 process with no Python in it runs two clipped ZeRO-2 steps through
    the header (plan, upload, dp_fused_zero_step, dp_read_norm) on inputs this
    test writes; its parameters, master, m, v, norms and coefficients equal the
    oracle's bit for bit."""
    import numpy as np
    import oracle as oracle_mod
    from harness import small_workload
    from workloads import configs, gen

    exe, r = _build_gpu_program(tmp_path, "zero_step_gpu")
    assert r.returncode == 0, r.stderr
    wl = small_workload(C_ZERO_SIZES, C_ZERO_P, C_ZERO_CAP, sigma=0.05, seed=77,
                        decay=C_ZERO_DECAY)
    n, P = wl.n_params, C_ZERO_P
    grads = [np.stack([gen.grad_values(wl, s, rk, 0, n).view(dps_int16()).numpy().view(np.uint16)
                       for rk in range(P)]) for s in range(1, C_ZERO_STEPS + 1)]
    master0 = gen.master_values(wl, 0, n).numpy()
    inp, out = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        for g in grads:
            f.write(g.tobytes())
        f.write(master0.astype(np.float32).tobytes())
    run = subprocess.run([str(exe), str(inp), str(out)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    raw = open(out, "rb").read()
    o = 0
    params = np.frombuffer(raw, np.uint16, P * n, o).reshape(P, n)
    o += 2 * P * n
    got = []
    for _ in range(3):
        got.append(np.frombuffer(raw, np.float32, n, o))
        o += 4 * n
    norms = np.frombuffer(raw, np.float64, C_ZERO_STEPS, o)
    o += 8 * C_ZERO_STEPS
    coefs = np.frombuffer(raw, np.float32, C_ZERO_STEPS, o)
    adamw = configs.AdamW(max_norm=1.0)          # the C program's settings
    master, m, v = master0, np.zeros_like(master0), np.zeros_like(master0)
    for s, g in enumerate(grads, start=1):
        p_ref, master, m, v, _, st = orc.zero_step(C_ZERO_SIZES, C_ZERO_DECAY, C_ZERO_CAP, P, g,
                                                   master, m, v, oracle_mod.adamw_cfg(adamw, s))
        assert np.float32(coefs[s - 1]) == np.float32(st.coef) < 1.0
        assert abs(norms[s - 1] - st.norm) <= 1e-10 * st.norm
    assert np.array_equal(params, p_ref)
    for a, b in zip(got, (master, m, v)):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def dps_int16():
    import torch
    return torch.int16

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
    src.write_text('#include "dpsync.h"\nint main(void) { return dp_version() == 1 ? 0 : 1; }\n')
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


def _cuda_home():
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build_gpu_program(tmp_path):
    lib = dbuild.build()
    cuda = _cuda_home()
    exe = tmp_path / "allreduce_gpu"
    r = subprocess.run([CC, "-std=c99", "-Wall", "-Werror", "-I", INC, "-I", os.path.join(cuda, "include"),
                        os.path.join(ROOT, "tests", "c", "allreduce_gpu.c"), "-o", str(exe), lib,
                        f"-Wl,-rpath,{os.path.dirname(lib)}", "-L", os.path.join(cuda, "lib64"),
                        "-lcudart", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"],
                       capture_output=True, text=True)
    return exe, r


def test_c_gpu_program_builds(tmp_path):
    """The GPU caller compiles and links as C99 against the library and cudart."""
    if not os.path.exists(os.path.join(_cuda_home(), "include", "cuda_runtime.h")):
        pytest.skip("no CUDA headers")
    _, r = _build_gpu_program(tmp_path)
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

"""Build libdpsync.so (the CUDA library) in-tree for sm_103a.

Each translation unit compiles in parallel with nvcc; the objects link into one
shared library with the CUDA runtime linked statically, so loading it needs no
GPU and its only runtime dependency is the driver.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdpsync.so")
LIB_CHECKED = os.path.join(HERE, "libdpsync_checked.so")   # -DDPSYNC_CHECKED: index checks
SOURCES = ["plan.cpp", "api.cu", "kernels_reduce.cu", "kernels_update.cu", "noalloc.cu",
           "tracker.cu", "smstream.cu", "checkpoint.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def compile_cmd(src: str, obj: str, verbose_ptxas: bool = False, checked: bool = False):
    cmd = [nvcc(), "-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj]
    if checked:
        cmd.append("-DDPSYNC_CHECKED")
    if src.endswith(".cpp"):
        cmd[1:1] = ["-x", "cu"]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    return cmd


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [os.path.join(CSRC, src)] + [os.path.join(CSRC, h) for h in os.listdir(CSRC)
                                        if h.endswith((".h", ".cuh"))]
    deps.append(os.path.join(INCLUDE, "dpsync.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool = False) -> str:
    """Build libdpsync.so, or with checked=True libdpsync_checked.so (the same
    sources with the device index checks compiled in)."""
    bdir = os.path.join(BUILD, "checked") if checked else BUILD
    lib_path = LIB_CHECKED if checked else LIB
    os.makedirs(bdir, exist_ok=True)
    jobs = []
    for src in SOURCES:
        obj = os.path.join(bdir, os.path.splitext(src)[0] + ".o")
        if force or verbose_ptxas or _stale(obj, src):
            jobs.append(compile_cmd(src, obj, verbose_ptxas, checked))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        logs = list(ex.map(run, jobs))
    objs = [os.path.join(bdir, os.path.splitext(s)[0] + ".o") for s in SOURCES]
    if jobs or not os.path.exists(lib_path):
        link = [nvcc(), "-shared", *ARCH, "-o", lib_path, *objs]
        r = subprocess.run(link, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(link)}\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write("".join(logs))
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                checked="--checked" in sys.argv))

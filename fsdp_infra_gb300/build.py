"""Builds libdbuf.so in-tree (fsdp_infra_gb300/lib/) for sm_103a.

nvcc compiles each CUDA translation unit (-gencode arch=compute_103a,code=sm_103a,
no fast-math: IEEE division, no flush-to-zero), g++ the host planner, and nvcc
links the shared library against the shared CUDA runtime, the same one PyTorch
loads.  Translation units compile in parallel.  No CMake.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libdbuf.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc")
if not os.path.exists(NVCC):
    NVCC = shutil.which("nvcc") or "nvcc"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall", "-Wno-unused-function",
             f"-I{INCLUDE}", f"-I{CSRC}", f"-I{os.path.join(CUDA_HOME, 'include')}"]


def sources():
    cu = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    cpp = sorted(f for f in os.listdir(CSRC) if f.endswith(".cpp"))
    return cu, cpp


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "dbuf.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    objdir = os.path.join(LIBDIR, f"obj{os.getpid()}")
    os.makedirs(objdir, exist_ok=True)
    cu, cpp = sources()
    jobs = []
    for f in cu:
        extra = ["-Xptxas", "-v"] if verbose_ptxas else []
        jobs.append([NVCC, *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, f),
                     "-o", os.path.join(objdir, f + ".o")])
    for f in cpp:
        jobs.append(["g++", *CXX_FLAGS, "-c", os.path.join(CSRC, f),
                     "-o", os.path.join(objdir, f + ".o")])
    logs = []
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        for out in ex.map(_run, jobs):
            logs.append(out)
    objs = [os.path.join(objdir, f + ".o") for f in cu + cpp]
    tmp = LIB + f".tmp{os.getpid()}"
    _run([NVCC, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    shutil.rmtree(objdir, ignore_errors=True)
    if verbose_ptxas:
        sys.stdout.write("\n".join(l for l in logs if l))
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
    print(LIB)

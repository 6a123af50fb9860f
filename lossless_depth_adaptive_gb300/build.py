"""Build the DEX library ``_build/libdex.so`` for sm_103a with nvcc (in-tree).

Each translation unit compiles in parallel; the link uses the shared CUDA runtime so
the process shares one runtime with PyTorch.  Re-running is cheap: objects newer than
their sources and headers are reused.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libdex.so")
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU_SOURCES = ["gemm.cu", "attention.cu", "misc.cu", "dex_api.cu"]
CXX_SOURCES = ["lattice.cpp"]


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs + [os.path.join(ROOT, "include", "dex.h")]


def _stale(obj, src):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(p) > t for p in [src] + _headers())


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every translation unit and link libdex.so; returns the library path."""
    if not os.path.exists(NVCC):
        raise RuntimeError(f"nvcc not found at {NVCC}")
    os.makedirs(OUT, exist_ok=True)
    inc = ["-I", os.path.join(ROOT, "include"), "-I", CSRC]
    jobs = []
    for s in CU_SOURCES:
        src, obj = os.path.join(CSRC, s), os.path.join(OUT, s + ".o")
        if _stale(obj, src) or ptxas_info:
            cmd = [NVCC, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-c", src, "-o", obj, *inc]
            if ptxas_info:
                cmd += ["-Xptxas", "-v"]
            jobs.append(cmd)
    for s in CXX_SOURCES:
        src, obj = os.path.join(CSRC, s), os.path.join(OUT, s + ".o")
        if _stale(obj, src):
            jobs.append(["g++", "-O2", "-std=c++17", "-fPIC", "-c", src, "-o", obj, *inc,
                         "-I", os.path.join(CUDA_HOME, "include")])
    logs = []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
            for out in ex.map(_run, jobs):
                logs.append(out)
    objs = [os.path.join(OUT, s + ".o") for s in CU_SOURCES + CXX_SOURCES]
    if jobs or not os.path.exists(LIB):
        tmp = LIB + ".tmp"
        _run([NVCC, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
              "-Xlinker", "-rpath", "-Xlinker", os.path.join(CUDA_HOME, "lib64")])
        shutil.move(tmp, LIB)
    if verbose:
        print("\n".join(l for l in logs if l.strip()))
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv))

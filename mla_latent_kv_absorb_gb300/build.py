"""Build libmla_gb300.so in place with nvcc (sm_103a only).

Run ``python -m mla_latent_kv_absorb_gb300.build`` or call ``build_library()``.  The
translation units compile in parallel; the library links the CUDA runtime statically so it
loads without a CUDA install on the library path (the driver is found at first use).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libmla_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden"] + ARCH


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libmla_gb300.so")


def _sources():
    return [os.path.join(CSRC, f) for f in ("api.cu", "static_ws.cu", "append.cu", "gather.cu", "plan.cpp")]


def _deps():
    out = list(_sources())
    for f in os.listdir(CSRC):
        if f.endswith((".cuh", ".h")):
            out.append(os.path.join(CSRC, f))
    out.append(os.path.join(INCLUDE, "mla.h"))
    return out


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build_library(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    jobs = []
    for src in _sources():
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        extra = ["-Xptxas", "-v"] if (verbose and src.endswith(".cu")) else []
        jobs.append(([nvcc] + NVCC_FLAGS + extra + ["-I", INCLUDE, "-c", src, "-o", obj], obj))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        logs = list(ex.map(run, [c for c, _ in jobs]))
    if verbose:
        for lg in logs:
            sys.stdout.write(lg)
    tmp = LIB_PATH + ".tmp"
    run([nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + [o for _, o in jobs])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))

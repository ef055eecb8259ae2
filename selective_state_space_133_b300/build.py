"""Builds libmambascan.so in-tree with nvcc for sm_103a (no JIT, no torch extension).

Each .cu file is compiled to an object on its own (in parallel: the forward
kernels of each state size have a file of their own), then the objects are
linked into the shared library.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIBRARY = os.path.join(HERE, "libmambascan.so")
OBJDIR = os.path.join(HERE, "_build")
SOURCES = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
# every source and header the library is built from: any change triggers a rebuild
DEPENDS = SOURCES + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))) + [
    os.path.join(os.path.dirname(HERE), "include", "mamba_scan.h")]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def up_to_date() -> bool:
    if not os.path.exists(LIBRARY):
        return False
    t = os.path.getmtime(LIBRARY)
    return all(os.path.getmtime(f) <= t for f in DEPENDS)


def _compile(src: str, extra_flags) -> str:
    obj = os.path.join(OBJDIR, os.path.splitext(os.path.basename(src))[0] + ".o")
    subprocess.run([nvcc(), *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj], check=True)
    return obj


def build_library(force: bool = False, extra_flags=()) -> str:
    """Compile the CUDA sources into libmambascan.so next to this file."""
    if force or not up_to_date():
        os.makedirs(OBJDIR, exist_ok=True)
        workers = max(1, min(len(SOURCES), os.cpu_count() or 1))
        with concurrent.futures.ThreadPoolExecutor(workers) as pool:
            objs = list(pool.map(lambda src: _compile(src, extra_flags), SOURCES))
        tmp = LIBRARY + ".tmp"
        subprocess.run([nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", *objs, "-o", tmp],
                       check=True)
        os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build_library(force=True))

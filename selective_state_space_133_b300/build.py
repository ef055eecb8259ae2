"""Builds libmambascan.so in-tree with nvcc for sm_103a (no JIT, no torch extension).

Each .cu file is compiled to an object on its own (in parallel: the forward
kernels of each state size have a file of their own), then the objects are
linked into the shared library. ``build_library(checked=True)`` builds the
same sources with -DMAMBA_DEBUG_BOUNDS into libmambascan_checked.so, the
testing build whose kernels check every plain global access against its
tensor's extent (include/mamba_scan.h, mamba_checked_bounds).
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
CHECKED_LIBRARY = os.path.join(HERE, "libmambascan_checked.so")
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


def up_to_date(library: str = LIBRARY) -> bool:
    if not os.path.exists(library):
        return False
    t = os.path.getmtime(library)
    return all(os.path.getmtime(f) <= t for f in DEPENDS)


def _compile(src: str, objdir: str, extra_flags) -> str:
    obj = os.path.join(objdir, os.path.splitext(os.path.basename(src))[0] + ".o")
    subprocess.run([nvcc(), *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj], check=True)
    return obj


def build_library(force: bool = False, extra_flags=(), checked: bool = False) -> str:
    """Compile the CUDA sources into libmambascan.so (or, checked, libmambascan_checked.so) next to this file."""
    library = CHECKED_LIBRARY if checked else LIBRARY
    objdir = os.path.join(OBJDIR, "checked") if checked else OBJDIR
    flags = (*extra_flags, "-DMAMBA_DEBUG_BOUNDS") if checked else tuple(extra_flags)
    if force or not up_to_date(library):
        os.makedirs(objdir, exist_ok=True)
        workers = max(1, min(len(SOURCES), os.cpu_count() or 1))
        with concurrent.futures.ThreadPoolExecutor(workers) as pool:
            objs = list(pool.map(lambda src: _compile(src, objdir, flags), SOURCES))
        tmp = library + ".tmp"
        subprocess.run([nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", *objs, "-o", tmp],
                       check=True)
        os.replace(tmp, library)
    return library


if __name__ == "__main__":
    print(build_library(force=True))
    print(build_library(force=True, checked=True))

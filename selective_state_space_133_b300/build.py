"""Builds libmambascan.so in-tree with nvcc for sm_103a (no JIT, no torch extension)."""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIBRARY = os.path.join(HERE, "libmambascan.so")
SOURCES = [os.path.join(CSRC, "mamba_scan.cu")]
# every source and header the library is built from: any change triggers a rebuild
DEPENDS = SOURCES + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [
    os.path.join(os.path.dirname(HERE), "include", "mamba_scan.h")]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared"]


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


def build_library(force: bool = False, extra_flags=()) -> str:
    """Compile the CUDA sources into libmambascan.so next to this file."""
    if force or not up_to_date():
        tmp = LIBRARY + ".tmp"
        subprocess.run([nvcc(), *NVCC_FLAGS, *extra_flags, *SOURCES, "-o", tmp], check=True)
        os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build_library(force=True))

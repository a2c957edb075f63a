"""Build ``libvattn.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

One translation unit, one ``-gencode`` (compute_103a -> sm_103a), CUDA
runtime linked statically so the library loads on hosts without a GPU
driver (the tests check its exported symbols there).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, "vattn_api.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "attn_kernel.cuh"), os.path.join(CSRC, "stage_kernel.cuh"),
                  os.path.join(CSRC, "rope_kernel.cuh"),
                  os.path.join(CSRC, "conv1d_kernel.cuh"),
                  os.path.join(CSRC, "ptx.cuh"),
                  os.path.join(ROOT, "include", "vattn.h")]
LIB = os.path.join(PKG, "libvattn.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libvattn.so")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc_path(), ARCH, "-O3", "-std=c++17", "-lineinfo", "--cudart=static",
           "-Xcompiler", "-fPIC", "-shared", "-I", os.path.join(ROOT, "include"),
           "-o", tmp] + SOURCES
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

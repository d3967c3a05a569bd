"""Compile libmuon.so in-tree for sm_103a with nvcc.

Usage: ``python -m pretraining_optimizer_step_b300.build`` (or ``build_library()``).
The library statically links the CUDA runtime and resolves the driver's
tensor-map encoder at run time, so it loads on a machine without a GPU driver
(only the compute calls need one).
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
LIB_PATH = os.path.join(PKG_DIR, "libmuon.so")
SOURCES = ["muon_api.cu", "momentum_norm.cu", "ns_pair.cu", "noalloc.cu", "adamw.cu", "normuon.cu"]
HEADERS = ["kernels.cuh", "ptx.cuh"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "muon.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build_library(force: bool = False, verbose: bool = False, extra=None) -> str:
    if not force and not _stale():
        return LIB_PATH
    cmd = [_nvcc(), "-O3", "-std=c++17", *ARCH_FLAGS, "-lineinfo", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-shared", "-I", os.path.join(ROOT, "include"),
           "-o", LIB_PATH + ".tmp"]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    if extra:
        cmd += list(extra)
    cmd += [os.path.join(CSRC, f) for f in SOURCES]
    subprocess.run(cmd, check=True)
    os.replace(LIB_PATH + ".tmp", LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build_library(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB_PATH)

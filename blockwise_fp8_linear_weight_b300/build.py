"""Builds libbfp8.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Usage: ``python -m blockwise_fp8_linear_weight_b300.build [--force]``.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libbfp8.so")
SOURCES = [os.path.join(CSRC, "bfp8.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("ptx.cuh", "quant.cuh", "gemm.cuh", "muonh.cuh")] + [
    os.path.join(ROOT, "include", "bfp8.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    # IEEE division and subnormals are part of the quantiser's definition
    "-prec-div=true", "-ftz=false", "-fmad=true",
    "-Xcompiler", "-fPIC", "-shared",
]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    if force or stale():
        cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), *SOURCES, "-o", LIB + ".tmp"]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        subprocess.run(cmd, check=True)
        os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)

"""Builds libfp8bs.so in-tree with nvcc for sm_103a (B300).

Usage: python -m fp8_fine_grained_17_b300.build [--verbose]
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libfp8bs.so")
SOURCES = ["fp8bs_common.cu", "fp8bs_quant.cu", "fp8bs_norm.cu", "fp8bs_gemm.cu"]
HEADERS = ["fp8bs_device.cuh", "fp8bs_e4m3.cuh", "fp8bs_host.h"]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
# No fast-math: the quantizers must round every binary32 operation as IEEE does.
FLAGS = [
    "-O3", "-std=c++17", "-lineinfo",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
    "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-I", os.path.join(ROOT, "include"),
]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "fp8bs.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    tmp = LIB + ".tmp"
    cmd = [NVCC, *FLAGS, *(["-Xptxas", "-v"] if verbose else []), "-o", tmp,
           *[os.path.join(CSRC, f) for f in SOURCES]]
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose="--verbose" in sys.argv)
    print(LIB)

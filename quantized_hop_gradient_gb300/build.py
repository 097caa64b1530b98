"""Builds libdq (the CUDA library) in-tree for sm_103a with nvcc.

Flags that matter for the method: ``-fmad=false`` (no multiply-add
contraction in device code) and ``-ffp-contract=off`` for the host compiler
(the level tables are computed on the host), so every fp32 step is rounded
exactly once as written.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libdq.so")
SOURCES = ["dq_api.cu", "dq_codec.cu", "dq_hop.cu", "dq_mx.cu", "dq_plan.cu", "dq_static.cu"]
HEADERS = ["dq_common.cuh", "dq_internal.h", "dq_sched.h"]
INCLUDE = os.path.join(os.path.dirname(HERE), "include", "dq.h")


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = os.path.join(home, "bin", "nvcc")
    return p if os.path.exists(p) else "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [INCLUDE, __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
           "-fmad=false", "-Xcompiler", "-fPIC,-ffp-contract=off", "--threads", "0", "-shared",
           *[os.path.join(CSRC, f) for f in SOURCES], "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

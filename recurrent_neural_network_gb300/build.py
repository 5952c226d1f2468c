"""Builds librnn.so (the CUDA kernels and the C-ABI) for sm_103a, in-tree.

    python -m recurrent_neural_network_gb300.build

Each translation unit is compiled by nvcc in parallel, then linked into
recurrent_neural_network_gb300/_lib/librnn.so against the shared CUDA runtime.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT, "librnn.so")
UNITS = ["api.cu", "gemm.cu", "step_fwd.cu", "step_bwd.cu", "persist.cu", "stack.cu", "stack_bwd.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# a variable read before it is set (diagnostic 549) fails the build instead of warning
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--diag-error", "549"]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found")
    return p


def _deps():
    files = [os.path.join(SRC, f) for f in os.listdir(SRC)]
    files.append(os.path.join(os.path.dirname(HERE), "include", "rnn.h"))
    return max(os.path.getmtime(f) for f in files)


def _compile(unit: str, tmpdir: str) -> str:
    obj = os.path.join(tmpdir, unit.replace(".cu", ".o"))
    cmd = [nvcc()] + ARCH + FLAGS + ["-c", os.path.join(SRC, unit), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {unit}:\n{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit for sm_103a and link librnn.so."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps():
        return LIB
    os.makedirs(OUT, exist_ok=True)
    tmpdir = os.path.join(OUT, f"obj{os.getpid()}")
    os.makedirs(tmpdir, exist_ok=True)
    units = [u for u in UNITS if os.path.exists(os.path.join(SRC, u))]
    with cf.ThreadPoolExecutor(max_workers=len(units)) as ex:
        objs = list(ex.map(lambda u: _compile(u, tmpdir), units))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    shutil.rmtree(tmpdir, ignore_errors=True)
    if verbose:
        print("built", LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)

"""Build the in-tree CUDA library libgemm_f16.so for sm_103a with nvcc.

One translation unit, one -gencode target, position-independent, static CUDA
runtime.  Rebuilt only when a source or header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libgemm_f16.so")
SOURCES = [os.path.join(HERE, "csrc", "gemm_f16.cu")]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
    "-I" + os.path.join(ROOT, "include"),
]


def _inputs():
    return (SOURCES + glob.glob(os.path.join(HERE, "csrc", "*.cuh"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")))


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and up_to_date():
        return LIB
    nvcc = NVCC if os.path.exists(NVCC) else "nvcc"
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *FLAGS, *extra_flags, "-o", tmp, *SOURCES]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)

"""Build the CUDA library in-tree: bit_quantization_matmul_row_b300/libllmint8.so.

One nvcc invocation, sm_103a only.  Run as a module (python -m
bit_quantization_matmul_row_b300.build) or call build().
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libllmint8.so")
SOURCES = [os.path.join(CSRC, "api.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")] + [
    os.path.join(INCLUDE, "llmint8.h")]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
    "-cudart", "shared",
    "-Xlinker", "-rpath,/usr/local/cuda/lib64",
    "-I", INCLUDE, "-I", CSRC,
]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in DEPENDS)


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    if force or stale():
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [NVCC, *FLAGS, *extra, *SOURCES, "-o", tmp]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else [])
    print(LIB)

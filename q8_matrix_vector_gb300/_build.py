"""Build step for the q8mv CUDA library (sm_103a only).

Compiles ``csrc/q8mv.cu`` into ``libq8mv.so`` inside the package directory
with nvcc.  Run ``python -m q8_matrix_vector_gb300._build`` or call
``build_library()``; nothing here needs a GPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "q8mv.cu")
HDR = os.path.join(ROOT, "include", "q8mv.h")
LIB = os.path.join(PKG, "libq8mv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
    # IEEE f32: no flush of subnormals, correctly rounded division/sqrt, no
    # contraction beyond the fused multiply-adds the source asks for
    "-ftz=false", "-prec-div=true", "-prec-sqrt=true", "-fmad=true",
    "-Xptxas", "-warn-spills",
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the q8mv library needs the CUDA toolkit to build")


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile libq8mv.so if it is missing or older than its sources."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(SRC), os.path.getmtime(HDR))):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, SRC, "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))

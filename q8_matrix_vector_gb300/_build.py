"""Build step for the q8mv CUDA library (sm_103a only).

Compiles the translation units under ``csrc/`` (``q8mv.cu``: the single-row
kernels and the C ABI; ``batched.cu``: the batched kernel; ``pair.cu``: the
feed-forward pair kernel) in parallel with
nvcc and links them into ``libq8mv.so`` inside the package directory.  Run
``python -m q8_matrix_vector_gb300._build`` or call ``build_library()``;
nothing here needs a GPU.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
UNITS = [os.path.join(CSRC, "q8mv.cu"), os.path.join(CSRC, "batched.cu"), os.path.join(CSRC, "pair.cu")]
SRC = UNITS[0]
HDR = os.path.join(ROOT, "include", "q8mv.h")
LIB = os.path.join(PKG, "libq8mv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
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


def sources() -> list:
    """Every file the library is built from."""
    files = [HDR]
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            files.append(os.path.join(CSRC, name))
    return files


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile libq8mv.so if it is missing or older than any of its sources."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(f) for f in sources())):
        return LIB
    tag = f"{os.getpid()}"
    objs, procs = [], []
    for unit in UNITS:
        obj = os.path.join(CSRC, os.path.basename(unit) + f".{tag}.o")
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", unit, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
            print(" ".join(cmd), file=sys.stderr)
        objs.append(obj)
        procs.append(subprocess.Popen(cmd))
    try:
        failed = [unit for unit, proc in zip(UNITS, procs) if proc.wait() != 0]
        if failed:
            raise RuntimeError(f"nvcc failed on {', '.join(os.path.basename(u) for u in failed)}")
        tmp = LIB + f".tmp{tag}"
        subprocess.run([nvcc(), *ARCH, "-shared", *objs, "-o", tmp], check=True)
        os.replace(tmp, LIB)
    finally:
        for proc in procs:
            if proc.poll() is None:
                proc.kill()
                proc.wait()
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))

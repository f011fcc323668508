"""Build libaveris.so (sm_103a) in-tree with nvcc, and its bounds-checked
debug variant libaveris_debug.so (-DAVERIS_DEBUG: every global address a
kernel computes is checked against its buffer, see csrc/debug.cuh).

Usage: python -m mean_residual_gemm_col_b300.build [--force] [--debug]
"""

from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libaveris.so")
DEBUG_LIB = os.path.join(PKG, "libaveris_debug.so")

SOURCES = [os.path.join(CSRC, "averis_api.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("ptx.cuh", "quant.cuh", "gemm.cuh", "debug.cuh")] + [
    os.path.join(INCLUDE, "averis.h")
]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
    "-cudart", "shared",
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in DEPENDS)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile the library (debug: the bounds-checked variant) if any source is
    newer than it; return its path."""
    lib = DEBUG_LIB if debug else LIB
    if not force and up_to_date(lib):
        return lib
    tmp = lib + ".tmp"
    cmd = [nvcc(), *NVCC_FLAGS, *(["-DAVERIS_DEBUG"] if debug else []), "-I" + INCLUDE, "-o", tmp, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))

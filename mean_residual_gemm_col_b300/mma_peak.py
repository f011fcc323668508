"""Build and run the tensor-core instruction throughput measurement (csrc/mma_peak.cu).

Prints, per MMA form, the SM cycles one instruction takes when issued back to
back and the rate with one CTA per SM on every SM.  The GEMM's roofline is
reported against the measured bf16 peak (MEASURED_PEAKS.json) times the nominal FP4:BF16
ratio; this measures what the NVFP4 instruction itself delivers here.

Usage: python -m mean_residual_gemm_col_b300.mma_peak
"""

from __future__ import annotations

import os
import subprocess
import sys

from .build import CSRC, PKG, nvcc

BIN = os.path.join(PKG, "mma_peak")
SRC = os.path.join(CSRC, "mma_peak.cu")


def build() -> str:
    deps = [SRC, os.path.join(CSRC, "ptx.cuh")]
    if os.path.exists(BIN) and all(os.path.getmtime(f) <= os.path.getmtime(BIN) for f in deps):
        return BIN
    subprocess.run([nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-I" + CSRC,
                    "-o", BIN, SRC], check=True)
    return BIN


if __name__ == "__main__":
    sys.exit(subprocess.run([build()]).returncode)

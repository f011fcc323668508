"""Run the mean-split NVFP4 quantize pass on a list of activation shapes.

A driver for profiling the quantize kernels through the C ABI: for every
shape, a seeded synthetic bf16 activation (the bench's recipe: planted
rank-one mean, unit normal noise, sparse spikes) is quantized once outside
and `--iters` times inside the NVTX range "quantize" (one range per shape,
in the order given), eagerly on the current stream, so that a profiler sees
every launch (stats, quantize; plus the rotated-maximum pass with --mode
averis_h16).

  python -m mean_residual_gemm_col_b300.run_quantize --shapes 8192x1024,65536x8192 [--iters 1] [--mode averis]
"""

from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

SWEEP = ",".join(f"{l}x{m}" for l in (4096, 16384, 65536) for m in (1024, 2048, 4096, 8192))
STEP = "8192x1024,8192x2048,8192x3072,8192x4096,8192x6144"


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--shapes", default=STEP + "," + SWEEP, help="comma-separated LxM (tokens x features)")
    ap.add_argument("--iters", type=int, default=1)
    ap.add_argument("--mode", default="averis", choices=["averis", "nvfp4", "averis_h16", "nvfp4_h16"])
    ap.add_argument("--spike", type=float, default=30.0)
    args = ap.parse_args(argv)

    import torch

    import workloads
    from mean_residual_gemm_col_b300 import capi

    dev = torch.device("cuda", torch.cuda.current_device())
    capi.load()
    flags = (capi.AVERIS_MEAN_SPLIT if args.mode.startswith("averis") else 0) | (
        capi.AVERIS_HADAMARD16 if args.mode.endswith("h16") else 0)
    for i, shape in enumerate(args.shapes.split(",")):
        l, m = (int(v) for v in shape.lower().split("x"))
        x = workloads.torch_activation(i, l, m, spike=args.spike, device=dev)
        out = capi.averis_quantize(x, flags)
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.nvtx.range_push("quantize")
        start.record()
        for _ in range(args.iters):
            out = capi.averis_quantize(x, flags)
        end.record()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        if capi.averis_last_device_error() != 0:
            raise RuntimeError("device-side wait timed out")
        ms = start.elapsed_time(end) / args.iters
        print(f"{l}x{m} {args.mode}: {ms * 1e3:.1f} us per call (eager, includes launch gaps)")
        del x, out
        torch.cuda.empty_cache()
    return 0


if __name__ == "__main__":
    sys.exit(main())

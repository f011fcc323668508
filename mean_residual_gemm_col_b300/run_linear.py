"""Run one Averis (or vanilla NVFP4) linear layer forward + backward on the GPU.

A small driver for profiling a single layer shape through the C ABI: the
inputs are the seeded synthetic activations, weights and output gradients,
each iteration is weight quantize, forward and backward, launched eagerly
on the current stream (no graph, so a profiler sees every kernel launch in
order: per iteration 3 quantize-weight kernels, then per tensor the stats,
quantize and GEMM launches).

  python -m mean_residual_gemm_col_b300.run_linear --l 8192 --m 1024 --n 4096 [--iters 3] [--mode averis]
"""

from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--l", type=int, default=8192)
    ap.add_argument("--m", type=int, default=1024)
    ap.add_argument("--n", type=int, default=4096)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--mode", default="averis", choices=["averis", "nvfp4", "averis_h16", "nvfp4_h16"])
    ap.add_argument("--spike", type=float, default=30.0)
    args = ap.parse_args(argv)

    import torch

    import workloads
    from mean_residual_gemm_col_b300 import capi

    dev = torch.device("cuda", torch.cuda.current_device())
    capi.load()
    x, w, d = workloads.torch_linear_case(0, args.l, args.m, args.n, spike=args.spike, device=dev)
    split = args.mode.startswith("averis")
    hf = capi.AVERIS_HADAMARD16 if args.mode.endswith("h16") else 0
    state = capi.FwdState.empty(args.l, args.m, dev)
    y = torch.empty(args.l, args.n, dtype=torch.bfloat16, device=dev)
    dx = torch.empty(args.l, args.m, dtype=torch.bfloat16, device=dev)
    dw = torch.empty(args.m, args.n, dtype=torch.float32, device=dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record()
    for _ in range(args.iters):
        w_n, w_m = capi.averis_quantize_weight(w, hf)
        if split:
            capi.averis_linear_fwd(x, w_m, capi.AVERIS_MEAN_SPLIT | hf, out_bf16=True, state=state, y=y)
            capi.averis_linear_bwd(d, state, w_n, capi.AVERIS_MEAN_SPLIT | hf, out_bf16=True, dx=dx, dw=dw)
        else:
            capi.nvfp4_linear_fwd(x, w_m, hf, out_bf16=True, state=state, y=y)
            capi.nvfp4_linear_bwd(d, state, w_n, hf, out_bf16=True, dx=dx, dw=dw)
    end.record()
    torch.cuda.synchronize()
    err = capi.averis_last_device_error()
    if err != 0:
        raise SystemExit(f"device-side wait gave up (code {err})")
    print(f"{args.mode} l={args.l} m={args.m} n={args.n}: {start.elapsed_time(end) / args.iters:.4f} ms/iter "
          f"(eager, includes host launch overhead)")


if __name__ == "__main__":
    main()

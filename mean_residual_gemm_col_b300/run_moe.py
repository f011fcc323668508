"""Run the mixture-of-experts expert FFN forward + backward on the GPU.

A small driver for profiling the grouped path through the C ABI: hidden 2048,
64 experts, top-8 of 16384 tokens routed with Zipf(1.1) popularity, expert
FFN 768 (gate_up 2048 -> 1536, down 768 -> 2048), seeded synthetic inputs.
Each iteration is, per linear, the grouped weight quantize of the stacked
expert weights, the grouped forward and the grouped backward, launched
eagerly on the current stream (no graph: a profiler sees every launch).

  python -m mean_residual_gemm_col_b300.run_moe [--iters 2] [--mode averis|nvfp4]
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
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--mode", default="averis", choices=["averis", "nvfp4"])
    args = ap.parse_args(argv)

    import numpy as np
    import torch

    import workloads
    from mean_residual_gemm_col_b300 import capi

    cfg = workloads.MOE
    dev = torch.device("cuda", torch.cuda.current_device())
    capi.load()
    counts = workloads.moe_routing(0, cfg["tokens"], cfg["experts"], cfg["top_k"], cfg["zipf"])
    offsets = np.concatenate([[0], np.cumsum(counts)])
    rows = int(offsets[-1])
    flags = capi.AVERIS_MEAN_SPLIT if args.mode == "averis" else 0
    lin = []
    for i, (m, n) in enumerate(((cfg["hidden"], 2 * cfg["ffn"]), (cfg["ffn"], cfg["hidden"]))):
        x = workloads.torch_activation(31 + i, rows, m, spike=workloads.QWEN3_SPIKE, device=dev)
        _, _, d = workloads.torch_linear_case(41 + i, rows, 16, n, device=dev)
        w = torch.stack([workloads.torch_linear_case(100 * i + e, 16, m, n, device=dev)[1]
                         for e in range(cfg["experts"])])
        wn = [capi.NVFP4Tensor.empty(m, n, dev) for _ in range(cfg["experts"])]
        wm = [capi.NVFP4Tensor.empty(n, m, dev) for _ in range(cfg["experts"])]
        lin.append((x, d, w, wn, wm, capi.GroupedLinear(offsets, m, n, wm, wn, dev)))
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record()
    for _ in range(args.iters):
        for x, d, w, wn, wm, gl in lin:
            capi.averis_quantize_weight_grouped(w, 0, w_n=wn, w_m=wm)
            gl.fwd(x, flags, out_bf16=True)
            gl.bwd(d, flags, out_bf16=True)
    end.record()
    torch.cuda.synchronize()
    err = capi.averis_last_device_error()
    if err != 0:
        raise SystemExit(f"device-side wait gave up (code {err})")
    print(f"moe {args.mode}: {start.elapsed_time(end) / args.iters:.3f} ms/iter (eager, includes host launch overhead)")


if __name__ == "__main__":
    main()

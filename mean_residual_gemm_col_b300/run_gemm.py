"""Run one NVFP4 GEMM (averis_gemm, bf16 output) of M x N x K on the GPU.

A small driver for profiling the GEMM kernel alone through the C ABI: the
operands are NVFP4 quantizations (no mean split) of seeded synthetic
activations of M x K and N x K; each iteration is one eager launch on the
current stream, timed with CUDA events.

  python -m mean_residual_gemm_col_b300.run_gemm --m 8192 --n 8192 --k 8192 [--iters 3]
"""

from __future__ import annotations

import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--m", type=int, default=8192)
    ap.add_argument("--n", type=int, default=8192)
    ap.add_argument("--k", type=int, default=8192)
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args(argv)

    import torch

    import workloads
    from mean_residual_gemm_col_b300 import capi

    dev = torch.device("cuda", torch.cuda.current_device())
    capi.load()
    ops = []
    for seed, rows in ((1, args.m), (2, args.n)):
        x = workloads.torch_activation(seed, rows, args.k, spike=30.0, device=dev)
        ops.append(capi.averis_quantize(x, 0, want_col=False)["row"])
        del x
    out = torch.empty(args.m, args.n, dtype=torch.bfloat16, device=dev)
    times = []
    for _ in range(args.iters):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        capi.averis_gemm(ops[0], ops[1], out_bf16=True, out=out)
        e.record()
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e) * 1e3)
    err = capi.averis_last_device_error()
    print(json.dumps({"m": args.m, "n": args.n, "k": args.k, "us_per_launch": [round(t, 1) for t in times],
                      "device_error": err}))
    if err != 0:
        raise SystemExit(1)


if __name__ == "__main__":
    main()

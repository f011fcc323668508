"""Benchmark: Averis W4A4G4 linear fwd+bwd on the Qwen3-0.6B linears (l = 8192).

One step = forward + backward of the four Qwen3-0.6B-shaped linears (QKV
1024->4096, o_proj 2048->1024, gate_up 1024->6144, down 3072->1024) at
l = 8192 tokens (b=4, s=2048): weight quantize, mean-split quantize of X,
rank-one row, forward GEMM, mean-split quantize of D, rank-one row,
input-gradient GEMM, weight-gradient GEMM -- all through the C ABI, captured
in one CUDA graph.  Useful FLOPs per linear: 6 l m n + 5 m n.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  Under torchrun each rank runs an independent replica
(weak scaling: the linears of different batches are independent problems,
no data-path collective); rank 0 reports the whole-job throughput over the
max-over-ranks time.  ``--impl reference`` times the CPU float64 oracle on a
bounded sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "Averis W4A4G4 linear fwd+bwd TFLOP/s, % FP4 peak, overhead vs vanilla NVFP4"
L = workloads.QWEN3_L
LINEARS = workloads.QWEN3_06B_LINEARS
FP4_OVER_BF16 = 13.5 / 2.25     # nominal dense FP4 : BF16 tensor-core ratio
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
CPU_SAMPLE_TOKENS = 256


# DRAM bytes (read + write) per GEMM launch, averaged over the 12 one-GEMM
# launches that the per-kernel timing replays (NVTX range gemm_group_timed) in
# one ncu capture, keyed by a hash of the GEMM sources the capture was taken
# on; any other source reports null.
GEMM_TRAFFIC = {"50c6fd9531fd4445": 244.70e6 / 12}


def gemm_traffic_per_launch():
    import hashlib

    h = hashlib.sha256()
    for f in ("gemm.cuh", "ptx.cuh", "debug.cuh"):
        with open(os.path.join(ROOT, "mean_residual_gemm_col_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return GEMM_TRAFFIC.get(h.hexdigest()[:16])


def flops_per_step(l=L):
    return sum(6.0 * l * m * n + 5.0 * m * n for _, m, n in LINEARS)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------ distributed --

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch
        import torch.distributed as dist

        rank = int(os.environ["RANK"])
        local = int(os.environ.get("LOCAL_RANK", rank))
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return rank, ws
    return 0, 1


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v, ws):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks --

class _Nvml:
    """Read-only NVML queries through ctypes (libnvidia-ml ships with the NVIDIA driver)."""

    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, cuda_index):
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        bus = self._pci_bus_id(cuda_index)
        if bus is None or lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) != 0:
            n = ctypes.c_uint()
            lib.nvmlDeviceGetCount_v2(ctypes.byref(n))
            if lib.nvmlDeviceGetHandleByIndex_v2(0 if n.value == 1 else cuda_index, ctypes.byref(self.h)) != 0:
                raise OSError("no NVML handle for the device")
        self._reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
        self.max_mhz = float(mx.value)

    @staticmethod
    def _pci_bus_id(i):
        try:
            import torch

            p = torch.cuda.get_device_properties(i)
            return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        except Exception:
            return None

    def sample(self, with_power=True):
        u, r = ctypes.c_uint(), ctypes.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(u)) != 0:       # NVML_CLOCK_SM
            raise OSError("nvmlDeviceGetClockInfo failed")
        self._reasons(self.h, ctypes.byref(r))
        pw = None
        if with_power:                      # the slowest query: not on every tick
            p = ctypes.c_uint()
            if self.lib.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(p)) == 0:
                pw = p.value / 1000.0
        return (float(u.value), self.max_mhz, pw, {k for k, b in self.REASONS.items() if r.value & b})


class ClockSampler:
    """SM clock, power and throttle reasons sampled while the timed region runs.

    Read-only NVML queries every millisecond or so on a thread, so that even a timed region
    of a few milliseconds gets samples; nvidia-smi at 200 ms if NVML cannot be
    loaded.  ``mark()`` opens and closes the timed region: the summary reports
    the samples taken inside it, and separately every sample from the start of
    the sampler (warm-up and timed region) as the under-load record.
    """

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.rows = []       # (t, sm_mhz, max_mhz, power_w, set of active reason names)
        self.window = [None, None]
        self.proc = None
        self.path = None
        self.thread = None
        self.stop = None
        self.nvml_error = None

    def mark(self, which):
        self.window[0 if which == "start" else 1] = time.perf_counter()

    def _poll(self, nv):
        k = 0
        while not self.stop.is_set():
            try:
                t = time.perf_counter()
                self.rows.append((t,) + nv.sample(with_power=k % 10 == 0))
            except Exception as e:
                self.nvml_error = f"{type(e).__name__}: {e}"[:120]
                break
            k += 1
            time.sleep(0.001)

    def __enter__(self):
        import threading

        try:
            nv = _Nvml(self.dev)
            self.stop = threading.Event()
            self.thread = threading.Thread(target=self._poll, args=(nv,), daemon=True)
            self.thread.start()
            return self
        except Exception as e:  # no NVML: fall back to nvidia-smi
            self.thread = None
            self.nvml_error = f"{type(e).__name__}: {e}"[:120]
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.4)
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            self.stop.set()
            self.thread.join(timeout=5)
            return
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.close()
        if self.path and os.path.exists(self.path):
            def num(v):
                try:
                    return float(v)
                except ValueError:
                    return None
            now = time.perf_counter()
            with open(self.path) as f:
                for ln in f:
                    p = [v.strip() for v in ln.split(",")]
                    if len(p) >= 9 and num(p[1]) is not None:
                        self.rows.append((now, num(p[1]), num(p[2]), num(p[3]),
                                          {self.NAMES[i] for i in range(4) if p[5 + i].lower().startswith("active")}))
            os.unlink(self.path)

    @staticmethod
    def _stats(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [r[1] for r in rows]
        mx = [r[2] for r in rows if r[2] is not None]
        pw = [r[3] for r in rows if r[3] is not None]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": sorted(set().union(*(r[4] for r in rows))), "samples": len(rows)}

    def summary(self):
        t0, t1 = self.window
        inside = [r for r in self.rows if t0 is not None and t1 is not None and t0 <= r[0] <= t1]
        if self.thread is None:            # nvidia-smi rows carry no time of their own
            inside = list(self.rows)
        out = self._stats(inside)
        out["source"] = "nvml ~1 ms" if self.thread is not None else "nvidia-smi 200 ms"
        out["window"] = "timed region"
        out["under_load"] = self._stats(self.rows)
        out["under_load"]["window"] = "warm-up and timed region"
        if self.nvml_error:
            out["nvml_error"] = self.nvml_error
        return out


# ----------------------------------------------------------- GPU workload --

class Layer:
    """One linear's inputs, outputs and every intermediate buffer, preallocated."""

    def __init__(self, name, m, n, seed, device, l=L, share=None):
        import torch
        from mean_residual_gemm_col_b300 import capi

        self.name, self.m, self.n = name, m, n
        if share is None:
            self.x, self.w, self.d = workloads.torch_linear_case(seed, l, m, n, spike=workloads.QWEN3_SPIKE,
                                                                 device=device)
            self.state = capi.FwdState.empty(l, m, device)
            self.y = torch.empty(l, n, dtype=torch.bfloat16, device=device)
            self.dx = torch.empty(l, m, dtype=torch.bfloat16, device=device)
            self.dw = torch.empty(m, n, dtype=torch.float32, device=device)
        else:
            # another layer of a stack: its own weights, the shared activations and buffers
            _, self.w, _ = workloads.torch_linear_case(seed, 64, m, n, device=device)
            self.x, self.d, self.state, self.y, self.dx, self.dw = (share.x, share.d, share.state, share.y,
                                                                   share.dx, share.dw)
        self.w_n = capi.NVFP4Tensor.empty(m, n, device)
        self.w_m = capi.NVFP4Tensor.empty(n, m, device)
        self.xq = None   # standalone quantized X / D (same kernels) for the per-kernel timing
        self.dq = None


def quant_weight_into(ly, flags, key="wq"):
    from mean_residual_gemm_col_b300 import capi

    lib = capi.load()
    ws = capi.workspace(lib.averis_quantize_workspace_bytes(ly.m, ly.n, flags), ly.w.device, key)
    a, b = ly.w_n.struct(), ly.w_m.struct()
    capi._check(lib.averis_quantize_weight(capi._ptr(ly.w), ly.m, ly.n, flags, ctypes.byref(a), ctypes.byref(b),
                                           capi._ptr(ws), ws.numel(), capi._stream(ly.w.device)),
                "averis_quantize_weight")


_SIDE = {}


def side_stream(device, k=0):
    import torch

    if (device, k) not in _SIDE:
        _SIDE[(device, k)] = torch.cuda.Stream(device)
    return _SIDE[(device, k)]


def run_step(layers, mode):
    """Enqueue one fwd+bwd step of every layer.

    The weights do not depend on the activations, so the layers' weight
    quantizations run in layer order on one side stream (joined per layer by
    an event) while the main stream runs the layers' forward and backward
    passes in order.  Measured on the Qwen3 step: 0.566 ms against 0.571 ms
    with one side stream per layer (four quantizes competing for the SMs at
    once) and 0.597 ms with the weight quantizes on the main stream.
    """
    import torch
    from mean_residual_gemm_col_b300 import capi

    split = mode in ("averis", "averis_h16")
    hf = capi.AVERIS_HADAMARD16 if mode in ("averis_h16", "nvfp4_h16") else 0
    main = torch.cuda.current_stream()
    side = side_stream(main.device)
    side.wait_stream(main)
    ready = []
    with torch.cuda.stream(side):
        for ly in layers:
            quant_weight_into(ly, hf, key="wq")
            ev = torch.cuda.Event()
            ev.record(side)
            ready.append(ev)
    for ly, ev in zip(layers, ready):
        main.wait_event(ev)
        if split:
            capi.averis_linear_fwd(ly.x, ly.w_m, capi.AVERIS_MEAN_SPLIT | hf, out_bf16=True, state=ly.state, y=ly.y)
            capi.averis_linear_bwd(ly.d, ly.state, ly.w_n, capi.AVERIS_MEAN_SPLIT | hf, out_bf16=True, dx=ly.dx,
                                   dw=ly.dw)
        else:
            capi.nvfp4_linear_fwd(ly.x, ly.w_m, hf, out_bf16=True, state=ly.state, y=ly.y)
            capi.nvfp4_linear_bwd(ly.d, ly.state, ly.w_n, hf, out_bf16=True, dx=ly.dx, dw=ly.dw)


def launches_per_step(mode):
    """Kernels one step enqueues: per linear, weight quantize (stats, quantize),
    forward (stats, quantize, GEMM), backward (stats, quantize, one GEMM launch
    carrying both dW and dX).  With the rotation, a quantize without the mean
    split (the weights; every activation in nvfp4_h16) runs the rotated-maximum
    pass instead of the stats pass, and one with the split runs both."""
    w = 2
    a = 3 if mode == "averis_h16" else 2
    return (w + (a + 1) + (a + 1)) * len(LINEARS)


def kernel_groups(layers):
    """Callables that each enqueue one family of launches of a step (for per-kernel timing)."""
    from mean_residual_gemm_col_b300 import capi

    lib = capi.load()

    def gemms():
        for ly in layers:
            st = ly.state
            capi.averis_gemm(st.x_row, ly.w_m, col_add=None, out_bf16=True, out=ly.y)
            capi.averis_gemm(ly.dq["row"], ly.w_n, out_bf16=True, out=ly.dx)
            capi.averis_gemm(st.x_col, ly.dq["col"], row_vec=st.mu_hat, col_vec=ly.dq["mu_hat"], outer=float(L),
                             out=ly.dw)

    def quants():
        for ly in layers:
            for t, rows, cols, q in ((ly.x, L, ly.m, ly.xq), (ly.d, L, ly.n, ly.dq)):
                ws = capi.workspace(lib.averis_quantize_workspace_bytes(rows, cols, 1), t.device, "kq")
                ms, rs, cs = q["mu_q"].struct(), q["row"].struct(), q["col"].struct()
                capi._check(lib.averis_quantize(capi._ptr(t), rows, cols, capi.AVERIS_MEAN_SPLIT, capi._ptr(q["mu"]),
                                                ctypes.byref(ms), capi._ptr(q["mu_hat"]), ctypes.byref(rs),
                                                ctypes.byref(cs), capi._ptr(ws), ws.numel(),
                                                capi._stream(t.device)), "averis_quantize")

    return {"gemm": gemms, "quantize": quants}


def gemm_bytes_and_flops(layers):
    """Algorithmic bytes and flops of the 12 GEMMs of one step (Y, dX, dW per linear)."""
    from mean_residual_gemm_col_b300 import layout

    def nv(rows, cols):                                   # codes + block scales
        return rows * layout.cdiv(cols, 16) * 8 + rows * layout.cdiv(cols, 16)

    byts = flops = 0.0
    for ly in layers:
        m, n = ly.m, ly.n
        byts += nv(L, m) + nv(n, m) + 2.0 * L * n        # Y (bf16)
        byts += nv(L, n) + nv(m, n) + 2.0 * L * m        # dX (bf16)
        byts += nv(m, L) + nv(n, L) + 4.0 * m * n        # dW (fp32)
        flops += 6.0 * L * m * n
    return byts, flops


def time_graph(graph, steps, stream):
    import torch

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        graph.replay()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def capture(fn):
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def run_ours(args, rank, ws):
    import torch
    from mean_residual_gemm_col_b300 import capi

    device = torch.device("cuda", torch.cuda.current_device())
    capi.load()
    layers = [Layer(name, m, n, seed=1000 * rank + i, device=device) for i, (name, m, n) in enumerate(LINEARS)]
    for ly in layers:
        ly.xq = capi.averis_quantize(ly.x, capi.AVERIS_MEAN_SPLIT)
        ly.dq = capi.averis_quantize(ly.d, capi.AVERIS_MEAN_SPLIT)
    modes = ["averis", "nvfp4", "averis_h16", "nvfp4_h16"]
    for mode in modes:       # eager warm-up: kernel attributes, workspaces, first-call setup
        run_step(layers, mode)
    torch.cuda.synchronize()
    if capi.averis_last_device_error() != 0:
        raise RuntimeError("device-side wait timed out during warm-up")
    graphs = {mode: capture(lambda mode=mode: run_step(layers, mode)) for mode in modes}
    groups = kernel_groups(layers)
    for g in groups.values():
        g()
    torch.cuda.synchronize()
    ggraphs = {k: capture(v) for k, v in groups.items()}
    stream = torch.cuda.current_stream()

    # ---- headline: K steps of the Averis fwd+bwd, barrier + sync on both sides
    with ClockSampler(torch.cuda.current_device()) as clk:
        for _ in range(args.warmup):
            graphs["averis"].replay()
        torch.cuda.synchronize()
        barrier(ws)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        clk.mark("start")
        torch.cuda.nvtx.range_push("averis_timed")
        ms = time_graph(graphs["averis"], args.steps, stream)
        torch.cuda.nvtx.range_pop()
        clk.mark("end")
        wall = time.perf_counter() - t0
        barrier(ws)
    clocks = clk.summary()
    ms = max_over_ranks(ms, ws)

    # ---- comparison modes and per-kernel timing (same inputs, same launches)
    for _ in range(args.warmup):
        for m in ("nvfp4", "averis_h16", "nvfp4_h16"):
            graphs[m].replay()
    def timed(mode):
        torch.cuda.nvtx.range_push(f"{mode}_timed")
        t = time_graph(graphs[mode], args.steps, stream)
        torch.cuda.nvtx.range_pop()
        return max_over_ranks(t, ws)

    ms_van = timed("nvfp4")
    ms_had = timed("averis_h16")
    ms_vhad = timed("nvfp4_h16")
    kern = {}
    for k, g in ggraphs.items():
        g.replay()
        torch.cuda.nvtx.range_push(f"{k}_group_timed")
        kern[k] = time_graph(g, args.steps, stream)
        torch.cuda.nvtx.range_pop()

    # ---- end to end through the API with host buffers: H2D inputs, step, D2H outputs
    # two sets of the step's device tensors, each with its own graph: step k uses set
    # k % 2, so the inputs of step k+1 go up while step k computes and step k-1's
    # outputs come down (one copy stream per direction)
    layers_b = [Layer(name, m, n, seed=1000 * rank + i, device=device) for i, (name, m, n) in enumerate(LINEARS)]
    run_step(layers_b, "averis")
    torch.cuda.synchronize()
    sets = [(layers, graphs["averis"]), (layers_b, capture(lambda: run_step(layers_b, "averis")))]
    dev_in = [[t for ly in lys for t in (ly.x, ly.w, ly.d)] for lys, _ in sets]
    dev_out = [[t for ly in lys for t in (ly.y, ly.dx, ly.dw)] for lys, _ in sets]
    host_in = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dev_in[0]]
    for h, t in zip(host_in, dev_in[0]):
        h.copy_(t)
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dev_out[0]]
    h2d = sum(t.numel() * t.element_size() for t in dev_in[0])
    d2h = sum(t.numel() * t.element_size() for t in dev_out[0])
    h2d_s, d2h_s = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def e2e_steps(n, first):
        comp_done, out_done = [None, None], [None, None]
        for k in range(n):
            s = k % 2
            in_done = torch.cuda.Event()
            h2d_s.wait_event(first if comp_done[s] is None else comp_done[s])  # step k-2 has read set s
            with torch.cuda.stream(h2d_s):
                for h, t in zip(host_in, dev_in[s]):
                    t.copy_(h, non_blocking=True)
            in_done.record(h2d_s)
            stream.wait_event(in_done)
            if out_done[s] is not None:
                stream.wait_event(out_done[s])  # step k-2's outputs have left set s
            sets[s][1].replay()
            comp_done[s] = torch.cuda.Event()
            comp_done[s].record(stream)
            d2h_s.wait_event(comp_done[s])
            with torch.cuda.stream(d2h_s):
                for h, t in zip(host_out, dev_out[s]):
                    h.copy_(t, non_blocking=True)
            out_done[s] = torch.cuda.Event()
            out_done[s].record(d2h_s)
        stream.wait_event(out_done[(n - 1) % 2])  # the copy stream is in order: the last copy ends last

    go = torch.cuda.Event()
    go.record(stream)
    e2e_steps(1, go)
    torch.cuda.synchronize()
    e_steps = max(3, args.steps // 4)
    barrier(ws)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    e2e_steps(e_steps, start)
    end.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(start.elapsed_time(end) / e_steps, ws)
    if capi.averis_last_device_error() != 0:
        raise RuntimeError("device-side wait timed out during the timed region")

    flops = flops_per_step()
    peaks, src = load_peaks()
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    fp4_sus = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * FP4_OVER_BF16
    value = flops * ws / (ms * 1e-3) / 1e12
    gb, gf = gemm_bytes_and_flops(layers)
    n_gemm = 3 * len(LINEARS)
    g_ms = kern["gemm"] / n_gemm                  # average GEMM launch
    q_ms = kern["quantize"] / (2 * len(LINEARS))  # average quantize call (stats + quantize kernels)
    q_bytes = sum(3.125 * L * (ly.m + ly.n) for ly in layers) / (2 * len(LINEARS))
    t_tensor = gf / (fp4_peak * 1e12)
    t_hbm = gb / (peaks["hbm_gbs"] * 1e9)
    if t_tensor >= t_hbm:
        roof = {"bound": "tensor", "achieved": gf / n_gemm / (g_ms * 1e-3) / 1e12, "peak": fp4_peak,
                "unit": "TFLOP/s"}
        psrc = f"{src} bf16_tflops x {FP4_OVER_BF16:g} (nominal FP4:BF16 ratio)"
    else:
        roof = {"bound": "hbm", "achieved": gb / n_gemm / (g_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
        psrc = f"{src} hbm_gbs"
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = gemm_traffic_per_launch()
    roof["kernel"] = ("gemm_nvfp4_kernel, mean of the 12 GEMMs of a step, one launch each "
                      "(the step itself runs a layer's dW and dX GEMMs in one launch)")
    roof["peak_source"] = psrc
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 (e2m1 x e2m1, fp32 accumulate; bf16 inputs, bf16 Y/dX, fp32 dW)",
        "data": "synthetic: planted rank-one mean + N(0,1) + 0.1% spikes x30 (seeded torch generator per layer)",
        "config": {"workload": "Qwen3-0.6B linears (qkv 1024->4096, o_proj 2048->1024, gate_up 1024->6144, "
                               "down 3072->1024), fwd+bwd", "l": L, "b": 4, "s": 2048,
                   "parallelism": f"replicas x{ws}", "l2": "step inputs 318 MB > 126 MB L2; no flush",
                   "cuda_graph": True},
        "fp4_peak_frac": round(value / ws / fp4_peak, 4),
        "fp4_peak_tflops": round(fp4_peak, 1),
        "fp4_peak_sustained_tflops": round(fp4_sus, 1),
        "overhead_vs_vanilla": round((ms - ms_van) / ms_van, 4),
        "overhead_h16_vs_vanilla": round((ms_had - ms_van) / ms_van, 4),
        "overhead_nvfp4_h16_vs_vanilla": round((ms_vhad - ms_van) / ms_van, 4),
        "averis_overhead_over_hadamard_overhead": round((ms - ms_van) / max(ms_vhad - ms_van, 1e-9), 4),
        "ms_per_step_vanilla": round(ms_van, 4),
        "ms_per_step_averis_h16": round(ms_had, 4),
        "ms_per_step_nvfp4_h16": round(ms_vhad, 4),
        "roofline": {k: (round(v, 4) if isinstance(v, float) else v) for k, v in roof.items()},
        "kernels_ms_per_step": {k: round(v, 4) for k, v in kern.items()},
        "quantize_pass": {"avg_ms": round(q_ms, 4), "algorithmic_gbs": round(q_bytes / (q_ms * 1e-3) / 1e9, 1),
                          "hbm_frac": round(q_bytes / (q_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                          "bytes_per_elem": 3.125},
        "e2e": {"value": round(flops * ws / (ms_e2e * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 3),
                "copies": "pinned host buffers; two sets of device buffers, step k on set k % 2; one copy "
                          "stream per direction: step k+1's inputs go up while step k computes and step k-1's "
                          "outputs come down"},
        "gpu_launches": launches_per_step("averis") * args.steps,
        "clocks": clocks,
        "wall_s_timed": round(wall, 4),
    }
    if not args.no_extras:
        del graphs, ggraphs
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        # each extra measurement reports its own failure instead of losing the line
        for key, fn, fargs in (("gemm_alone", gemm_alone, (fp4_peak,)), ("quantize_sweep", quantize_sweep, (peaks,)),
                               ("preprocess_vs_hadamard", preprocess_comparison, ()),
                               ("stack_28_layers", stack_comparison, ()), ("moe_expert_ffn", moe_comparison, ()),
                               ("quant_error_qkv", quant_error_diagnostic, (layers[0],))):
            try:
                line[key] = fn(*fargs)
            except Exception as e:  # noqa: BLE001
                line[key] = {"error": f"{type(e).__name__}: {e}"[:300]}
                try:
                    torch.cuda.synchronize()
                    torch.cuda.empty_cache()
                except Exception:  # noqa: BLE001
                    pass
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return line


# ------------------------------------------------ quantize-only measurements --

def _time_each(fn, iters, flush, stream):
    """Median device time of ``fn`` (ms), L2 flushed before each timed call."""
    import torch

    ts = []
    for _ in range(iters):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        torch.cuda.synchronize()
        ts.append(s.elapsed_time(e))
    return statistics.median(ts)


def _quantizer(x, flags):
    """A closure that runs the fused quantize pass on x with preallocated outputs."""
    import torch
    from mean_residual_gemm_col_b300 import capi

    lib = capi.load()
    R, C = x.shape
    dev = x.device
    row = capi.NVFP4Tensor.empty(R, C, dev)
    col = capi.NVFP4Tensor.empty(C, R, dev)
    mu = torch.zeros(C, device=dev)
    muh = torch.zeros(C, device=dev)
    muq = capi.NVFP4Tensor.empty(1, C, dev)
    ws = capi.workspace(lib.averis_quantize_workspace_bytes(R, C, flags), dev, "sweep")
    rs, cs, ms = row.struct(), col.struct(), muq.struct()
    st = capi._stream(dev)

    def run():
        capi._check(lib.averis_quantize(capi._ptr(x), R, C, flags, capi._ptr(mu), ctypes.byref(ms), capi._ptr(muh),
                                        ctypes.byref(rs), ctypes.byref(cs), capi._ptr(ws), ws.numel(), st),
                    "averis_quantize")
    return run, (row, col, mu, muh, muq, ws)


def quantize_sweep(peaks, iters=5):
    """The quantize-only sweep: fused mean-split NVFP4 of an l x m bf16 activation
    into both layouts, l in {4096, 16384, 65536} x m in {1024, 2048, 4096, 8192}.
    Algorithmic bytes per element: 2 (bf16 read) + 2 x (0.5 + 1/16) (both layouts)."""
    import torch
    from mean_residual_gemm_col_b300 import capi

    dev = torch.device("cuda", torch.cuda.current_device())
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    out = []
    for l in workloads.QUANT_SWEEP_L:
        for m in workloads.QUANT_SWEEP_M:
            x = workloads.torch_activation(l * 10 + m, l, m, spike=50.0, device=dev)
            run, keep = _quantizer(x, capi.AVERIS_MEAN_SPLIT)
            run()
            torch.cuda.synchronize()
            ms = _time_each(run, iters, flush, stream)
            gbs = 3.125 * l * m / (ms * 1e-3) / 1e9
            out.append({"l": l, "m": m, "us": round(ms * 1e3, 1), "algorithmic_gbs": round(gbs, 1),
                        "hbm_frac": round(gbs / peaks["hbm_gbs"], 3)})
            del x, run, keep
    torch.cuda.empty_cache()
    return out


def gemm_alone(fp4_peak, n=8192, sets=3, reps=10, iters=9):
    """One NVFP4 GEMM of n x n x n (bf16 output, no epilogue terms) through
    averis_gemm, its operands quantized from seeded synthetic activations.
    Timed two ways: back to back in a CUDA graph over `sets` operand pairs taken
    in turn (226 MB of operands for n = 8192, more than L2, so each launch
    streams its operands from HBM), and as the median of single launches with
    L2 flushed (overwritten) before each."""
    import torch
    from mean_residual_gemm_col_b300 import capi

    dev = torch.device("cuda", torch.cuda.current_device())
    ops = []
    for k in range(sets):
        pair = []
        for seed in (2 * k + 1, 2 * k + 2):
            x = workloads.torch_activation(seed, n, n, spike=30.0, device=dev)
            pair.append(capi.averis_quantize(x, 0, want_col=False)["row"])
            del x
        ops.append(pair)
    out = torch.empty(n, n, dtype=torch.bfloat16, device=dev)

    def run_all():
        for a, b in ops:
            capi.averis_gemm(a, b, out_bf16=True, out=out)

    run_all()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run_all()
    g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(reps):
        g.replay()
    end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / (reps * sets)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ms_flush = _time_each(lambda: capi.averis_gemm(ops[0][0], ops[0][1], out_bf16=True, out=out), iters, flush,
                          stream)
    tflops = 2.0 * n ** 3 / (ms * 1e-3) / 1e12
    tflops_flush = 2.0 * n ** 3 / (ms_flush * 1e-3) / 1e12
    del ops, out, flush, g
    torch.cuda.empty_cache()
    return {"m": n, "n": n, "k": n, "us": round(ms * 1e3, 1), "tflops": round(tflops, 1),
            "fp4_peak_frac": round(tflops / fp4_peak, 4),
            "l2": f"{sets} operand pairs taken in turn, more than L2 together; CUDA graph",
            "us_l2_flushed": round(ms_flush * 1e3, 1), "fp4_peak_frac_l2_flushed": round(tflops_flush / fp4_peak, 4)}


def preprocess_comparison(iters=3):
    """Quantize-pass latency of vanilla NVFP4, Averis (mean split) and NVFP4 with the
    16x16 Hadamard rotation on activations of 512 x 2048 tokens, d = 4096 / 8192
    (the shapes of the pages' preprocessing-latency table).  The Averis and
    Hadamard preprocessing costs are the differences to the vanilla pass."""
    import torch
    from mean_residual_gemm_col_b300 import capi

    dev = torch.device("cuda", torch.cuda.current_device())
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    res = []
    for d in (4096, 8192):
        l = 512 * 2048
        x = workloads.torch_activation(d, l, d, spike=50.0, device=dev)
        t = {}
        for name, flags in (("vanilla", 0), ("averis", capi.AVERIS_MEAN_SPLIT), ("hadamard", capi.AVERIS_HADAMARD16)):
            run, keep = _quantizer(x, flags)
            run()
            torch.cuda.synchronize()
            t[name] = _time_each(run, iters, flush, stream)
            del run, keep
            torch.cuda.empty_cache()
        ov_a, ov_h = t["averis"] - t["vanilla"], t["hadamard"] - t["vanilla"]
        res.append({"tokens": l, "d": d, "ms_vanilla": round(t["vanilla"], 3), "ms_averis": round(t["averis"], 3),
                    "ms_hadamard": round(t["hadamard"], 3), "averis_extra_ms": round(ov_a, 3),
                    "hadamard_extra_ms": round(ov_h, 3),
                    "hadamard_extra_over_averis_extra": round(ov_h / ov_a, 2) if ov_a > 0 else None})
        del x
        torch.cuda.empty_cache()
    return res


def _dequant_gpu(t):
    """float32 [rows, cols] value of an NVFP4 tensor of the library (measurement only)."""
    import torch
    from mean_residual_gemm_col_b300 import layout

    dev = t.codes.device
    e2m1 = torch.tensor([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6], device=dev)
    c = t.codes.long()
    vals = torch.stack([e2m1[c & 15], e2m1[c >> 4]], dim=-1).reshape(t.rows, -1)[:, : t.cols]
    off = torch.from_numpy(layout.scale_offsets(t.rows, t.cols)).to(dev)
    sc = t.scales.view(torch.float8_e4m3fn).float()[off]
    return (vals.reshape(t.rows, -1, 16) * sc[:, :, None]).reshape(t.rows, -1)[:, : t.cols] * t.tensor_scale


def quant_error_diagnostic(layer):
    """Relative NVFP4 error ||deq(Q(T)) - T|| / ||T|| of one linear's activation X and
    output gradient D, quantized directly (vanilla) and as mean + residual (Averis:
    deq(Q(T - 1 mu)) + 1 deq(Q(mu)))."""
    import torch
    from mean_residual_gemm_col_b300 import capi

    res = {}
    for name, t in (("X", layer.x), ("D", layer.d)):
        ref = t.float()
        van = capi.averis_quantize(t, 0, want_col=False)
        av = capi.averis_quantize(t, capi.AVERIS_MEAN_SPLIT, want_col=False)
        e_van = _dequant_gpu(van["row"]) - ref
        e_av = _dequant_gpu(av["row"]) + av["mu_hat"][None, :] - ref
        nrm = torch.linalg.vector_norm(ref)
        res[name] = {"vanilla": round(float(torch.linalg.vector_norm(e_van) / nrm), 5),
                     "averis": round(float(torch.linalg.vector_norm(e_av) / nrm), 5)}
        del ref, van, av, e_van, e_av
    return res


def moe_comparison(steps=3, warmup=2):
    """Mixture-of-experts expert FFN: hidden 2048, 64 experts, top-8, expert FFN
    768 (gate_up 2048 -> 1536, down 768 -> 2048), 16384 tokens routed with
    Zipf(1.1) popularity; the means are per expert over its tokens.  One step is
    the weight quantize, forward and backward of both grouped linears."""
    import torch
    from mean_residual_gemm_col_b300 import capi

    cfg = workloads.MOE
    dev = torch.device("cuda", torch.cuda.current_device())
    counts = workloads.moe_routing(0, cfg["tokens"], cfg["experts"], cfg["top_k"], cfg["zipf"])
    offsets = np.concatenate([[0], np.cumsum(counts)])
    rows = int(offsets[-1])
    shapes = (("gate_up", cfg["hidden"], 2 * cfg["ffn"]), ("down", cfg["ffn"], cfg["hidden"]))
    lin = []
    for i, (name, m, n) in enumerate(shapes):
        x = workloads.torch_activation(31 + i, rows, m, spike=workloads.QWEN3_SPIKE, device=dev)
        _, _, d = workloads.torch_linear_case(41 + i, rows, 16, n, device=dev)
        # the experts' weights stacked [E, m, n], quantized in one grouped call per step
        w = torch.stack([workloads.torch_linear_case(100 * i + e, 16, m, n, device=dev)[1]
                         for e in range(cfg["experts"])])
        wn = [capi.NVFP4Tensor.empty(m, n, dev) for _ in w]
        wm = [capi.NVFP4Tensor.empty(n, m, dev) for _ in w]
        gl = capi.GroupedLinear(offsets, m, n, wm, wn, dev)
        y = torch.empty(rows, n, dtype=torch.bfloat16, device=dev)
        dx = torch.empty(rows, m, dtype=torch.bfloat16, device=dev)
        lin.append((m, n, x, d, w, wn, wm, gl, y, dx))

    def step(flags):
        for m, n, x, d, w, wn, wm, gl, y, dx in lin:
            capi.averis_quantize_weight_grouped(w, 0, w_n=wn, w_m=wm)
            gl.fwd(x, flags, out_bf16=True, y=y)
            gl.bwd(d, flags, out_bf16=True, dx=dx)

    flops = sum(6.0 * rows * m * n + 5.0 * m * n * cfg["experts"] for m, n, *_ in lin)
    stream = torch.cuda.current_stream()
    res = {"experts": cfg["experts"], "top_k": cfg["top_k"], "tokens": cfg["tokens"],
           "rows_per_expert_max": int(counts.max()), "rows_per_expert_min": int(counts.min()),
           "gflop_per_step": round(flops / 1e9, 1),
           "note": "all experts quantized in one launch chain per tensor (weights: one grouped call per linear), "
                   "expert GEMMs in one persistent launch per product (Y; dW; dX), pair ranges balanced by K"}
    for name, flags in (("nvfp4", 0), ("averis", capi.AVERIS_MEAN_SPLIT)):
        step(flags)
        torch.cuda.synchronize()
        g = capture(lambda flags=flags: step(flags))
        for _ in range(warmup):
            g.replay()
        t = time_graph(g, steps, stream)
        res[f"ms_{name}"] = round(t, 3)
        res[f"tflops_{name}"] = round(flops / (t * 1e-3) / 1e12, 1)
        del g
    res["overhead_averis"] = round((res["ms_averis"] - res["ms_nvfp4"]) / res["ms_nvfp4"], 4)
    del lin
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def stack_comparison(steps=3, warmup=2):
    """28-layer stack of the Qwen3-0.6B linears at l = 16384 (b = 8, s = 2048),
    fwd + bwd, in three modes: vanilla NVFP4, Averis, Averis + 16x16 Hadamard on
    the residual.  Every layer has its own weights (seed = layer); the planted-mean
    activations and output gradients are shared by all layers."""
    import torch

    dev = torch.device("cuda", torch.cuda.current_device())
    lst = workloads.STACK_L
    base = [Layer(name, m, n, seed=5000 + i, device=dev, l=lst) for i, (name, m, n) in enumerate(LINEARS)]
    stack = []
    for layer in range(workloads.STACK_LAYERS):
        for i, (name, m, n) in enumerate(LINEARS):
            stack.append(Layer(name, m, n, seed=layer, device=dev, l=lst, share=base[i]))
    flops = workloads.STACK_LAYERS * flops_per_step(lst)
    out = {"layers": workloads.STACK_LAYERS, "l": lst, "tflop_per_step": round(flops / 1e12, 3)}
    stream = torch.cuda.current_stream()
    ms = {}
    for mode in ("nvfp4", "averis", "averis_h16"):
        run_step(stack, mode)
        torch.cuda.synchronize()
        g = capture(lambda mode=mode: run_step(stack, mode))
        for _ in range(warmup):
            g.replay()
        ms[mode] = time_graph(g, steps, stream)
        del g
    for mode, t in ms.items():
        out[f"ms_{mode}"] = round(t, 3)
        out[f"tflops_{mode}"] = round(flops / (t * 1e-3) / 1e12, 1)
    out["overhead_averis"] = round((ms["averis"] - ms["nvfp4"]) / ms["nvfp4"], 4)
    out["overhead_averis_h16"] = round((ms["averis_h16"] - ms["nvfp4"]) / ms["nvfp4"], 4)
    del stack, base
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


# --------------------------------------------------------- CPU baseline ----

def blas_threads():
    """Threads of the BLAS NumPy calls into (threadpoolctl), else the OpenMP
    setting; with a note saying where the number came from (or why not)."""
    note = "threadpoolctl"
    try:
        from threadpoolctl import threadpool_info

        info = threadpool_info()
        n = [p["num_threads"] for p in info if p.get("user_api") == "blas"]
        if n:
            return max(n), "threadpoolctl: " + ", ".join(sorted({str(p.get("internal_api")) for p in info
                                                                  if p.get("user_api") == "blas"}))
        note = "threadpoolctl found no BLAS among " + ", ".join(str(p.get("internal_api")) for p in info)
    except Exception as e:  # report, do not fail the bench
        note = f"threadpoolctl unavailable: {type(e).__name__}"
    # the OpenBLAS that NumPy loaded, asked directly (its exported thread-count query)
    try:
        import ctypes

        with open("/proc/self/maps") as fh:
            libs = sorted({ln.split()[-1] for ln in fh if "openblas" in ln.lower() and ln.rstrip().endswith(".so")})
        for lib in libs:
            so = ctypes.CDLL(lib)
            for sym in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_", "openblas_get_num_threads"):
                fn = getattr(so, sym, None)
                if fn is not None:
                    fn.restype = ctypes.c_int
                    return int(fn()), note + f"; {os.path.basename(lib)} {sym}()"
    except Exception as e:
        note += f"; OpenBLAS query failed: {type(e).__name__}"
    v = os.environ.get("OMP_NUM_THREADS")
    if v and v.isdigit():
        return int(v), note + "; OMP_NUM_THREADS"
    return None, note


def cpu_baseline(target_s=10.0):
    """The oracle, as it stands, on a bounded sample of the workload.

    Sample: the first CPU_SAMPLE_TOKENS tokens of each of the four linears
    (same m, n), full forward + backward in float64 NumPy, repeated until
    ``target_s`` seconds of CPU time; throughput in the headline unit.
    """
    from oracle import averis as oav

    tok = CPU_SAMPLE_TOKENS
    total_flops = 0.0
    t_total = 0.0
    rep = 0
    while True:
        for i, (_, m, n) in enumerate(LINEARS):
            c = workloads.linear_case(100 + i + 10 * rep, tok, m, n, spike=workloads.QWEN3_SPIKE)
            x, w, d = (c.x.astype(np.float64), c.w.astype(np.float64), c.d.astype(np.float64))
            t0 = time.perf_counter()
            oav.linear_fwd_bwd(x, w, d)
            t_total += time.perf_counter() - t0
            total_flops += 6.0 * tok * m * n + 5.0 * m * n
        rep += 1
        if t_total >= target_s:
            break
    threads, note = blas_threads()          # after the oracle ran: its BLAS is loaded by now
    return {"value": round(total_flops / t_total / 1e12, 6), "unit": "TFLOP/s",
            "cores": threads or os.cpu_count(), "host_cpus": os.cpu_count(), "blas_threads": threads,
            "blas_threads_source": note,
            "kind": "oracle",
            "sample": f"{rep} x ({tok} of {L} tokens of each of the 4 linears, fwd+bwd), float64 NumPy, "
                      f"{t_total:.1f} s"}


def run_reference(args, rank, ws):
    """The CPU oracle as the reference arm: each step is one bounded sample of the workload."""
    if rank != 0:
        return None
    for _ in range(args.warmup):
        cpu_baseline(target_s=0.0)
    per = [cpu_baseline(target_s=0.0) for _ in range(args.steps)]
    v = statistics.median(c["value"] for c in per)
    step_flops = flops_per_step(CPU_SAMPLE_TOKENS)
    ms = step_flops / (v * 1e12) * 1e3
    cb = {"value": v, "unit": "TFLOP/s", "cores": per[-1]["cores"], "kind": "oracle",
          "sample": f"{CPU_SAMPLE_TOKENS} of {L} tokens of each of the 4 linears per step, fwd+bwd, float64 NumPy"}
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (NumPy PCG64, same recipe)",
        "config": {"workload": "Qwen3-0.6B linears (qkv 1024->4096, o_proj 2048->1024, gate_up 1024->6144, "
                               "down 3072->1024), fwd+bwd; bounded sample", "l": L},
        "cpu_baseline": cb,
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the quantize sweep and the preprocessing table")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, ws = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, rank, ws)
    else:
        line = run_ours(args, rank, ws)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()

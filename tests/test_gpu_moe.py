"""GPU parity of the grouped (mixture-of-experts) Averis linear layer.

Each expert's rows of the grouped input are an independent linear layer with
the expert's own weights and means (taken over the expert's tokens only); the
oracle runs the single-layer reference per expert, given the GPU's binary32
means.  The row split includes an empty expert and a one-row expert.
"""

import numpy as np
import pytest

from oracle import averis as oav
import workloads
from tests.gpu_util import to_dev_bf16, rel_fro

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.mark.parametrize("split", [True, False])
def test_grouped_linear_matches_per_expert_oracle(cuda_lib, split):
    import torch
    from mean_residual_gemm_col_b300 import capi

    m, n = 64, 128
    counts = [37, 0, 163, 1, 129]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    L = int(offsets[-1])
    g = workloads.rng(21)
    x = workloads.activation(g, L, m, spike=50.0)
    d = workloads.output_grad(g, L, n)
    ws = [workloads.weight(g, m, n) for _ in counts]
    w_n, w_m = zip(*[capi.averis_quantize_weight(to_dev_bf16(w)) for w in ws])
    gl = capi.GroupedLinear(offsets, m, n, list(w_m), list(w_n), "cuda")
    flags = capi.AVERIS_MEAN_SPLIT if split else 0
    xd, dd = to_dev_bf16(x), to_dev_bf16(d)
    y = gl.fwd(xd, flags).cpu().numpy()
    dx, dw = gl.bwd(dd, flags)
    dx = dx.cpu().numpy()
    torch.cuda.synchronize()
    assert capi.averis_last_device_error() == 0
    for e, (a, b) in enumerate(zip(offsets[:-1], offsets[1:])):
        if b == a:
            continue
        xe, de = x[a:b].astype(np.float64), d[a:b].astype(np.float64)
        mu_x = mu_d = None
        if split:
            mu_x = gl.states[e].mu.cpu().numpy().astype(np.float64)
            mu_d = capi.averis_quantize(dd[a:b].contiguous(), capi.AVERIS_MEAN_SPLIT, want_row=False,
                                        want_col=False)["mu"].cpu().numpy().astype(np.float64)
        f, bw = oav.linear_fwd_bwd(xe, ws[e].astype(np.float64), de, do_split=split, mu_x=mu_x, mu_d=mu_d)
        assert rel_fro(y[a:b], f.y) < TOL, e
        assert rel_fro(dx[a:b], bw.dx) < TOL, e
        assert rel_fro(dw[e].cpu().numpy(), bw.dw) < TOL, e


@pytest.mark.parametrize("linear", ["gate_up", "down"])
def test_grouped_moe_expert_ffn_full_shape(cuda_lib, linear):
    """The mixture-of-experts expert FFN at its benchmarked shape: hidden 2048, 64
    experts, top-8 of 16384 tokens with Zipf(1.1) popularity, expert FFN 768.  The
    smallest, the median-size and the largest expert are compared with the
    single-layer oracle over their own rows (means per expert, given the GPU's),
    Averis and vanilla; the mean of each is checked against the exact mean."""
    import torch
    from mean_residual_gemm_col_b300 import capi
    from tests.gpu_util import mu_close

    cfg = workloads.MOE
    counts = workloads.moe_routing(0, cfg["tokens"], cfg["experts"], cfg["top_k"], cfg["zipf"])
    offsets = np.concatenate([[0], np.cumsum(counts)])
    L = int(offsets[-1])
    m, n = (cfg["hidden"], 2 * cfg["ffn"]) if linear == "gate_up" else (cfg["ffn"], cfg["hidden"])
    x = workloads.torch_activation(31, L, m, spike=workloads.QWEN3_SPIKE, device="cuda")
    _, _, d = workloads.torch_linear_case(41, L, 16, n, device="cuda")
    order = np.argsort(counts, kind="stable")
    picks = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    ws = {e: workloads.torch_linear_case(100 + e, 16, m, n, device="cuda")[1] for e in range(cfg["experts"])}
    w_n, w_m = zip(*[capi.averis_quantize_weight(ws[e]) for e in range(cfg["experts"])])
    X, D = x.float().cpu().numpy(), d.float().cpu().numpy()
    for split in (True, False):
        gl = capi.GroupedLinear(offsets, m, n, list(w_m), list(w_n), "cuda")
        flags = capi.AVERIS_MEAN_SPLIT if split else 0
        y = gl.fwd(x, flags).cpu().numpy()
        dx, dw = gl.bwd(d, flags)
        dx = dx.cpu().numpy()
        torch.cuda.synchronize()
        assert capi.averis_last_device_error() == 0
        for e in picks:
            a, b = int(offsets[e]), int(offsets[e + 1])
            xe, de = X[a:b].astype(np.float64), D[a:b].astype(np.float64)
            mu_x = mu_d = None
            if split:
                mu_x = gl.states[e].mu.cpu().numpy().astype(np.float64)
                mu_d = capi.averis_quantize(d[a:b].contiguous(), capi.AVERIS_MEAN_SPLIT, want_row=False,
                                            want_col=False)["mu"].cpu().numpy().astype(np.float64)
                assert mu_close(mu_x, xe, oav.column_mean(xe))[0], e
                assert mu_close(mu_d, de, oav.column_mean(de))[0], e
            we = ws[e].float().cpu().numpy().astype(np.float64)
            f, bw = oav.linear_fwd_bwd(xe, we, de, do_split=split, mu_x=mu_x, mu_d=mu_d)
            tag = f"{linear} expert {e} ({b - a} rows) split={split}"
            assert rel_fro(y[a:b], f.y) < TOL, tag
            assert rel_fro(dx[a:b], bw.dx) < TOL, tag
            assert rel_fro(dw[e].cpu().numpy(), bw.dw) < TOL, tag
        del gl


def _same_bits(a, b, what):
    """Codes (the bytes that hold codes: row padding is not written), scales, tensor scale."""
    import torch

    nb = -(-a.cols // 16) * 8
    assert torch.equal(a.codes[:, :nb], b.codes[:, :nb]), what + " codes"
    assert torch.equal(a.scales, b.scales), what + " scales"
    assert torch.equal(a.tensor_scale, b.tensor_scale), what + " tensor scale"


@pytest.mark.parametrize("hadamard", [False, True])
def test_grouped_weight_quantize_matches_per_expert(cuda_lib, hadamard):
    """The experts' weights of a stacked [E, m, n] tensor in one launch chain:
    every expert's two layouts and tensor scales carry the same bits as its own
    averis_quantize_weight call, and those of one expert match the oracle."""
    import torch
    from mean_residual_gemm_col_b300 import capi
    from oracle import nvfp4 as onv
    from oracle.hadamard import rotate_fp32

    E, m, n = 5, 200, 144  # ragged against the 128-row tiles and 64-column strips
    g = workloads.rng(57)
    w = np.stack([workloads.weight(g, m, n) for _ in range(E)])
    wd = to_dev_bf16(w.reshape(E * m, n)).view(E, m, n)
    flags = capi.AVERIS_HADAMARD16 if hadamard else 0
    g_n, g_m = capi.averis_quantize_weight_grouped(wd, flags)
    torch.cuda.synchronize()
    assert capi.averis_last_device_error() == 0
    for e in range(E):
        s_n, s_m = capi.averis_quantize_weight(wd[e].contiguous(), flags)
        _same_bits(g_n[e], s_n, f"expert {e} w_n")
        _same_bits(g_m[e], s_m, f"expert {e} w_m")
    w2 = w[2].astype(np.float64)
    w2t = np.zeros((n, -(-m // 16) * 16))  # the column layout's partial last block is zero-padded
    w2t[:, :m] = w2.T
    for dev_t, ref_in, what in ((g_n[2], w2, "w_n"), (g_m[2], w2t, "w_m")):
        ref = onv.quantize(rotate_fp32(ref_in) if hadamard else ref_in)
        codes, scales, s_g = dev_t.canonical()
        assert s_g == np.float32(ref.s_g), what
        assert np.array_equal(codes, ref.codes) and np.array_equal(scales, ref.scales), what


def test_grouped_weight_quantize_moe_shape(cuda_lib):
    """The benchmarked expert weights (64 experts of the gate_up linear, 2048 x 1536):
    the grouped call gives every expert's bits of its own call."""
    import torch
    from mean_residual_gemm_col_b300 import capi

    cfg = workloads.MOE
    E, m, n = cfg["experts"], cfg["hidden"], 2 * cfg["ffn"]
    wd = torch.stack([workloads.torch_linear_case(100 + e, 16, m, n, device="cuda")[1] for e in range(E)])
    g_n, g_m = capi.averis_quantize_weight_grouped(wd)
    for e in (0, 31, E - 1):
        s_n, s_m = capi.averis_quantize_weight(wd[e].contiguous())
        _same_bits(g_n[e], s_n, f"expert {e} w_n")
        _same_bits(g_m[e], s_m, f"expert {e} w_m")
    torch.cuda.synchronize()
    assert capi.averis_last_device_error() == 0

"""Parity at full workload sizes, on sampled outputs.

The Qwen3-0.6B QKV linear (l = 8192, m = 1024, n = 4096) runs forward and
backward exactly as the benchmark launches it; the oracle then recomputes a
random sample of Y, dX and dW entries one by one.  NVFP4 quantization is
row-local once the tensor scale is fixed, so the oracle quantizes only the
rows a sampled entry needs, with the tensor scale taken from the whole
tensor's maximum (its own computation, from the GPU's binary32 mean, as in
"given the same mean").  The largest quantize-sweep shape (65536 x 8192) is
checked the same way: sampled rows of both layouts bit-exact.
"""

import numpy as np
import pytest

from oracle import averis as oav, nvfp4 as onv
from oracle.formats import f32
import workloads
from tests.gpu_util import mu_close, _mu_check

pytestmark = pytest.mark.gpu

E2M1_X_E4M3 = 6.0 * 448.0


def _s_g(amax):
    return float(f32(amax / E2M1_X_E4M3))


def _deq_rows(a, s_g):
    """Dequantized NVFP4 rows of a (float64, binary32 values), blocked along the last axis."""
    return onv.quantize(a, s_g=s_g).dequantize()


def _to_np(t):
    import torch

    return t.float().cpu().numpy().astype(np.float64) if t.dtype == torch.bfloat16 else t.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("out_bf16", [False, True])
def test_qwen_qkv_layer_sampled_outputs(cuda_lib, out_bf16):
    import torch
    from mean_residual_gemm_col_b300 import capi

    l, m, n = workloads.QWEN3_L, 1024, 4096
    x, w, d = workloads.torch_linear_case(7, l, m, n, spike=workloads.QWEN3_SPIKE, device="cuda")
    w_n, w_m = capi.averis_quantize_weight(w)
    y, st = capi.averis_linear_fwd(x, w_m, out_bf16=out_bf16)
    dx, dw = capi.averis_linear_bwd(d, st, w_n, out_bf16=out_bf16)
    mu_d_gpu = capi.averis_quantize(d, capi.AVERIS_MEAN_SPLIT, want_row=False, want_col=False)["mu"]
    torch.cuda.synchronize()
    assert capi.averis_last_device_error() == 0

    X, W, D = _to_np(x), _to_np(w), _to_np(d)
    mu_x, mu_d = _to_np(st.mu), _to_np(mu_d_gpu)
    assert mu_close(mu_x, X, oav.column_mean(X))[0]
    assert mu_close(mu_d, D, oav.column_mean(D))[0]
    XR, DR = oav.residual_fp32(X, mu_x), oav.residual_fp32(D, mu_d)
    sx, sd, sw = _s_g(np.abs(XR).max()), _s_g(np.abs(DR).max()), _s_g(np.abs(W).max())
    # the means as their own one-row tensors
    mux_hat = onv.quantize(mu_x[None, :]).dequantize()[0]
    mud_hat = onv.quantize(mu_d[None, :]).dequantize()[0]

    rng = np.random.default_rng(0)
    Y, DX, DW = _to_np(y), _to_np(dx), _to_np(dw)
    wm_all = _deq_rows(W.T, sw)                 # W blocked along m: [n, m] (small)
    wn_all = _deq_rows(W, sw)                   # W blocked along n: [m, n]
    r_x = mux_hat @ wm_all.T
    r_d = mud_hat @ wn_all.T
    tol_elem = (2.0 ** -8) if out_bf16 else 1e-5

    def check(got, want, what):
        err = np.abs(got - want)
        scale = np.abs(want) + 1e-3 * np.abs(want).max()
        bad = np.argwhere(err > tol_elem * scale)
        assert bad.size == 0, f"{what}: {len(bad)} sampled entries off, worst rel {float((err / scale).max()):.3g}"
        if not out_bf16:
            assert np.linalg.norm(got - want) <= 1e-4 * np.linalg.norm(want), what

    # Y[i, j]
    ii, jj = rng.integers(0, l, 48), rng.integers(0, n, 48)
    xq = _deq_rows(XR[ii], sx)
    want = np.einsum("sk,sk->s", xq, wm_all[jj]) + r_x[jj]
    check(Y[ii, jj], want, "Y")
    # dX[i, k]
    ii, kk = rng.integers(0, l, 48), rng.integers(0, m, 48)
    dq = _deq_rows(DR[ii], sd)
    want = np.einsum("sk,sk->s", dq, wn_all[kk]) + r_d[kk]
    check(DX[ii, kk], want, "dX")
    # dW[k, j]: X_R^T blocked along l, D_R^T blocked along l
    kk, jj = rng.integers(0, m, 24), rng.integers(0, n, 24)
    # both layouts of a residual share its one maximum, hence its tensor scale
    xc = _deq_rows(np.ascontiguousarray(XR[:, kk].T), sx)
    dc = _deq_rows(np.ascontiguousarray(DR[:, jj].T), sd)
    want = np.einsum("sl,sl->s", xc, dc) + l * mux_hat[kk] * mud_hat[jj]
    got = DW[kk, jj]
    err = np.abs(got - want)
    scale = np.abs(want) + 1e-3 * np.abs(want).max()
    assert np.all(err <= 1e-5 * scale), f"dW sampled entries off, worst rel {float((err / scale).max()):.3g}"


def test_quantize_sweep_largest_shape_sampled_rows(cuda_lib):
    import torch
    from mean_residual_gemm_col_b300 import capi, layout

    R, C = 65536, 8192
    x = workloads.torch_activation(R * 10 + C, R, C, spike=50.0, device="cuda")
    out = capi.averis_quantize(x, capi.AVERIS_MEAN_SPLIT)
    torch.cuda.synchronize()
    mu = out["mu"].cpu().numpy().astype(np.float64)
    # exact column means and the residual maximum, in float64 over row chunks
    s = np.zeros(C)
    amax = 0.0
    absmean = np.zeros(C)
    for r0 in range(0, R, 8192):
        xb = x[r0:r0 + 8192].float().cpu().numpy().astype(np.float64)
        s += xb.sum(axis=0)
        absmean += np.abs(xb).sum(axis=0)
        amax = max(amax, float(np.abs(f32(xb - mu[None, :])).max()))
    ok, worst = _mu_check(mu, s / R, absmean / R)
    assert ok, f"mean off by {worst:.3g} (relative)"
    s_row = _s_g(amax)
    assert float(out["row"].tensor_scale.item()) == np.float32(s_row)
    assert float(out["col"].tensor_scale.item()) == np.float32(s_row)
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(R, 16, replace=False))
    xr = x[torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64)
    ref = onv.quantize(oav.residual_fp32(xr, mu), s_g=s_row)
    codes = out["row"].codes[torch.from_numpy(rows).cuda()].cpu().numpy()
    got = layout.unpack_codes(codes, len(rows), C)
    assert np.array_equal(got, ref.codes)
    sc_all = out["row"].scales.cpu().numpy()
    off = layout.scale_offsets(R, C, rows)
    assert np.array_equal(sc_all[off].astype(np.int64), ref.scales)
    # column layout: sampled columns of X become rows of the transposed tensor
    cols = np.sort(rng.choice(C, 8, replace=False))
    xc = x[:, torch.from_numpy(cols).cuda()].float().cpu().numpy().astype(np.float64).T
    refc = onv.quantize(oav.residual_fp32(xc.T, mu[cols]).T, s_g=s_row)
    codes_c = out["col"].codes[torch.from_numpy(cols).cuda()].cpu().numpy()
    assert np.array_equal(layout.unpack_codes(codes_c, len(cols), R), refc.codes)
    offc = layout.scale_offsets(C, R, cols)
    assert np.array_equal(out["col"].scales.cpu().numpy()[offc].astype(np.int64), refc.scales)

"""Full-size parity of every benchmarked configuration, on sampled outputs.

Each layer runs through the C ABI exactly as the benchmark launches it (same
seeded device inputs, same flags), once with binary32 outputs (the parity
mode: relative Frobenius error over the samples <= 1e-4) and once with the
benchmark's bf16 Y / dX (each sample within bf16 rounding).  The oracle
recomputes a random sample of Y, dX and dW entries from only the rows a
sample needs (``tests/sampled_ref.py``, itself checked against the whole
oracle), given the GPU's binary32 means, which are checked against the exact
float64 means.  Sampled rows and columns of X's two quantized layouts must
equal the oracle's codes and block scales bit for bit.

Shapes ("均值偏置的诅咒与祝福" summary, experiments on Qwen3 models):
* the four Qwen3-0.6B linears at l = 8192, vanilla NVFP4 and Averis, and the
  QKV linear with the 16x16 rotation;
* the same linears at l = 16384, the token count of the 28-layer stack, in
  its three modes (vanilla, Averis, Averis + rotation): the weight gradient's
  contraction runs over 16384 tokens here.
"""

import numpy as np
import pytest

from oracle.formats import f32
import workloads
from mean_residual_gemm_col_b300 import layout
from tests.gpu_util import mu_close_chunked
from tests.sampled_ref import SampledLinear

pytestmark = pytest.mark.gpu

LINEARS = {name: (m, n) for name, m, n in workloads.QWEN3_06B_LINEARS}
FRO_TOL = 1e-4
ELEM_TOL_F32 = 1e-5
ELEM_TOL_BF16 = 2.0 ** -8


def _host(t):
    import torch

    return t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()


def _run_layer(x, w, d, mode, out_bf16):
    from mean_residual_gemm_col_b300 import capi

    had = capi.AVERIS_HADAMARD16 if mode.endswith("h16") else 0
    w_n, w_m = capi.averis_quantize_weight(w, had)
    if mode.startswith("averis"):
        y, st = capi.averis_linear_fwd(x, w_m, capi.AVERIS_MEAN_SPLIT | had, out_bf16=out_bf16)
        dx, dw = capi.averis_linear_bwd(d, st, w_n, capi.AVERIS_MEAN_SPLIT | had, out_bf16=out_bf16)
    else:
        y, st = capi.nvfp4_linear_fwd(x, w_m, had, out_bf16=out_bf16)
        dx, dw = capi.nvfp4_linear_bwd(d, st, w_n, had, out_bf16=out_bf16)
    return y, dx, dw, st


def _check(got, want, bf16, what):
    got = np.asarray(got, np.float64)
    err = np.abs(got - want)
    if bf16:
        bound = ELEM_TOL_BF16 * (np.abs(want) + 1e-3 * np.abs(want).max())
    else:
        bound = ELEM_TOL_F32 * (np.abs(want) + 1e-3 * np.abs(want).max())
    bad = int((err > bound).sum())
    assert bad == 0, f"{what}: {bad} of {len(want)} samples off, worst {float((err / (bound + 1e-300)).max()):.3g} x bound"
    if not bf16:
        fro = float(np.linalg.norm(got - want) / np.linalg.norm(want))
        assert fro <= FRO_TOL, f"{what}: relative Frobenius error {fro:.3g} over the samples"


def _run_config(l, m, n, mode, seed):
    import torch
    from mean_residual_gemm_col_b300 import capi

    x, w, d = workloads.torch_linear_case(seed, l, m, n, spike=workloads.QWEN3_SPIKE, device="cuda")
    split = mode.startswith("averis")
    had = mode.endswith("h16")
    outs = {}
    for out_bf16 in (False, True):
        y, dx, dw, st = _run_layer(x, w, d, mode, out_bf16)
        torch.cuda.synchronize()
        assert capi.averis_last_device_error() == 0
        outs[out_bf16] = (_host(y), _host(dx), _host(dw))
        if not out_bf16:
            state = st
    mu_d = None
    if split:
        flags = capi.AVERIS_MEAN_SPLIT | (capi.AVERIS_HADAMARD16 if had else 0)
        mu_d = capi.averis_quantize(d, flags, want_row=False, want_col=False)["mu"].cpu().numpy().astype(np.float64)
    X, W, D = _host(x), _host(w), _host(d)
    mu_x = state.mu.cpu().numpy().astype(np.float64) if split else None
    if split:
        ok, worst = mu_close_chunked(mu_x, X)
        assert ok, f"mu_X off by {worst:.3g} relative"
        ok, worst = mu_close_chunked(mu_d, D)
        assert ok, f"mu_D off by {worst:.3g} relative"
        assert np.array_equal(f32(mu_x), mu_x) and np.array_equal(f32(mu_d), mu_d)
    ref = SampledLinear(X, W, D, mu_x=mu_x, mu_d=mu_d, hadamard=had)

    rng = np.random.default_rng(seed)
    # X's quantized layouts, sampled rows / columns, bit for bit
    rows = np.sort(rng.choice(l, 8, replace=False))
    q = ref.x_rows_q(rows)
    codes = layout.unpack_codes(state.x_row.codes.cpu().numpy()[rows], len(rows), m)
    assert np.array_equal(codes, q.codes), "X_R row-layout codes"
    sc = state.x_row.scales.cpu().numpy()[layout.scale_offsets(l, m, rows)]
    assert np.array_equal(sc.astype(np.int64), q.scales), "X_R row-layout block scales"
    assert float(state.x_row.tensor_scale.item()) == q.s_g, "X_R row-layout tensor scale"
    cols = np.sort(rng.choice(m, 4, replace=False))
    qc = ref.x_cols_q(cols)
    lc = layout.cdiv(l, 16) * 16
    codes = layout.unpack_codes(state.x_col.codes.cpu().numpy()[cols], len(cols), l)
    assert np.array_equal(codes, qc.codes[:, :lc]), "X_R column-layout codes"
    sc = state.x_col.scales.cpu().numpy()[layout.scale_offsets(m, l, cols)]
    assert np.array_equal(sc.astype(np.int64), qc.scales), "X_R column-layout block scales"
    assert float(state.x_col.tensor_scale.item()) == qc.s_g, "X_R column-layout tensor scale"

    ii, jj = rng.integers(0, l, 48), rng.integers(0, n, 48)
    want_y = ref.y(ii, jj)
    ik, kk = rng.integers(0, l, 48), rng.integers(0, m, 48)
    want_dx = ref.dx(ik, kk)
    wk, wj = rng.integers(0, m, 24), rng.integers(0, n, 24)
    want_dw = ref.dw(wk, wj)
    for bf16, (Y, DX, DW) in outs.items():
        tag = f"{mode} l={l} m={m} n={n} {'bf16' if bf16 else 'fp32'}"
        _check(Y[ii, jj], want_y, bf16, "Y " + tag)
        _check(DX[ik, kk], want_dx, bf16, "dX " + tag)
        _check(DW[wk, wj], want_dw, False, "dW " + tag)     # dW is always binary32


@pytest.mark.parametrize("mode", ["averis", "nvfp4"])
@pytest.mark.parametrize("linear", ["qkv", "o_proj", "gate_up", "down"])
def test_qwen3_linears_l8192(cuda_lib, linear, mode):
    m, n = LINEARS[linear]
    _run_config(workloads.QWEN3_L, m, n, mode, seed=11 + list(LINEARS).index(linear))


def test_qwen3_qkv_l8192_hadamard(cuda_lib):
    m, n = LINEARS["qkv"]
    _run_config(workloads.QWEN3_L, m, n, "averis_h16", seed=29)


@pytest.mark.parametrize("mode", ["nvfp4", "averis", "averis_h16"])
@pytest.mark.parametrize("linear", ["qkv", "o_proj", "gate_up", "down"])
def test_stack_linears_l16384(cuda_lib, linear, mode):
    m, n = LINEARS[linear]
    _run_config(workloads.STACK_L, m, n, mode, seed=5000 + list(LINEARS).index(linear))

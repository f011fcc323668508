"""GPU parity of the whole Averis / vanilla NVFP4 linear layer (fwd + bwd) via the C ABI.

The oracle is given the GPU's binary32 means (checked separately against
its own within 1e-6), so both sides quantize identical operands; Y, dX and
dW must then agree within 1e-4 relative Frobenius error (binary32 outputs).
"""

import numpy as np
import pytest

from oracle import averis as oav
import workloads
from tests.gpu_util import to_dev_bf16, rel_fro, mu_close

pytestmark = pytest.mark.gpu

TOL = 1e-4

SHAPES = [(256, 256, 256), (200, 272, 144), (1, 16, 32), (37, 48, 80), (300, 512, 384), (1024, 1024, 512)]


def _run(l, m, n, split, hadamard, seed, spike=50.0):
    from mean_residual_gemm_col_b300 import capi

    case = workloads.linear_case(seed, l, m, n, spike=spike)
    x, w, d = to_dev_bf16(case.x), to_dev_bf16(case.w), to_dev_bf16(case.d)
    hflag = capi.AVERIS_HADAMARD16 if hadamard else 0
    w_n, w_m = capi.averis_quantize_weight(w, hflag)
    if split:
        y, st = capi.averis_linear_fwd(x, w_m, capi.AVERIS_MEAN_SPLIT | hflag)
        dx, dw = capi.averis_linear_bwd(d, st, w_n, capi.AVERIS_MEAN_SPLIT | hflag)
        mu_d = capi.averis_quantize(d, capi.AVERIS_MEAN_SPLIT | hflag, want_row=False, want_col=False)["mu"]
        mu_x = st.mu.cpu().numpy().astype(np.float64)
        mu_d = mu_d.cpu().numpy().astype(np.float64)
    else:
        y, st = capi.nvfp4_linear_fwd(x, w_m, hflag)
        dx, dw = capi.nvfp4_linear_bwd(d, st, w_n, hflag)
        mu_x = mu_d = None
    assert capi.averis_last_device_error() == 0
    return case, y.cpu().numpy(), dx.cpu().numpy(), dw.cpu().numpy(), mu_x, mu_d


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("split", [True, False])
def test_linear_fwd_bwd_matches_oracle(cuda_lib, shape, split):
    l, m, n = shape
    case, y, dx, dw, mu_x, mu_d = _run(l, m, n, split, False, seed=l + m + n)
    x64, w64, d64 = (case.x.astype(np.float64), case.w.astype(np.float64), case.d.astype(np.float64))
    if split:
        assert mu_close(mu_x, x64, oav.column_mean(x64))[0]
        assert mu_close(mu_d, d64, oav.column_mean(d64))[0]
    f, b = oav.linear_fwd_bwd(x64, w64, d64, do_split=split, mu_x=mu_x, mu_d=mu_d)
    assert rel_fro(y, f.y) < TOL
    assert rel_fro(dx, b.dx) < TOL
    assert rel_fro(dw, b.dw) < TOL


@pytest.mark.parametrize("split", [True, False])
def test_long_token_axis_few_weight_gradient_tiles(cuda_lib, split):
    """A long token axis (K of the weight gradient) and only a few dW tiles;
    the result is also bit-for-bit reproducible."""
    l, m, n = 8192, 256, 512
    case, y, dx, dw, mu_x, mu_d = _run(l, m, n, split, False, seed=77)
    x64, w64, d64 = (case.x.astype(np.float64), case.w.astype(np.float64), case.d.astype(np.float64))
    f, b = oav.linear_fwd_bwd(x64, w64, d64, do_split=split, mu_x=mu_x, mu_d=mu_d)
    assert rel_fro(dw, b.dw) < TOL
    assert rel_fro(y, f.y) < TOL
    # deterministic: a second backward gives the same bits
    _, _, _, dw2, _, _ = _run(l, m, n, split, False, seed=77)
    assert np.array_equal(dw, dw2)


@pytest.mark.parametrize("shape", [(256, 256, 256), (200, 272, 144)])
@pytest.mark.parametrize("split", [True, False])
def test_linear_hadamard_matches_oracle(cuda_lib, shape, split):
    l, m, n = shape
    case, y, dx, dw, mu_x, mu_d = _run(l, m, n, split, True, seed=3 * l + m)
    x64, w64, d64 = (case.x.astype(np.float64), case.w.astype(np.float64), case.d.astype(np.float64))
    f, b = oav.linear_fwd_bwd(x64, w64, d64, do_split=split, hadamard=True, mu_x=mu_x, mu_d=mu_d)
    assert rel_fro(y, f.y) < TOL
    assert rel_fro(dx, b.dx) < TOL
    assert rel_fro(dw, b.dw) < TOL


def test_bf16_outputs(cuda_lib):
    import torch
    from mean_residual_gemm_col_b300 import capi

    l, m, n = 512, 256, 384
    case = workloads.linear_case(11, l, m, n)
    x, w, d = to_dev_bf16(case.x), to_dev_bf16(case.w), to_dev_bf16(case.d)
    w_n, w_m = capi.averis_quantize_weight(w)
    y32, st = capi.averis_linear_fwd(x, w_m)
    y16, _ = capi.averis_linear_fwd(x, w_m, out_bf16=True)
    assert y16.dtype == torch.bfloat16
    assert torch.equal(y16, y32.to(torch.bfloat16))
    dx32, dw32 = capi.averis_linear_bwd(d, st, w_n)
    dx16, dw16 = capi.averis_linear_bwd(d, st, w_n, out_bf16=True)
    assert torch.equal(dx16, dx32.to(torch.bfloat16))
    assert torch.equal(dw16, dw32)

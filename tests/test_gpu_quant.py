"""GPU parity of the fused mean-split quantize pass against the oracle.

Bar: mu within 1e-6 (relative to max(|mu|, mean |x|)); given the GPU's mu,
every E2M1 code, E4M3 block scale and tensor scale bit-exact, in both layouts.
"""

import numpy as np
import pytest

from oracle import averis as oav, nvfp4 as onv
from oracle.hadamard import rotate_fp32, rotate_exact
import workloads
from tests.gpu_util import to_dev_bf16, mu_close

pytestmark = pytest.mark.gpu

SHAPES = [(256, 256), (200, 272), (1, 16), (37, 48), (129, 144), (1000, 512), (2048, 1024)]


def _check_nvfp4(dev_t, ref: onv.NVFP4, what):
    codes, scales, s_g = dev_t.canonical()
    assert s_g == np.float32(ref.s_g), f"{what}: tensor scale {s_g} vs {ref.s_g}"
    assert codes.shape == ref.codes.shape, what
    bad = np.argwhere(codes != ref.codes)
    assert bad.size == 0, f"{what}: {len(bad)} code mismatches, first {bad[:4].tolist()}"
    bad = np.argwhere(scales != ref.scales)
    assert bad.size == 0, f"{what}: {len(bad)} scale mismatches, first {bad[:4].tolist()}"


def _pad16_cols(a):
    c16 = -(-a.shape[1] // 16) * 16
    out = np.zeros((a.shape[0], c16))
    out[:, : a.shape[1]] = a
    return out


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("hadamard", [False, True])
def test_split_quantize_bit_exact(cuda_lib, shape, hadamard):
    from mean_residual_gemm_col_b300 import capi

    R, C = shape
    x = workloads.activation(workloads.rng(R * 7 + C), R, C, spike=50.0)
    flags = capi.AVERIS_MEAN_SPLIT | (capi.AVERIS_HADAMARD16 if hadamard else 0)
    out = capi.averis_quantize(to_dev_bf16(x), flags)
    mu_gpu = out["mu"].cpu().numpy().astype(np.float64)
    x64 = x.astype(np.float64)
    ok, worst = mu_close(mu_gpu, x64, oav.column_mean(x64))
    assert ok, f"mu off by {worst:.3g} (relative)"
    r = oav.residual_fp32(x64, mu_gpu)
    row_in = rotate_fp32(r) if hadamard else r
    col_in = rotate_fp32(_pad16_cols(r.T)) if hadamard else r.T
    _check_nvfp4(out["row"], onv.quantize(row_in), "row layout")
    _check_nvfp4(out["col"], onv.quantize(col_in), "column layout")
    mu_in = rotate_fp32(mu_gpu[None, :]) if hadamard else mu_gpu[None, :]
    ref_mu = onv.quantize(mu_in)
    _check_nvfp4(out["mu_q"], ref_mu, "mean")
    mu_hat = ref_mu.dequantize()
    if hadamard:
        mu_hat = rotate_exact(mu_hat)
    got = out["mu_hat"].cpu().numpy().astype(np.float64)
    assert np.allclose(got, mu_hat[0], rtol=1e-6, atol=1e-6 * np.abs(mu_hat).max())


@pytest.mark.parametrize("shape", [(256, 256), (200, 272), (1024, 4096)])
def test_vanilla_quantize_bit_exact(cuda_lib, shape):
    from mean_residual_gemm_col_b300 import capi

    R, C = shape
    x = workloads.activation(workloads.rng(R + C), R, C, spike=30.0)
    out = capi.averis_quantize(to_dev_bf16(x), 0)
    x64 = x.astype(np.float64)
    _check_nvfp4(out["row"], onv.quantize(x64), "row layout")
    _check_nvfp4(out["col"], onv.quantize(x64.T), "column layout")


@pytest.mark.parametrize("hadamard", [False, True])
def test_weight_quantize_bit_exact(cuda_lib, hadamard):
    from mean_residual_gemm_col_b300 import capi

    m, n = 272, 400
    w = workloads.weight(workloads.rng(5), m, n)
    w_n, w_m = capi.averis_quantize_weight(to_dev_bf16(w), capi.AVERIS_HADAMARD16 if hadamard else 0)
    w64 = w.astype(np.float64)
    rot = (lambda a: rotate_fp32(a)) if hadamard else (lambda a: a)
    _check_nvfp4(w_n, onv.quantize(rot(w64)), "W along n")
    _check_nvfp4(w_m, onv.quantize(rot(w64.T)), "W along m")


def test_constant_columns_give_zero_residual(cuda_lib):
    from mean_residual_gemm_col_b300 import capi

    mu = workloads.bf16_round(np.linspace(-5, 7, 64).astype(np.float32))
    x = np.tile(mu, (48, 1))
    out = capi.averis_quantize(to_dev_bf16(x), capi.AVERIS_MEAN_SPLIT)
    assert np.array_equal(out["mu"].cpu().numpy(), mu)
    codes, scales, s_g = out["row"].canonical()
    assert s_g == 0.0 and not codes.any() and not scales.any()


def test_quantize_is_deterministic(cuda_lib):
    from mean_residual_gemm_col_b300 import capi

    x = to_dev_bf16(workloads.activation(workloads.rng(9), 4096, 1024))
    a = capi.averis_quantize(x, capi.AVERIS_MEAN_SPLIT)
    b = capi.averis_quantize(x, capi.AVERIS_MEAN_SPLIT)
    assert (a["mu"] == b["mu"]).all()
    assert (a["row"].codes == b["row"].codes).all() and (a["col"].scales == b["col"].scales).all()


def test_split_quantize_wider_than_one_strip_per_cta(cuda_lib):
    """More 64-column strips (1040) than strip groups of the stats pass (1024):
    some CTAs take two strips in turn, and the quantize pass runs 520 column
    tiles; every code and scale still bit-exact."""
    from mean_residual_gemm_col_b300 import capi

    R, C = 64, 66560
    x = workloads.activation(workloads.rng(R * 7 + C), R, C, spike=50.0)
    out = capi.averis_quantize(to_dev_bf16(x), capi.AVERIS_MEAN_SPLIT)
    mu_gpu = out["mu"].cpu().numpy().astype(np.float64)
    x64 = x.astype(np.float64)
    ok, worst = mu_close(mu_gpu, x64, oav.column_mean(x64))
    assert ok, f"mu off by {worst:.3g} (relative)"
    r = oav.residual_fp32(x64, mu_gpu)
    _check_nvfp4(out["row"], onv.quantize(r), "row layout")
    _check_nvfp4(out["col"], onv.quantize(r.T), "column layout")
    _check_nvfp4(out["mu_q"], onv.quantize(mu_gpu[None, :]), "mean")

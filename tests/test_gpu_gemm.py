"""GPU parity of the tcgen05 block-scaled NVFP4 GEMM and the rank-one GEMV.

The operands are quantized by the ORACLE on the host and copied to the
device, so this isolates the GEMM: its output must match the oracle's
float64 product of the same dequantized operands within 1e-4 relative
Frobenius error (binary32 output).
"""

import numpy as np
import pytest

from oracle import nvfp4 as onv
import workloads
from tests.gpu_util import rel_fro

pytestmark = pytest.mark.gpu

TOL = 1e-4


def _operand(rng, rows, cols, scale=1.0, spikes=True):
    a = (rng.standard_normal((rows, cols)) * scale).astype(np.float32)
    if spikes:
        a[rng.random(a.shape) < 1e-3] *= 32
    return onv.quantize(a.astype(np.float64))


def _dev(q: onv.NVFP4, rows, cols):
    from mean_residual_gemm_col_b300.capi import NVFP4Tensor

    return NVFP4Tensor.from_canonical(q.codes, q.scales, q.s_g, rows, cols, "cuda")


@pytest.mark.parametrize("mnk", [(128, 128, 256), (256, 384, 1024), (300, 200, 272), (8, 16, 16),
                                 (129, 130 + 14, 64), (512, 256, 4096), (1024, 1024, 8192)])
def test_gemm_plain(cuda_lib, mnk):
    from mean_residual_gemm_col_b300 import capi

    M, N, K = mnk
    rng = np.random.default_rng(M * 31 + N * 7 + K)
    a = _operand(rng, M, K)
    b = _operand(rng, N, K, 0.05)
    out = capi.averis_gemm(_dev(a, M, K), _dev(b, N, K)).cpu().numpy()
    want = a.dequantize() @ b.dequantize().T
    assert rel_fro(out, want) < TOL


def test_gemm_single_nonzero_block_locates_layout(cuda_lib):
    """One non-zero 16-block per operand: checks row, column, K-block and scale placement."""
    from mean_residual_gemm_col_b300 import capi

    M, N, K = 256, 256, 512
    for (i, j, kb) in [(0, 0, 0), (37, 5, 3), (130, 200, 17), (255, 129, 31), (64, 64, 4)]:
        a = np.zeros((M, K))
        b = np.zeros((N, K))
        a[i, 16 * kb: 16 * kb + 16] = np.arange(1, 17) * 0.25
        b[j, 16 * kb: 16 * kb + 16] = np.linspace(-3, 3, 16).astype(np.float32)
        qa, qb = onv.quantize(a), onv.quantize(b)
        out = capi.averis_gemm(_dev(qa, M, K), _dev(qb, N, K)).cpu().numpy()
        want = qa.dequantize() @ qb.dequantize().T
        assert np.count_nonzero(want) == 1
        assert rel_fro(out, want) < TOL, (i, j, kb, np.argwhere(out != 0)[:4])


def test_gemm_epilogue_terms(cuda_lib):
    import torch
    from mean_residual_gemm_col_b300 import capi

    M, N, K = 384, 272, 512
    rng = np.random.default_rng(3)
    a = _operand(rng, M, K)
    b = _operand(rng, N, K, 0.02)
    col_add = rng.standard_normal(N).astype(np.float32)
    u = rng.standard_normal(M).astype(np.float32)
    v = rng.standard_normal(N).astype(np.float32)
    base = a.dequantize() @ b.dequantize().T
    dev = lambda z: torch.from_numpy(z).cuda()
    out = capi.averis_gemm(_dev(a, M, K), _dev(b, N, K), col_add=dev(col_add)).cpu().numpy()
    assert rel_fro(out, base + col_add[None, :]) < TOL
    out = capi.averis_gemm(_dev(a, M, K), _dev(b, N, K), row_vec=dev(u), col_vec=dev(v), outer=100.0).cpu().numpy()
    assert rel_fro(out, base + 100.0 * np.outer(u, v)) < TOL


def test_gemm_bf16_output(cuda_lib):
    from mean_residual_gemm_col_b300 import capi

    M, N, K = 256, 384, 1024
    rng = np.random.default_rng(4)
    a = _operand(rng, M, K)
    b = _operand(rng, N, K)
    out = capi.averis_gemm(_dev(a, M, K), _dev(b, N, K), out_bf16=True).float().cpu().numpy()
    want = a.dequantize() @ b.dequantize().T
    # bf16 rounding of the output: at most 2^-9 relative per element
    assert np.all(np.abs(out - want) <= 2.0 ** -8 * np.abs(want) + 1e-6 * np.abs(want).max())


def test_rank1_gemv(cuda_lib):
    from mean_residual_gemm_col_b300 import capi

    rng = np.random.default_rng(5)
    N, K = 300, 1040
    mu = onv.quantize(rng.standard_normal((1, K)).astype(np.float32).astype(np.float64) * 8)
    w = _operand(rng, N, K, 0.02)
    out = capi.averis_rank1(_dev(mu, 1, K), _dev(w, N, K)).cpu().numpy()
    want = (mu.dequantize() @ w.dequantize().T)[0]
    assert rel_fro(out, want) < 1e-6


def test_no_device_error_after_gemm(cuda_lib):
    from mean_residual_gemm_col_b300 import capi

    assert capi.averis_last_device_error() == 0

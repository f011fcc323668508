"""The bounds-checked debug build of the library on tiny shapes, against the oracle.

No memory checker runs on the GPU machines these tests use.  The debug build
(libaveris_debug.so, compiled with -DAVERIS_DEBUG) checks every global address
its kernels compute against the extent of the buffer the address belongs to,
and the inner coordinate of every TMA copy against the 16-byte rule; a check
that fails skips the access and leaves 100 + its site in the device error
word.  Every path of the library runs here through the debug build on tiny
shapes (l, m, n in {16, 32, 48}: ragged against the 128-row tiles, the
64-column strips and the 256-wide GEMM tiles), so every edge of every kernel
is checked: the error word must stay clear and the results must match the
oracle to the bars of the release tests (codes and scales bit-exact given
the GPU's mean, GEMM outputs within 1e-4 relative Frobenius error).
"""

import ctypes
import itertools
import os

import numpy as np
import pytest

from oracle import averis as oav, nvfp4 as onv
from oracle.hadamard import rotate_fp32
import workloads
from tests.gpu_util import to_dev_bf16, rel_fro, mu_close

pytestmark = pytest.mark.gpu

TOL = 1e-4
SIZES = (16, 32, 48)


@pytest.fixture(scope="module")
def debug_lib():
    """The debug build, bound in place of the release library for this module."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mean_residual_gemm_col_b300 import build, capi

    if not os.path.exists(build.DEBUG_LIB):
        build.build(debug=True)
    release = capi.load()
    lib = capi._declare(ctypes.CDLL(build.DEBUG_LIB))
    capi._lib = lib
    try:
        yield lib
    finally:
        capi._lib = release


def _clean():
    from mean_residual_gemm_col_b300 import capi

    code = capi.averis_last_device_error()
    assert code == 0, f"device error word {code} (100 + site: a bounds check caught an access)"


def _check_nvfp4(dev_t, ref: onv.NVFP4, what):
    codes, scales, s_g = dev_t.canonical()
    assert s_g == np.float32(ref.s_g), what
    assert np.array_equal(codes, ref.codes), what
    assert np.array_equal(scales, ref.scales), what


def test_debug_build_checks_itself(debug_lib):
    assert debug_lib.averis_debug_checks() == 1


def test_release_build_has_no_checks(debug_lib):
    from mean_residual_gemm_col_b300 import capi

    release = capi._declare(ctypes.CDLL(capi.LIB_PATH))
    assert release.averis_debug_checks() == 0


@pytest.mark.parametrize("R,C", list(itertools.product(SIZES, SIZES)))
@pytest.mark.parametrize("mode", ["split", "split_h16", "vanilla"])
def test_quantize_tiny(debug_lib, R, C, mode):
    from mean_residual_gemm_col_b300 import capi

    x = workloads.activation(workloads.rng(R * 5 + C), R, C, spike=50.0)
    had = mode == "split_h16"
    flags = (0 if mode == "vanilla" else capi.AVERIS_MEAN_SPLIT) | (capi.AVERIS_HADAMARD16 if had else 0)
    out = capi.averis_quantize(to_dev_bf16(x), flags)
    _clean()
    x64 = x.astype(np.float64)
    if mode == "vanilla":
        r = x64
    else:
        mu_gpu = out["mu"].cpu().numpy().astype(np.float64)
        assert mu_close(mu_gpu, x64, oav.column_mean(x64))[0]
        r = oav.residual_fp32(x64, mu_gpu)
    pad = np.zeros((C, -(-R // 16) * 16))
    pad[:, :R] = r.T
    _check_nvfp4(out["row"], onv.quantize(rotate_fp32(r) if had else r), "row layout")
    _check_nvfp4(out["col"], onv.quantize(rotate_fp32(pad) if had else r.T), "column layout")


@pytest.mark.parametrize("l,m,n", list(itertools.product(SIZES, SIZES, SIZES)))
@pytest.mark.parametrize("split", [True, False])
def test_linear_tiny(debug_lib, l, m, n, split):
    from mean_residual_gemm_col_b300 import capi

    case = workloads.linear_case(l * 100 + m * 10 + n, l, m, n, spike=50.0)
    x, w, d = to_dev_bf16(case.x), to_dev_bf16(case.w), to_dev_bf16(case.d)
    w_n, w_m = capi.averis_quantize_weight(w)
    mu_x = mu_d = None
    if split:
        y, st = capi.averis_linear_fwd(x, w_m)
        dx, dw = capi.averis_linear_bwd(d, st, w_n)
        mu_x = st.mu.cpu().numpy().astype(np.float64)
        mu_d = capi.averis_quantize(d, capi.AVERIS_MEAN_SPLIT, want_row=False, want_col=False)["mu"]
        mu_d = mu_d.cpu().numpy().astype(np.float64)
    else:
        y, st = capi.nvfp4_linear_fwd(x, w_m)
        dx, dw = capi.nvfp4_linear_bwd(d, st, w_n)
    _clean()
    f, b = oav.linear_fwd_bwd(case.x.astype(np.float64), case.w.astype(np.float64), case.d.astype(np.float64),
                              do_split=split, mu_x=mu_x, mu_d=mu_d)
    assert rel_fro(y.cpu().numpy(), f.y) < TOL
    assert rel_fro(dx.cpu().numpy(), b.dx) < TOL
    assert rel_fro(dw.cpu().numpy(), b.dw) < TOL


@pytest.mark.parametrize("l,m,n", [(16, 16, 16), (48, 32, 48), (32, 48, 16)])
def test_linear_hadamard_tiny(debug_lib, l, m, n):
    from mean_residual_gemm_col_b300 import capi

    case = workloads.linear_case(7 * l + m + n, l, m, n, spike=50.0)
    x, w, d = to_dev_bf16(case.x), to_dev_bf16(case.w), to_dev_bf16(case.d)
    flags = capi.AVERIS_MEAN_SPLIT | capi.AVERIS_HADAMARD16
    w_n, w_m = capi.averis_quantize_weight(w, capi.AVERIS_HADAMARD16)
    y, st = capi.averis_linear_fwd(x, w_m, flags)
    dx, dw = capi.averis_linear_bwd(d, st, w_n, flags)
    mu_d = capi.averis_quantize(d, flags, want_row=False, want_col=False)["mu"].cpu().numpy().astype(np.float64)
    _clean()
    f, b = oav.linear_fwd_bwd(case.x.astype(np.float64), case.w.astype(np.float64), case.d.astype(np.float64),
                              hadamard=True, mu_x=st.mu.cpu().numpy().astype(np.float64), mu_d=mu_d)
    assert rel_fro(y.cpu().numpy(), f.y) < TOL
    assert rel_fro(dx.cpu().numpy(), b.dx) < TOL
    assert rel_fro(dw.cpu().numpy(), b.dw) < TOL


@pytest.mark.parametrize("split", [True, False])
def test_grouped_tiny(debug_lib, split):
    import torch
    from mean_residual_gemm_col_b300 import capi

    m, n = 32, 48
    counts = [16, 0, 48, 1, 32]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    g = workloads.rng(31)
    x = workloads.activation(g, int(offsets[-1]), m, spike=50.0)
    d = workloads.output_grad(g, int(offsets[-1]), n)
    ws = [workloads.weight(g, m, n) for _ in counts]
    w_n, w_m = zip(*[capi.averis_quantize_weight(to_dev_bf16(w)) for w in ws])
    gl = capi.GroupedLinear(offsets, m, n, list(w_m), list(w_n), "cuda")
    flags = capi.AVERIS_MEAN_SPLIT if split else 0
    xd, dd = to_dev_bf16(x), to_dev_bf16(d)
    y = gl.fwd(xd, flags).cpu().numpy()
    dx, dw = gl.bwd(dd, flags)
    dx = dx.cpu().numpy()
    torch.cuda.synchronize()
    _clean()
    for e, (a, b) in enumerate(zip(offsets[:-1], offsets[1:])):
        if b == a:
            continue
        mu_x = mu_d = None
        if split:
            mu_x = gl.states[e].mu.cpu().numpy().astype(np.float64)
            mu_d = capi.averis_quantize(dd[a:b].contiguous(), capi.AVERIS_MEAN_SPLIT, want_row=False,
                                        want_col=False)["mu"].cpu().numpy().astype(np.float64)
        f, bw = oav.linear_fwd_bwd(x[a:b].astype(np.float64), ws[e].astype(np.float64), d[a:b].astype(np.float64),
                                   do_split=split, mu_x=mu_x, mu_d=mu_d)
        assert rel_fro(y[a:b], f.y) < TOL, e
        assert rel_fro(dx[a:b], bw.dx) < TOL, e
        assert rel_fro(dw[e].cpu().numpy(), bw.dw) < TOL, e
    _clean()


@pytest.mark.parametrize("N,K", [(16, 16), (48, 32), (33, 48)])
def test_rank1_tiny(debug_lib, N, K):
    from mean_residual_gemm_col_b300 import capi

    rng = np.random.default_rng(N + K)
    mu = onv.quantize((rng.standard_normal((1, K)) * 8).astype(np.float32).astype(np.float64))
    w = onv.quantize((rng.standard_normal((N, K)) * 0.02).astype(np.float32).astype(np.float64))
    dev = lambda q, r, c: capi.NVFP4Tensor.from_canonical(q.codes, q.scales, q.s_g, r, c, "cuda")  # noqa: E731
    out = capi.averis_rank1(dev(mu, 1, K), dev(w, N, K)).cpu().numpy()
    _clean()
    assert rel_fro(out, (mu.dequantize() @ w.dequantize().T)[0]) < 1e-6


@pytest.mark.parametrize("m,n", [(16, 16), (48, 32), (32, 48)])
@pytest.mark.parametrize("hadamard", [False, True])
def test_grouped_weight_quantize_tiny(debug_lib, m, n, hadamard):
    import torch
    from mean_residual_gemm_col_b300 import capi

    E = 3
    g = workloads.rng(m * 3 + n)
    w = np.stack([workloads.weight(g, m, n) for _ in range(E)])
    wd = to_dev_bf16(w.reshape(E * m, n)).view(E, m, n)
    flags = capi.AVERIS_HADAMARD16 if hadamard else 0
    g_n, g_m = capi.averis_quantize_weight_grouped(wd, flags)
    _clean()
    for e in range(E):
        s_n, s_m = capi.averis_quantize_weight(wd[e].contiguous(), flags)
        for a, b in ((g_n[e], s_n), (g_m[e], s_m)):
            nb = -(-a.cols // 16) * 8  # the bytes that hold codes (row padding is not written)
            assert torch.equal(a.codes[:, :nb], b.codes[:, :nb]) and torch.equal(a.scales, b.scales)
            assert torch.equal(a.tensor_scale, b.tensor_scale)
    _clean()

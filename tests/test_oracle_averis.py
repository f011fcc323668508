"""Pins of the oracle's mean split and linear forward / backward (CPU only)."""

from fractions import Fraction

import numpy as np
import pytest

from oracle import averis, formats, hadamard
from tests import _exact
import workloads


def _case(seed, l, m, n, spike=50.0):
    c = workloads.linear_case(seed, l, m, n, spike=spike)
    return c.x.astype(np.float64), c.w.astype(np.float64), c.d.astype(np.float64)


def _rel(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


# ------------------------------------------------------- mean / split ----

def test_residual_columns_sum_to_zero():
    x, _, d = _case(0, 96, 48, 32)
    for t in (x, d):
        s = averis.split(t, True, exact=True)
        assert np.all(np.abs(s.residual.sum(0)) <= 1e-12 * np.abs(t).sum(0))
        s32 = averis.split(t, True)
        # binary32 residual: each element off by at most half an ulp of itself
        bound = 0.5 * np.spacing(np.abs(s32.residual).astype(np.float32)).astype(np.float64).sum(0) + 1e-30
        assert np.all(np.abs(s32.residual.sum(0) - (t - s32.mu).sum(0)) <= bound)


def test_pythagoras_mean_and_residual_are_orthogonal():
    x, _, _ = _case(1, 80, 64, 16)
    s = averis.split(x, True, exact=True)
    l = x.shape[0]
    lhs = np.sum(x * x)
    rhs = l * np.sum(s.mu ** 2) + np.sum(s.residual ** 2)
    assert abs(lhs - rhs) <= 1e-12 * lhs


def test_mean_fp32_is_rounded_float64_mean():
    x, _, _ = _case(2, 33, 16, 16)
    mu = averis.mean_fp32(x)
    exact = [sum(Fraction(float(v)) for v in x[:, j]) / x.shape[0] for j in range(x.shape[1])]
    assert [Fraction(float(v)) for v in mu] == [_exact.rf32(e) for e in exact]


# ------------------------------------------------------ split algebra ----

@pytest.mark.parametrize("had", [False, True])
def test_identity_quantizer_reproduces_plain_products(had):
    x, w, d = _case(3, 64, 48, 80)
    f, b = averis.linear_fwd_bwd(x, w, d, do_split=True, hadamard=had, exact=True)
    assert _rel(f.y, x @ w) < 1e-12
    assert _rel(b.dx, d @ w.T) < 1e-12
    assert _rel(b.dw, x.T @ d) < 1e-12


def test_cross_terms_vanish():
    x, _, d = _case(4, 64, 32, 48)
    sx = averis.split(x, True, exact=True)
    sd = averis.split(d, True, exact=True)
    l = x.shape[0]
    c1 = sx.residual.T @ (np.ones((l, 1)) @ sd.mu[None, :])
    c2 = (np.ones((l, 1)) @ sx.mu[None, :]).T @ sd.residual
    scale = np.abs(x).T @ np.abs(d)
    assert np.all(np.abs(c1) <= 1e-12 * scale)
    assert np.all(np.abs(c2) <= 1e-12 * scale)


# --------------------------------------------------- quantized cases ----

def test_matches_exact_rational_bruteforce_tiny():
    """The whole quantized layer against an independent exact-rational re-derivation."""
    for seed, (l, m, n), split in [(5, (20, 32, 16), True), (6, (16, 16, 48), True), (7, (20, 32, 16), False)]:
        x, w, d = _case(seed, l, m, n)
        f, b = averis.linear_fwd_bwd(x, w, d, do_split=split)
        fr = lambda a: [[Fraction(float(v)) for v in row] for row in a]
        ref = _exact.averis_layer(fr(x), fr(w), fr(d), split=split)
        if split:
            assert [Fraction(float(v)) for v in f.x_split.mu] == ref["mu_x"]
            assert [Fraction(float(v)) for v in b.d_split.mu] == ref["mu_d"]
        for got, key in ((f.y, "y"), (b.dx, "dx"), (b.dw, "dw")):
            want = np.array([[float(v) for v in row] for row in ref[key]])
            assert _rel(got, want) < 1e-14, key


def test_identity_weight():
    """W = I: every column of Y is c * (dequantized input), c the dequantized diagonal."""
    x, _, _ = _case(8, 64, 64, 64)
    w = np.eye(64)
    f = averis.linear_fwd(x, w)
    c = 6.0 * 448.0 * float(formats.f32(1.0 / 2688.0))
    assert np.all(f.w_m.value[np.eye(64, dtype=bool)] == c)
    assert np.array_equal(f.y, c * f.x_k.value + c * f.mu_x.value)


def test_zero_mean_input_equals_vanilla():
    x, w, d = _case(9, 32, 48, 32)
    x = np.vstack([x, -x])                # columns sum to exactly zero
    d = np.vstack([d, -d])
    fs, bs = averis.linear_fwd_bwd(x, w, d, do_split=True)
    fv, bv = averis.linear_fwd_bwd(x, w, d, do_split=False)
    assert not fs.x_split.mu.any()
    assert np.array_equal(fs.y, fv.y)
    assert np.array_equal(bs.dx, bv.dx)
    assert np.array_equal(bs.dw, bv.dw)


def test_rank_one_input_reduces_to_mean_term():
    _, w, _ = _case(10, 8, 64, 48)
    mu = workloads.bf16_round(np.linspace(-3, 5, 64).astype(np.float32)).astype(np.float64)
    x = np.tile(mu, (24, 1))
    f = averis.linear_fwd(x, w)
    assert not f.x_split.residual.any()
    assert f.x_k.q.s_g == 0.0
    assert np.array_equal(f.y, np.tile(f.r_x, (24, 1)))
    assert np.array_equal(f.r_x, (f.mu_x.value @ f.w_m.value.T)[0])


def test_averis_reduces_activation_error_on_planted_mean():
    """The method's premise on spiked, mean-biased input: the split lowers X's NVFP4 error.

    The mean vector is itself quantized and broadcast to every token, so its own
    NVFP4 error bounds the gain; on this recipe the split wins by roughly 20%.
    """
    x, w, _ = _case(11, 256, 256, 256)
    fs = averis.linear_fwd(x, w, do_split=True)
    fv = averis.linear_fwd(x, w, do_split=False)
    recon = fs.x_k.value + fs.mu_x.value
    assert _rel(recon, x) < 0.9 * _rel(fv.x_k.value, x)


def test_ragged_token_count():
    x, w, d = _case(12, 37, 32, 16)
    f, b = averis.linear_fwd_bwd(x, w, d)
    assert f.x_l.q.codes.shape == (32, 48) and b.d_l.q.codes.shape == (16, 48)
    assert b.dw.shape == (32, 16) and b.dx.shape == (37, 32)


# ------------------------------------------------------------ hadamard ----

def test_hadamard_matrix():
    h = hadamard.sylvester_h16()
    assert np.array_equal(h @ h.T, 16 * np.eye(16))
    assert np.array_equal(h, h.T)


def test_fp32_butterfly_close_to_exact_rotation():
    rng = np.random.default_rng(20)
    x = rng.standard_normal((50, 64)).astype(np.float32).astype(np.float64)
    a = hadamard.rotate_fp32(x)
    e = hadamard.rotate_exact(x)
    # four rounded add stages: error bounded by a few ulps of the largest input of the block
    bound = 4 * np.spacing(np.abs(x).reshape(50, 4, 16).max(-1).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(a - e).reshape(50, 4, 16) <= bound[:, :, None] * 4)
    assert np.allclose(hadamard.rotate_exact(e), x, rtol=0, atol=1e-12)


def test_hadamard_quantized_layer_close_to_plain():
    x, w, d = _case(21, 64, 64, 64)
    f, b = averis.linear_fwd_bwd(x, w, d, hadamard=True)
    f0, b0 = averis.linear_fwd_bwd(x, w, d, hadamard=False)
    # a rotation applied to one operand only would leave an O(1) error
    assert _rel(f.y, x @ w) < 0.25 and _rel(b.dx, d @ w.T) < 0.25 and _rel(b.dw, x.T @ d) < 0.25
    assert not np.array_equal(f.y, f0.y)

"""Pins of the oracle's NVFP4 quantizer (CPU only)."""

from fractions import Fraction

import numpy as np
import pytest

from oracle import formats, nvfp4
from tests import _exact
from workloads import bf16_round


def _rand_fp32(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float32).astype(np.float64)


def test_matches_exact_rational_bruteforce():
    rng = np.random.default_rng(10)
    for shape in [(3, 16), (2, 40), (5, 7), (1, 33)]:
        r = _rand_fp32(rng, shape, 3.0)
        r[0, 0] *= 32.0                     # an outlier sets the tensor scale
        q = nvfp4.quantize(r)
        rows = [[Fraction(float(v)) for v in row] for row in r]
        codes, scales, s_g = _exact.quantize_rows(rows)
        assert Fraction(q.s_g) == s_g
        assert q.scales.tolist() == scales
        assert q.codes.tolist() == codes


def test_roundtrip_of_grid_values_is_exact():
    """Values built as code * scale * s_g with a 448 block and 6-codes quantize to themselves."""
    rng = np.random.default_rng(11)
    s_g = 2.0 ** -7
    rows, nb = 4, 3
    normal_scales = np.arange(0x08, 0x7F)                      # normal E4M3 codes
    e = rng.choice(normal_scales, (rows, nb))
    e[0, 0] = 0x7E                                             # 448: the tensor maximum's block
    codes = rng.integers(0, 16, (rows, nb * 16))
    codes[:, ::16] = 7                                         # each block holds a +6
    vals = formats.e2m1_decode(codes).reshape(rows, nb, 16) * formats.e4m3_decode(e)[:, :, None] * s_g
    vals = vals.reshape(rows, nb * 16)
    q = nvfp4.quantize(vals)
    assert q.s_g == s_g
    assert np.array_equal(q.scales, e)
    # -0 inputs are impossible here except where code is 8; compare values
    assert np.array_equal(formats.e2m1_decode(q.codes), formats.e2m1_decode(codes))
    assert np.array_equal(q.dequantize(), vals)


def test_block_max_maps_to_six_and_tensor_max_to_448():
    rng = np.random.default_rng(12)
    r = _rand_fp32(rng, (64, 256), 1.0)
    r[5, 17] = 50.0
    q = nvfp4.quantize(r)
    sc = formats.e4m3_decode(q.scales)
    assert q.scales[5, 1] == 0x7E
    mags = formats.E2M1_MAGNITUDES[q.codes & 7].reshape(64, 16, 16)
    normal = sc >= 2.0 ** -6
    assert np.all(mags.max(axis=2)[normal] == 6.0)


def test_elementwise_error_bound():
    """|r/sb - dec(code)| is at most half the local grid gap (RNE), up to the reciprocal's rounding."""
    rng = np.random.default_rng(13)
    r = _rand_fp32(rng, (32, 128), 2.0)
    r[rng.random(r.shape) < 0.01] *= 32
    q = nvfp4.quantize(r)
    sb = (formats.e4m3_decode(q.scales) * q.s_g)
    v = r.reshape(32, 8, 16) / sb[:, :, None]
    d = formats.e2m1_decode(q.codes).reshape(32, 8, 16)
    a = np.abs(v)                        # the grid interval that holds v sets the gap
    half_gap = np.where(a <= 2.0, 0.25, np.where(a <= 4.0, 0.5, 1.0))
    over = np.abs(v) > 6.0
    err = np.abs(v - d)
    assert np.all(err[~over] <= half_gap[~over] * (1 + 1e-6))
    assert np.all(np.abs(v[over]) <= 6.0 * 16 / 15 + 1e-6)    # e4m3 rounding can push the max past 6


def test_power_of_two_scaling_commutes():
    rng = np.random.default_rng(14)
    r = _rand_fp32(rng, (8, 64), 1.0)
    q1 = nvfp4.quantize(r)
    q2 = nvfp4.quantize(r * 2.0 ** 9)
    assert np.array_equal(q1.codes, q2.codes)
    assert np.array_equal(q1.scales, q2.scales)
    assert q2.s_g == q1.s_g * 2.0 ** 9


def test_zero_tensor_and_zero_block():
    z = np.zeros((2, 32))
    q = nvfp4.quantize(z)
    assert q.s_g == 0.0 and not q.codes.any() and not q.scales.any()
    r = np.zeros((1, 32))
    r[0, 20] = 3.0
    q = nvfp4.quantize(r)
    assert q.scales[0, 0] == 0 and not q.codes[0, :16].any()
    assert q.dequantize()[0, 20] == pytest.approx(3.0, rel=0.1)


def test_negative_values_carry_sign_bit():
    r = np.array([[-1.0, 1.0, -2.0 ** -9, 0.0] + [0.5] * 12])
    q = nvfp4.quantize(r)
    assert q.codes[0, 0] & 8 and not q.codes[0, 1] & 8
    assert q.codes[0, 2] == 8            # rounds to zero, sign kept
    assert q.codes[0, 3] == 0


def test_partial_block_padding():
    rng = np.random.default_rng(15)
    r = _rand_fp32(rng, (3, 20), 1.0)
    q = nvfp4.quantize(r)
    assert q.codes.shape == (3, 32)
    assert not q.codes[:, 20:].any()
    assert q.dequantize().shape == (3, 20)


def test_bf16_inputs_are_binary32():
    rng = np.random.default_rng(16)
    x = bf16_round(rng.standard_normal((4, 16)).astype(np.float32)).astype(np.float64)
    nvfp4.quantize(x)                    # accepted
    with pytest.raises(ValueError):
        nvfp4.quantize(np.array([[0.1] * 16]))   # not binary32

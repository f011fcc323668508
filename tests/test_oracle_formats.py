"""Pins of the oracle's E2M1 / E4M3 encoders (CPU only).

Each check pins the oracle against something other than itself: the golden
format fixtures, torch's independent float8_e4m3fn conversion, and an
exhaustive exact-rational nearest-code search (tests/_exact.py).
"""

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats
from tests import _exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_e2m1_grid_matches_golden():
    rows = _read("e2m1_grid.txt")
    grid = {int(r[0]): float(r[1]) for r in rows if r[0].isdigit()}
    assert [grid[c] for c in range(8)] == list(formats.E2M1_MAGNITUDES)
    for c in range(8):
        assert formats.e2m1_decode(c | 8) == -grid[c]


def test_e2m1_ties_and_saturation_golden():
    for kind, v, code in (r for r in _read("e2m1_grid.txt") if r[0] in ("tie", "sat")):
        assert formats.e2m1_encode(float(v)) == int(code), (kind, v)
        assert formats.e2m1_encode(-float(v)) == int(code) | 8


def _fp32_sweep(rng, lo, hi, n):
    vals = rng.uniform(lo, hi, n).astype(np.float32)
    # every grid midpoint and its binary32 neighbours
    g = formats.E2M1_MAGNITUDES
    mids = ((g[1:] + g[:-1]) / 2).astype(np.float32)
    nb = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(100))])
    grid = np.concatenate([g, np.nextafter(g.astype(np.float32), np.float32(100))]).astype(np.float32)
    fine = (np.arange(-8 * 64, 8 * 64 + 1) / 64.0).astype(np.float32)
    allv = np.concatenate([vals, nb, -nb, grid, -grid, fine])
    return allv.astype(np.float64)


def test_e2m1_encode_matches_exhaustive_search():
    rng = np.random.default_rng(1)
    vals = _fp32_sweep(rng, -8.0, 8.0, 3000)
    got = formats.e2m1_encode(vals)
    for v, c in zip(vals, got):
        want = _exact.e2m1_code(Fraction(float(v)), np.signbit(v))
        assert c == want, (v, c, want)


def test_e2m1_sign_of_zero_kept():
    assert formats.e2m1_encode(0.0) == 0
    assert formats.e2m1_encode(-0.0) == 8
    assert formats.e2m1_encode(-0.2) == 8          # rounds to zero, keeps the sign


def test_e4m3_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = formats.e4m3_decode(np.arange(256))
    both_nan = np.isnan(ref) & np.isnan(ours)
    assert np.array_equal(np.where(both_nan, 0, ref), np.where(both_nan, 0, ours))
    assert formats.E4M3_MAX == 448.0


def test_e4m3_golden_points():
    for r in _read("e4m3_points.txt"):
        if r[0] == "enc":
            assert formats.e4m3_encode_nonneg(float(r[1])) == int(r[2], 16), r
        else:
            assert formats.e4m3_decode(int(r[0], 16)) == float(r[1]), r


def test_e4m3_encode_matches_torch_rne_in_range():
    rng = np.random.default_rng(2)
    # log-uniform over the whole range incl. subnormals, plus exact midpoints
    v = np.exp2(rng.uniform(-12, np.log2(463.9), 20000)).astype(np.float32)
    t = formats.E4M3_NONNEG
    mids = ((t[1:] + t[:-1]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e4)),
                        t.astype(np.float32)])
    v = v[v < 464.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy().astype(np.int64)
    ours = formats.e4m3_encode_nonneg(v.astype(np.float64))
    assert np.array_equal(ours, ref)


def test_e4m3_saturates():
    assert formats.e4m3_encode_nonneg(470.0) == 0x7E
    assert formats.e4m3_encode_nonneg(3.0e38) == 0x7E


def test_e4m3_encode_matches_exhaustive_search():
    rng = np.random.default_rng(3)
    v = np.exp2(rng.uniform(-11, 9.5, 400)).astype(np.float32).astype(np.float64)
    for x, c in zip(v, formats.e4m3_encode_nonneg(v)):
        assert c == _exact.nearest_code(Fraction(float(x)), _exact.E4M3)


def test_f32_rounding_matches_exact_rational():
    rng = np.random.default_rng(4)
    v = rng.standard_normal(500) * np.exp2(rng.integers(-140, 100, 500))
    for x, r in zip(v, formats.f32(v)):
        assert Fraction(float(r)) == _exact.rf32(Fraction(float(x)))


@pytest.mark.parametrize("bad", [np.nan])
def test_e2m1_rejects_nan(bad):
    with pytest.raises(ValueError):
        formats.e2m1_encode(bad)

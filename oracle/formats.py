"""E2M1 and E4M3 number formats, float64 reference encoders.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[P1-quant] names NVFP4's element format, E2M1 (2 exponent bits, 1 mantissa
bit).  The pages give no further constants; this module takes the standard
definitions:

* E2M1: sign bit, exponent bias 1, one subnormal (0.5).  Magnitudes by code
  0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6.  No infinities, no NaN.
* E4M3 (the "FN" variant used for NVFP4 block scales): exponent bias 7,
  3 mantissa bits, subnormals m * 2^-9, maximum 448, code 0x7F / 0xFF is NaN,
  no infinities.

Encoders round to nearest with ties to the EVEN code (the code whose
least-significant bit is 0) and saturate to the largest finite magnitude
("satfinite").  The sign of the input is kept, so a negative input that
rounds to zero encodes as the negative-zero code (E2M1 0x8).  These are the
readings listed for the quantizer; no stochastic rounding anywhere.

Everything is float64 NumPy.  ``f32`` rounds float64 values to the nearest
binary32 value (ties to even), which is how every fp32 operation of the
method is emulated: an IEEE binary32 +, -, *, / of binary32 operands equals
the float64 result of the same operation rounded once to binary32, because
binary64 has more than 2*24+2 significand bits (double rounding is innocuous
for p' >= 2p + 2; S. Figueroa, "When is double rounding innocuous?", 1995).
"""

from __future__ import annotations

import numpy as np


def f32(x):
    """Round float64 value(s) to the nearest binary32 (RNE) and return float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


# ---------------------------------------------------------------- E2M1 ----

def e2m1_decode_magnitude(code3):
    """Magnitude of a 3-bit E2M1 code, from the format definition.

    Exponent field e (2 bits), mantissa bit m; bias 1.
    e == 0: subnormal, value = m * 2^(1-1) * 0.5 = m / 2.
    e >= 1: value = (1 + m/2) * 2^(e-1).
    """
    code3 = np.asarray(code3, dtype=np.int64)
    e = (code3 >> 1) & 3
    m = code3 & 1
    sub = m * 0.5
    norm = (1.0 + m * 0.5) * np.exp2(e - 1.0)
    return np.where(e == 0, sub, norm)


E2M1_MAGNITUDES = e2m1_decode_magnitude(np.arange(8))  # 0, .5, 1, 1.5, 2, 3, 4, 6


def e2m1_decode(code4):
    """Value of a 4-bit E2M1 code (bit 3 is the sign)."""
    code4 = np.asarray(code4, dtype=np.int64)
    mag = E2M1_MAGNITUDES[code4 & 7]
    return np.where(code4 & 8, -mag, mag)


def _rne_on_grid(mag, grid):
    """Index of the nearest grid point to ``mag`` (>= 0), ties to even index.

    ``grid`` is sorted ascending and its index equals the code, so "even
    index" is "even code".  Values above the last grid point saturate to it.
    """
    mag = np.asarray(mag, dtype=np.float64)
    hi = np.searchsorted(grid, mag, side="left")          # grid[hi-1] < mag <= grid[hi]
    hi = np.clip(hi, 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    d_lo = mag - grid[lo]
    d_hi = grid[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(mag >= grid[-1], len(grid) - 1, idx)    # satfinite
    idx = np.where(mag <= grid[0], 0, idx)
    return idx.astype(np.int64)


def e2m1_encode(v):
    """E2M1 code (0..15) of binary32 value(s) ``v``: RNE, satfinite, sign kept."""
    v = np.asarray(v, dtype=np.float64)
    if np.isnan(v).any():
        raise ValueError("E2M1 encode: NaN input is outside the method's domain")
    idx = _rne_on_grid(np.abs(v), E2M1_MAGNITUDES)
    neg = np.signbit(v)
    return (idx | np.where(neg, 8, 0)).astype(np.int64)


# ---------------------------------------------------------------- E4M3 ----

def e4m3_decode(code8):
    """Value of an 8-bit E4M3 (FN) code, from the format definition (NaN for 0x7F/0xFF)."""
    code8 = np.asarray(code8, dtype=np.int64)
    s = (code8 >> 7) & 1
    e = (code8 >> 3) & 15
    m = code8 & 7
    sub = m / 8.0 * 2.0 ** (1 - 7)
    norm = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    val = np.where(e == 0, sub, norm)
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return np.where(s == 1, -val, val)


# non-negative finite E4M3 values, indexed by code 0..126 (monotone in code)
E4M3_NONNEG = e4m3_decode(np.arange(127))
E4M3_MAX = float(E4M3_NONNEG[-1])  # 448


def e4m3_encode_nonneg(v):
    """E4M3 code of non-negative binary32 value(s): RNE, satfinite (max 448)."""
    v = np.asarray(v, dtype=np.float64)
    if (v < 0).any() or np.isnan(v).any():
        raise ValueError("E4M3 block-scale encode expects finite non-negative input")
    return _rne_on_grid(v, E4M3_NONNEG)

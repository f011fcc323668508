"""Exact-rational brute force of the NVFP4 quantizer and the Averis layer.

Test helper, written independently of ``oracle/``: plain Python loops over
``fractions.Fraction`` values, its own binary32 rounding, its own E2M1 / E4M3
tables spelled out by value, and exhaustive nearest-code search.  Used on tiny
inputs to pin the oracle (a dropped term, a wrong sign, index or axis in the
oracle shows up as a mismatch here).
"""

from __future__ import annotations

from fractions import Fraction
import math

# E2M1 magnitudes by code 0..7, spelled out (format definition)
E2M1 = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4), Fraction(6)]


def e4m3_table():
    """Non-negative finite E4M3 values by code 0..126, by enumeration of fields."""
    vals = []
    for code in range(127):
        e, m = code >> 3, code & 7
        if e == 0:
            vals.append(Fraction(m, 8) * Fraction(1, 64))
        else:
            vals.append((1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
    return vals


E4M3 = e4m3_table()
FLT_MAX = Fraction((2 - Fraction(1, 2 ** 23))) * Fraction(2) ** 127


def rf32(q: Fraction) -> Fraction:
    """Round a rational to the nearest binary32 value, ties to even (no overflow handling)."""
    q = Fraction(q)
    if q == 0:
        return Fraction(0)
    s = -1 if q < 0 else 1
    a = abs(q)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    # fix floating log2 error
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 23)
    n = a / ulp
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return s * fl * ulp


def nearest_code(v: Fraction, table) -> int:
    """Exhaustive nearest entry of ``table`` to v >= 0; ties to the even code; saturating."""
    if v >= table[-1]:
        return len(table) - 1
    best, bestd = None, None
    for c, t in enumerate(table):
        d = abs(v - t)
        if bestd is None or d < bestd or (d == bestd and c % 2 == 0 and best % 2 == 1):
            best, bestd = c, d
    return best


def e2m1_code(v: Fraction, negative: bool) -> int:
    c = nearest_code(abs(v), E2M1)
    return c | (8 if negative else 0)


def e2m1_value(code: int) -> Fraction:
    mag = E2M1[code & 7]
    return -mag if code & 8 else mag


def quantize_rows(rows, neg_flags=None):
    """Quantize a list of rows (lists of Fractions, binary32 values) along each row.

    Returns (codes, scale_codes, s_g) with codes padded to a multiple of 16.
    ``neg_flags`` marks elements that are negative zeros.
    """
    A = max((abs(v) for row in rows for v in row), default=Fraction(0))
    s_g = rf32(A / 2688)
    out_codes, out_scales = [], []
    for ri, row in enumerate(rows):
        n = len(row)
        nb = -(-n // 16)
        padded = list(row) + [Fraction(0)] * (nb * 16 - n)
        negs = [False] * (nb * 16)
        for j, v in enumerate(row):
            negs[j] = v < 0 or (neg_flags is not None and neg_flags[ri][j])
        codes, scales = [], []
        for b in range(nb):
            blk = padded[16 * b: 16 * b + 16]
            if s_g == 0:
                e = 0
            else:
                den = rf32(6 * s_g)
                e = nearest_code(rf32(max(abs(v) for v in blk) / den), E4M3)
            sb = rf32(E4M3[e] * s_g)
            inv = Fraction(0) if sb == 0 else min(rf32(1 / sb), FLT_MAX)
            scales.append(e)
            for j, v in enumerate(blk):
                codes.append(e2m1_code(rf32(v * inv), negs[16 * b + j]))
        out_codes.append(codes)
        out_scales.append(scales)
    return out_codes, out_scales, s_g


def dequant_rows(codes, scales, s_g, ncols):
    return [[e2m1_value(codes[r][j]) * E4M3[scales[r][j // 16]] * s_g for j in range(ncols)]
            for r in range(len(codes))]


def transpose(a):
    return [list(col) for col in zip(*a)]


def matmul(a, b):
    """a [p, q] times b [q, r] with Fractions."""
    bt = transpose(b)
    return [[sum((x * y for x, y in zip(row, col)), Fraction(0)) for col in bt] for row in a]


def averis_layer(x, w, d, split=True):
    """Exact Y, dX, dW of the Averis (split=True) or vanilla layer on tiny inputs.

    x [l][m], w [m][n], d [l][n]: lists of Fractions holding bf16 values.
    Follows the forward and gradient equations of the method: means over the
    token axis, binary32 residuals, NVFP4 along each GEMM's contraction axis.
    """
    l, m, n = len(x), len(x[0]), len(w[0])

    def mean_and_residual(t, cols):
        if not split:
            return [Fraction(0)] * cols, [row[:] for row in t]
        mu = [rf32(sum(t[i][j] for i in range(l)) / l) for j in range(cols)]
        return mu, [[rf32(t[i][j] - mu[j]) for j in range(cols)] for i in range(l)]

    mu_x, xr = mean_and_residual(x, m)
    mu_d, dr = mean_and_residual(d, n)

    def deq_along_rows(rows):
        c, s, g = quantize_rows(rows)
        return dequant_rows(c, s, g, len(rows[0]))

    wt = transpose(w)                          # [n][m]: W blocked along m
    wm = deq_along_rows(wt)
    wn = deq_along_rows(w)                     # [m][n]: W blocked along n
    xk = deq_along_rows(xr)                    # [l][m]
    dk = deq_along_rows(dr)                    # [l][n]
    xl = deq_along_rows(transpose(xr))         # [m][l]
    dl = deq_along_rows(transpose(dr))         # [n][l]

    y = matmul(xk, transpose(wm))              # [l][n]
    dx = matmul(dk, transpose(wn))             # [l][m]
    dw = matmul(xl, transpose(dl))             # [m][n]
    if split:
        mux = deq_along_rows([mu_x])[0]
        mud = deq_along_rows([mu_d])[0]
        rx = matmul([mux], transpose(wm))[0]
        rd = matmul([mud], transpose(wn))[0]
        y = [[y[i][j] + rx[j] for j in range(n)] for i in range(l)]
        dx = [[dx[i][j] + rd[j] for j in range(m)] for i in range(l)]
        dw = [[dw[i][j] + l * mux[i] * mud[j] for j in range(n)] for i in range(m)]
    return dict(mu_x=mu_x, mu_d=mu_d, y=y, dx=dx, dw=dw)

"""Two-level NVFP4 block quantizer Q_b and its dequantizer, float64 reference.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[P1-quant] states the idea: a tensor is cut into fixed-size blocks, each
block shares one scale set by the block's largest magnitude, and the values
are mapped to low-bit codes; the element format is E2M1.  The pages fix no
block size, scale format or formula.  The reading taken here (the standard
two-level NVFP4 layout) is:

* blocks of 16 consecutive elements along the chosen axis (the contraction
  axis of the GEMM that will consume the tensor); a last partial block is
  padded with zeros, which changes neither its maximum nor any product;
* one E4M3 scale per block and one binary32 "tensor scale" per tensor;
* every arithmetic step is one binary32 operation, rounded to nearest even:

    A    = max |r| over the whole tensor
    s_g  = fl32(A / (6 * 448))                  tensor (decode) scale
    if s_g == 0: every code and every block scale is 0
    den  = fl32(6 * s_g)
    a_b  = max |r| over block b
    e_b  = E4M3_rne_satfinite(fl32(a_b / den))  block scale code
    sb   = fl32(dec(e_b) * s_g)                  block decode scale
    inv  = min(fl32(1 / sb), FLT_MAX)            (inv = 0 when sb == 0)
    code = E2M1_rne_satfinite(fl32(r * inv))     sign kept

* dequantized value = dec(code) * dec(e_b) * s_g, exact in float64.

The block maximum lands on code 6 (or saturates) whenever e_b is a normal
E4M3 value, and the tensor maximum's block gets e_b = 448.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .formats import f32, e2m1_encode, e2m1_decode, e4m3_encode_nonneg, e4m3_decode

BLOCK = 16
E4M3_MAX = 448.0
E2M1_MAX = 6.0
FLT_MAX = float(np.finfo(np.float32).max)


@dataclass
class NVFP4:
    """An NVFP4 tensor in canonical (unpacked) form.

    codes   int64 [rows, nblocks*16]  E2M1 codes 0..15 (bit 3 = sign)
    scales  int64 [rows, nblocks]     E4M3 codes of the block scales
    s_g     float                     binary32 tensor scale (as float64)
    cols    int                       logical length of the blocked axis
    """

    codes: np.ndarray
    scales: np.ndarray
    s_g: float
    cols: int

    def dequantize(self) -> np.ndarray:
        """float64 [rows, cols]: dec(code) * dec(e_b) * s_g (exact)."""
        rows, padded = self.codes.shape
        vals = e2m1_decode(self.codes).reshape(rows, padded // BLOCK, BLOCK)
        sc = e4m3_decode(self.scales)[:, :, None]
        return (vals * sc * self.s_g).reshape(rows, padded)[:, : self.cols]


def quantize(r, s_g=None) -> NVFP4:
    """Q_b along the LAST axis of a 2-D array of binary32 values ``r``.

    ``r`` holds binary32 values (stored as float64).  ``s_g`` overrides the
    tensor scale (used only by tests); by default it is computed from the
    tensor's own maximum as stated in the module docstring.  Follows the
    blockwise-quantization description of [P1-quant] with the NVFP4 reading
    above.
    """
    r = np.asarray(r, dtype=np.float64)
    if r.ndim != 2:
        raise ValueError("quantize expects a 2-D array blocked along its last axis")
    if not np.array_equal(f32(r), r):
        raise ValueError("quantize expects binary32-representable values")
    rows, cols = r.shape
    nb = -(-cols // BLOCK)
    padded = np.zeros((rows, nb * BLOCK), dtype=np.float64)
    padded[:, :cols] = r

    if s_g is None:
        amax = float(np.max(np.abs(r))) if r.size else 0.0
        s_g = float(f32(amax / (E2M1_MAX * E4M3_MAX)))

    blocks = padded.reshape(rows, nb, BLOCK)
    if s_g == 0.0:
        # all-zero tensor: every block scale is 0 and so is every reciprocal
        e_b = np.zeros((rows, nb), np.int64)
    else:
        den = float(f32(E2M1_MAX * s_g))
        a_b = np.max(np.abs(blocks), axis=2)
        e_b = e4m3_encode_nonneg(f32(a_b / den))
    sb = f32(e4m3_decode(e_b) * s_g)
    with np.errstate(divide="ignore"):
        inv = np.where(sb > 0, np.minimum(f32(1.0 / np.where(sb > 0, sb, 1.0)), FLT_MAX), 0.0)
    # a zero reciprocal maps every element of the block to a signed zero code
    v = f32(blocks * inv[:, :, None])
    codes = e2m1_encode(v).reshape(rows, nb * BLOCK)
    return NVFP4(codes, e_b.astype(np.int64), s_g, cols)


def quantize_vector(v) -> NVFP4:
    """Q_b of a 1-D vector (a column mean), treated as one row of length m."""
    return quantize(np.asarray(v, dtype=np.float64)[None, :])

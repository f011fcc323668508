"""16x16 Hadamard rotation of the Averis-Hadamard variant, float64 reference.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[P1-hadamard]: reshape the activation to [l, m/16, 16] and apply a 16x16
Hadamard transform along the last axis.  Reading taken here:

* H16 is the Sylvester Hadamard matrix (H1 = [1], H2k = [[Hk, Hk], [Hk, -Hk]]),
  scaled by 1/4 so that H16/4 is orthogonal and symmetric: (H/4)(H/4) = I.
* It is applied to 16-element blocks along the contraction axis of each GEMM
  (m for the forward, n for the input gradient, l for the weight gradient),
  to both operands, so every exact product is unchanged.
* The rotation of a block of binary32 values is computed in binary32 as a
  fast Walsh-Hadamard butterfly with stage strides 1, 2, 4, 8 (each a+b and
  a-b rounded once), followed by a multiplication by 1/4 (rounded once).  The
  oracle emulates exactly these roundings, so both sides feed identical
  binary32 values to the quantizer.  ``rotate_exact`` is the plain float64
  matrix product, used to bound the butterfly's rounding error.
"""

from __future__ import annotations

import numpy as np

from .formats import f32


def sylvester_h16() -> np.ndarray:
    """The 16x16 Sylvester Hadamard matrix (entries +/-1), float64."""
    h = np.array([[1.0]])
    while h.shape[0] < 16:
        h = np.block([[h, h], [h, -h]])
    return h


def rotate_exact(x: np.ndarray) -> np.ndarray:
    """float64 (H16/4) applied to 16-blocks along the last axis (length % 16 == 0)."""
    x = np.asarray(x, dtype=np.float64)
    shp = x.shape
    if shp[-1] % 16:
        raise ValueError("rotation axis must be a multiple of 16")
    blk = x.reshape(shp[:-1] + (shp[-1] // 16, 16))
    out = blk @ (sylvester_h16() / 4.0).T
    return out.reshape(shp)


def rotate_fp32(x: np.ndarray) -> np.ndarray:
    """binary32 butterfly rotation of 16-blocks along the last axis.

    Stage strides 1, 2, 4, 8; in each stage element j (with bit ``h`` of j
    clear) and element j+h become a+b and a-b, each rounded to binary32;
    finally every value is multiplied by 0.25 and rounded.
    """
    x = np.asarray(x, dtype=np.float64)
    shp = x.shape
    if shp[-1] % 16:
        raise ValueError("rotation axis must be a multiple of 16")
    if not np.array_equal(f32(x), x):
        raise ValueError("rotate_fp32 expects binary32-representable values")
    v = x.reshape(shp[:-1] + (shp[-1] // 16, 16)).copy()
    for h in (1, 2, 4, 8):
        for j in range(16):
            if j & h:
                continue
            a = v[..., j].copy()
            b = v[..., j + h].copy()
            v[..., j] = f32(a + b)
            v[..., j + h] = f32(a - b)
    v = f32(v * 0.25)
    return v.reshape(shp)

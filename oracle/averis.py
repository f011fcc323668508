"""Averis mean-residual split linear layer, forward and backward, float64 reference.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Notation of [P1-method]: X in R^{l x m} (tokens x features, the [b, s, m]
activation reshaped), W in R^{m x n}, Y = X W, output gradient D in R^{l x n},
dX = D W^T, dW = X^T D.

Forward ([P1-method], forward equation; [P2-method]):
    mu_X = (1/l) 1^T X,  X_R = X - 1 mu_X
    Y = 1 (Q(mu_X) Q(W)) + Q(X_R) Q(W)            (mean term broadcast, not materialised)
Backward ([P1-method], gradient equations):
    mu_D = (1/l) 1^T D,  D_R = D - 1 mu_D
    dX = 1 (Q(mu_D) Q(W)^T) + Q(D_R) Q(W)^T
    dW = Q(X_R)^T Q(D_R) + l Q(mu_X)^T Q(mu_D)     (cross terms dropped as written)

Readings taken where the pages are silent (each applies to both sides):
* mu is stored in binary32: mu32 = fl32(float64 column mean); the residual is
  one binary32 subtraction r = fl32(x - mu32).  Functions accept ``mu_x`` /
  ``mu_d`` to take a given binary32 mean instead ("given the same mu").
* Q is the NVFP4 quantizer of ``oracle.nvfp4`` blocked along the contraction
  axis of the GEMM that consumes the operand: X_R along m and W along m for Y;
  D_R along n and W along n for dX; X_R and D_R along l for dW.  The same
  real X_R is therefore quantized twice (once per axis), each with the
  tensor's one global maximum.
* mu is quantized as its own one-row tensor along m (resp. n).
* The rank-one terms use the same quantized W as the residual GEMM of that
  pass (W blocked along m in Y, along n in dX).
* Vanilla NVFP4 ("split=False") quantizes X, D, W directly, with no mean
  terms: Y = Q(X)Q(W), dX = Q(D)Q(W)^T, dW = Q(X)^T Q(D).
* Hadamard variant ("hadamard=True", [P1-hadamard]): the operand values are
  rotated by H16/4 in 16-blocks along each GEMM's contraction axis before
  quantization (``oracle.hadamard.rotate_fp32``); the mean vectors are rotated
  along m (resp. n) for the rank-one terms of Y and dX.  For the dW outer
  product the dequantized rotated means are rotated back (H16/4 is its own
  inverse) in float64.  Along l the residuals are zero-padded to a multiple
  of 16 before rotating, and dW's contraction runs over the padded length.
* ``exact=True`` replaces every quantizer by the identity and every binary32
  rounding by float64 (used to check the split algebra).
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

from .formats import f32
from .nvfp4 import NVFP4, quantize
from .hadamard import rotate_fp32, rotate_exact


def column_mean(t: np.ndarray) -> np.ndarray:
    """float64 column mean mu = (1/l) 1^T T  ([P1-method])."""
    t = np.asarray(t, dtype=np.float64)
    return t.sum(axis=0) / t.shape[0]


def mean_fp32(t: np.ndarray) -> np.ndarray:
    """The binary32 mean that both sides store: fl32 of the float64 mean."""
    return f32(column_mean(t))


def residual_fp32(t: np.ndarray, mu32: np.ndarray) -> np.ndarray:
    """X_R = X - 1 mu as one binary32 subtraction per element ([P1-method])."""
    return f32(np.asarray(t, np.float64) - np.asarray(mu32, np.float64)[None, :])


def _pad_cols16(a: np.ndarray) -> np.ndarray:
    rows, cols = a.shape
    c16 = -(-cols // 16) * 16
    if c16 == cols:
        return a
    out = np.zeros((rows, c16), dtype=np.float64)
    out[:, :cols] = a
    return out


@dataclass
class Operand:
    """One quantized operand: NVFP4 form (None in exact mode) and its float64 value."""

    q: Optional[NVFP4]
    value: np.ndarray          # dequantized values (exact mode: the unquantized values)


def _operand(a: np.ndarray, rotate: bool, exact: bool) -> Operand:
    """Rotate (optional) then quantize ``a`` along its last axis."""
    if rotate:
        a = _pad_cols16(a)
        a = rotate_exact(a) if exact else rotate_fp32(a)
    if exact:
        return Operand(None, a)
    q = quantize(a)
    return Operand(q, q.dequantize())


@dataclass
class Split:
    """Mean / residual of one activation-like tensor ([P1-method])."""

    mu: np.ndarray            # binary32 mean (float64 in exact mode); zeros when split=False
    residual: np.ndarray      # X_R (or X itself when split=False)


def split(t: np.ndarray, do_split: bool, mu: Optional[np.ndarray] = None, exact: bool = False) -> Split:
    t = np.asarray(t, dtype=np.float64)
    if not do_split:
        return Split(np.zeros(t.shape[1]), t.copy())
    if exact:
        m = column_mean(t) if mu is None else np.asarray(mu, np.float64)
        return Split(m, t - m[None, :])
    m = mean_fp32(t) if mu is None else np.asarray(mu, np.float64)
    if not np.array_equal(f32(m), m):
        raise ValueError("a given mean must be binary32-representable")
    return Split(m, residual_fp32(t, m))


@dataclass
class Forward:
    y: np.ndarray
    x_split: Split
    x_k: Operand               # X_R blocked along m   [l, m]
    x_l: Operand               # X_R^T blocked along l [m, l (padded to 16 under Hadamard)]
    mu_x: Optional[Operand]    # mu_X blocked along m  [1, m]
    w_m: Operand               # W^T blocked along m   [n, m]
    r_x: Optional[np.ndarray]  # rank-one row Q(mu_X) Q(W)  [n]
    mu_x_hat: Optional[np.ndarray]  # dequantized mean in the unrotated basis [m]


@dataclass
class Backward:
    dx: np.ndarray
    dw: np.ndarray
    d_split: Split
    d_k: Operand               # D_R blocked along n   [l, n]
    d_l: Operand               # D_R^T blocked along l [n, l]
    mu_d: Optional[Operand]    # mu_D blocked along n  [1, n]
    w_n: Operand               # W blocked along n     [m, n]
    r_d: Optional[np.ndarray]  # rank-one row Q(mu_D) Q(W)^T  [m]
    mu_d_hat: Optional[np.ndarray]


def linear_fwd(x, w, *, do_split=True, hadamard=False, mu_x=None, exact=False) -> Forward:
    """Y of the Averis (or vanilla) linear layer ([P1-method] forward equation)."""
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    l, m = x.shape
    m2, n = w.shape
    if m != m2:
        raise ValueError("X and W disagree on m")
    xs = split(x, do_split, mu_x, exact)
    x_k = _operand(xs.residual, hadamard, exact)
    x_l = _operand(xs.residual.T, hadamard, exact)
    w_m = _operand(w.T, hadamard, exact)
    y = x_k.value @ w_m.value.T
    mu_op = r_x = mu_hat = None
    if do_split:
        mu_op = _operand(xs.mu[None, :], hadamard, exact)
        r_x = (mu_op.value @ w_m.value.T)[0]
        y = y + r_x[None, :]           # broadcast over tokens, never materialised as a matrix
        mu_hat = mu_op.value[0]
        if hadamard:
            mu_hat = rotate_exact(mu_hat[None, :])[0]
    return Forward(y, xs, x_k, x_l, mu_op, w_m, r_x, mu_hat)


def linear_bwd(d, w, fwd: Forward, *, do_split=True, hadamard=False, mu_d=None, exact=False) -> Backward:
    """dX and dW of the Averis (or vanilla) linear layer ([P1-method] gradient equations)."""
    d = np.asarray(d, np.float64)
    w = np.asarray(w, np.float64)
    l, n = d.shape
    m, n2 = w.shape
    if n != n2:
        raise ValueError("D and W disagree on n")
    ds = split(d, do_split, mu_d, exact)
    d_k = _operand(ds.residual, hadamard, exact)
    d_l = _operand(ds.residual.T, hadamard, exact)
    w_n = _operand(w, hadamard, exact)
    dx = d_k.value @ w_n.value.T
    dw = fwd.x_l.value @ d_l.value.T
    mu_op = r_d = mu_hat = None
    if do_split:
        mu_op = _operand(ds.mu[None, :], hadamard, exact)
        r_d = (mu_op.value @ w_n.value.T)[0]
        dx = dx + r_d[None, :]
        mu_hat = mu_op.value[0]
        if hadamard:
            mu_hat = rotate_exact(mu_hat[None, :])[0]
        dw = dw + l * np.outer(fwd.mu_x_hat[:m], mu_hat[:n])
    return Backward(dx, dw, ds, d_k, d_l, mu_op, w_n, r_d, mu_hat)


def linear_fwd_bwd(x, w, d, *, do_split=True, hadamard=False, mu_x=None, mu_d=None, exact=False):
    """Convenience: (Forward, Backward) for one linear layer."""
    f = linear_fwd(x, w, do_split=do_split, hadamard=hadamard, mu_x=mu_x, exact=exact)
    b = linear_bwd(d, w, f, do_split=do_split, hadamard=hadamard, mu_d=mu_d, exact=exact)
    return f, b

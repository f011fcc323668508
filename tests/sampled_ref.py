"""Oracle values of one linear layer's outputs at sampled positions (full-size parity).

At full workload sizes the oracle cannot form every product, but NVFP4
quantization is row-local once the tensor scale is fixed: a sampled entry of
Y, dX or dW needs only the rows (or columns) of its two operands, quantized
with the tensor scale of the whole operand.  This module takes the whole
operand's maximum in row or column chunks and quantizes only the rows a
sample needs, composing the oracle's own steps in the order
``oracle.averis.linear_fwd`` / ``linear_bwd`` apply them ("均值偏置的诅咒与祝福"
summary, section 方法步骤详情; the Hadamard variant of section Hadamard变换):

  residual  X_R = fl32(X - 1 mu)            (oracle.averis.residual_fp32)
  rotation  H16/4 along the blocked axis    (oracle.hadamard.rotate_fp32)
  quantize  Q_b along the blocked axis      (oracle.nvfp4.quantize, given s_g)
  Y[i, j]   = <deq A_y[i], deq B_y[j]> + r_X[j]
  dX[i, k]  = <deq A_dx[i], deq B_dx[k]> + r_D[k]
  dW[k, j]  = <deq X_R^T[k], deq D_R^T[j]>_l + l mu_hat_X[k] mu_hat_D[j]

``tests/test_sampled_ref.py`` checks these values against the full oracle on
small shapes in every mode, so the sampling adds no arithmetic of its own.
Everything here is float64 NumPy on the host; test infrastructure only.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np

from oracle import averis as oav, nvfp4 as onv
from oracle.formats import f32
from oracle.hadamard import rotate_fp32, rotate_exact

E2M1_X_E4M3 = 6.0 * 448.0
CHUNK = 2048


def tensor_scale(amax: float) -> float:
    """s_g = fl32(A / (6 * 448)), the tensor scale of ``oracle.nvfp4``."""
    return float(f32(amax / E2M1_X_E4M3))


def _pad16(a: np.ndarray) -> np.ndarray:
    rows, cols = a.shape
    c16 = -(-cols // 16) * 16
    if c16 == cols:
        return a
    out = np.zeros((rows, c16))
    out[:, :cols] = a
    return out


def _prep(rows: np.ndarray, had: bool) -> np.ndarray:
    """Rows of binary32 values as the quantizer sees them (rotated under the variant)."""
    return rotate_fp32(_pad16(rows)) if had else rows


def _resid(t: np.ndarray, mu: Optional[np.ndarray]) -> np.ndarray:
    t = np.asarray(t, np.float64)
    return t if mu is None else oav.residual_fp32(t, mu)


@dataclass
class Operand:
    """The 2-D input T of one operand ([l, k]), its binary32 mean and the mode."""

    t: np.ndarray                 # float32 or float64 [l, k] holding bf16 values
    mu: Optional[np.ndarray]      # binary32 mean (float64) or None (vanilla)
    had: bool

    def rows(self, idx) -> np.ndarray:
        """Quantizer input of the rows ``idx`` blocked along k: [len(idx), k]."""
        return _prep(_resid(self.t[idx], self.mu), self.had)

    def cols(self, idx) -> np.ndarray:
        """Quantizer input of the columns ``idx`` blocked along l: [len(idx), l]."""
        mu = None if self.mu is None else np.asarray(self.mu)[idx]
        return _prep(np.ascontiguousarray(_resid(self.t[:, idx], mu).T), self.had)

    def amax_rows(self) -> float:
        a = 0.0
        for r0 in range(0, self.t.shape[0], CHUNK):
            a = max(a, float(np.abs(self.rows(slice(r0, r0 + CHUNK))).max(initial=0.0)))
        return a

    def amax_cols(self) -> float:
        if not self.had:                 # the same values, only blocked differently
            return self.amax_rows()
        a = 0.0
        step = max(16, (CHUNK * 1024) // max(1, self.t.shape[0]))   # about 2 M values per chunk
        for c0 in range(0, self.t.shape[1], step):
            a = max(a, float(np.abs(self.cols(np.arange(c0, min(c0 + step, self.t.shape[1])))).max(initial=0.0)))
        return a


def _deq(rows: np.ndarray, s_g: float) -> np.ndarray:
    return onv.quantize(rows, s_g=s_g).dequantize()


def _mean_hat(mu: np.ndarray, had: bool):
    """(dequantized mean in the quantized basis, in the unrotated basis) of the one-row mean."""
    q = onv.quantize(_prep(np.asarray(mu, np.float64)[None, :], had)).dequantize()[0]
    return q, (rotate_exact(q[None, :])[0] if had else q)


class SampledLinear:
    """Oracle values of Y, dX, dW entries of one layer (Averis or vanilla, optional H16).

    x [l, m], w [m, n], d [l, n] hold bf16 values; ``mu_x`` / ``mu_d`` are the
    binary32 means both sides use ("given the same mean"), None for vanilla.
    """

    def __init__(self, x, w, d, *, mu_x=None, mu_d=None, hadamard=False):
        self.split = mu_x is not None
        if self.split != (mu_d is not None):
            raise ValueError("give both means (Averis) or neither (vanilla)")
        self.l, self.m = x.shape
        self.n = w.shape[1]
        self.had = hadamard
        self.X = Operand(x, mu_x, hadamard)
        self.D = Operand(d, mu_d, hadamard)
        w = np.asarray(w, np.float64)
        # weights in full (small): W^T blocked along m for Y, W blocked along n for dX
        bw_m, bw_n = _prep(np.ascontiguousarray(w.T), hadamard), _prep(w, hadamard)
        self.w_m = _deq(bw_m, tensor_scale(float(np.abs(bw_m).max())))    # [n, m(+pad)]
        self.w_n = _deq(bw_n, tensor_scale(float(np.abs(bw_n).max())))    # [m, n(+pad)]
        self.s_x_row = tensor_scale(self.X.amax_rows())
        self.s_d_row = tensor_scale(self.D.amax_rows())
        self.s_x_col = tensor_scale(self.X.amax_cols())
        self.s_d_col = tensor_scale(self.D.amax_cols())
        self.r_x = self.r_d = self.mu_x_hat = self.mu_d_hat = None
        if self.split:
            qx, self.mu_x_hat = _mean_hat(mu_x, hadamard)
            qd, self.mu_d_hat = _mean_hat(mu_d, hadamard)
            self.r_x = self.w_m @ qx           # [n]
            self.r_d = self.w_n @ qd           # [m]

    def x_rows_q(self, ii):
        """NVFP4 (oracle) of the sampled rows of X_R blocked along m."""
        return onv.quantize(self.X.rows(ii), s_g=self.s_x_row)

    def x_cols_q(self, kk):
        """NVFP4 (oracle) of the sampled columns of X_R (rows of X_R^T) blocked along l."""
        return onv.quantize(self.X.cols(kk), s_g=self.s_x_col)

    def y(self, ii, jj):
        a = self.x_rows_q(ii).dequantize()
        out = np.einsum("sk,sk->s", a, self.w_m[jj])
        return out + self.r_x[jj] if self.split else out

    def dx(self, ii, kk):
        a = _deq(self.D.rows(ii), self.s_d_row)
        out = np.einsum("sk,sk->s", a, self.w_n[kk])
        return out + self.r_d[kk] if self.split else out

    def dw(self, kk, jj):
        a = self.x_cols_q(kk).dequantize()
        b = _deq(self.D.cols(jj), self.s_d_col)
        out = np.einsum("sl,sl->s", a, b)
        if self.split:
            out = out + self.l * self.mu_x_hat[kk] * self.mu_d_hat[jj]
        return out

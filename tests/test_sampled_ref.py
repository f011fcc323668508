"""The sampled full-size reference agrees with the whole-tensor oracle.

``tests/sampled_ref.py`` recomputes single entries of Y, dX and dW from the
oracle's steps on the rows a sample needs, with tensor scales taken over the
whole operands.  On shapes small enough for ``oracle.averis.linear_fwd_bwd``
every entry must agree with it (float64 round-off of a different summation
order only), in each mode: vanilla, Averis, and both with the 16x16 rotation,
including a token count that is not a multiple of 16.
"""

import numpy as np
import pytest

from oracle import averis as oav
import workloads
from tests.sampled_ref import SampledLinear


@pytest.mark.parametrize("shape", [(96, 48, 64), (40, 32, 80)])
@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("had", [False, True])
def test_sampled_entries_equal_full_oracle(shape, split, had):
    l, m, n = shape
    c = workloads.linear_case(5 + l + m, l, m, n, spike=50.0)
    x, w, d = (c.x.astype(np.float64), c.w.astype(np.float64), c.d.astype(np.float64))
    mu_x = oav.mean_fp32(x) if split else None
    mu_d = oav.mean_fp32(d) if split else None
    f, b = oav.linear_fwd_bwd(x, w, d, do_split=split, hadamard=had, mu_x=mu_x, mu_d=mu_d)
    s = SampledLinear(x, w, d, mu_x=mu_x, mu_d=mu_d, hadamard=had)
    ii, jj = np.meshgrid(np.arange(l), np.arange(n), indexing="ij")
    np.testing.assert_allclose(s.y(ii.ravel(), jj.ravel()).reshape(l, n), f.y, rtol=1e-12, atol=1e-12)
    ii, kk = np.meshgrid(np.arange(l), np.arange(m), indexing="ij")
    np.testing.assert_allclose(s.dx(ii.ravel(), kk.ravel()).reshape(l, m), b.dx, rtol=1e-12, atol=1e-12)
    kk, jj = np.meshgrid(np.arange(m), np.arange(n), indexing="ij")
    np.testing.assert_allclose(s.dw(kk.ravel(), jj.ravel()).reshape(m, n), b.dw, rtol=1e-12, atol=1e-10)
    # the quantized X rows / columns are the oracle's own
    q = s.x_rows_q(np.arange(l))
    assert np.array_equal(q.codes, f.x_k.q.codes) and np.array_equal(q.scales, f.x_k.q.scales)
    qc = s.x_cols_q(np.arange(m))
    assert np.array_equal(qc.codes, f.x_l.q.codes) and np.array_equal(qc.scales, f.x_l.q.scales)
    assert q.s_g == f.x_k.q.s_g and qc.s_g == f.x_l.q.s_g

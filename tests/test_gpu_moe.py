"""GPU parity of the grouped (mixture-of-experts) Averis linear layer.

Each expert's rows of the grouped input are an independent linear layer with
the expert's own weights and means (taken over the expert's tokens only); the
oracle runs the single-layer reference per expert, given the GPU's binary32
means.  The row split includes an empty expert and a one-row expert.
"""

import numpy as np
import pytest

from oracle import averis as oav
import workloads
from tests.gpu_util import to_dev_bf16, rel_fro

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.mark.parametrize("split", [True, False])
def test_grouped_linear_matches_per_expert_oracle(cuda_lib, split):
    import torch
    from mean_residual_gemm_col_b300 import capi

    m, n = 64, 128
    counts = [37, 0, 163, 1, 129]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    L = int(offsets[-1])
    g = workloads.rng(21)
    x = workloads.activation(g, L, m, spike=50.0)
    d = workloads.output_grad(g, L, n)
    ws = [workloads.weight(g, m, n) for _ in counts]
    w_n, w_m = zip(*[capi.averis_quantize_weight(to_dev_bf16(w)) for w in ws])
    gl = capi.GroupedLinear(offsets, m, n, list(w_m), list(w_n), "cuda")
    flags = capi.AVERIS_MEAN_SPLIT if split else 0
    xd, dd = to_dev_bf16(x), to_dev_bf16(d)
    y = gl.fwd(xd, flags).cpu().numpy()
    dx, dw = gl.bwd(dd, flags)
    dx = dx.cpu().numpy()
    torch.cuda.synchronize()
    assert capi.averis_last_device_error() == 0
    for e, (a, b) in enumerate(zip(offsets[:-1], offsets[1:])):
        if b == a:
            continue
        xe, de = x[a:b].astype(np.float64), d[a:b].astype(np.float64)
        mu_x = mu_d = None
        if split:
            mu_x = gl.states[e].mu.cpu().numpy().astype(np.float64)
            mu_d = capi.averis_quantize(dd[a:b].contiguous(), capi.AVERIS_MEAN_SPLIT, want_row=False,
                                        want_col=False)["mu"].cpu().numpy().astype(np.float64)
        f, bw = oav.linear_fwd_bwd(xe, ws[e].astype(np.float64), de, do_split=split, mu_x=mu_x, mu_d=mu_d)
        assert rel_fro(y[a:b], f.y) < TOL, e
        assert rel_fro(dx[a:b], bw.dx) < TOL, e
        assert rel_fro(dw[e].cpu().numpy(), bw.dw) < TOL, e

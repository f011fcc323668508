"""The timeout path of the bounded device waits, exercised without any fault.

A host-side diagnostics switch (``averis_debug_starve_next_quantize``) makes
the next quantize call's statistics pass request no input, so every one of its
bounded waits runs out after a short limit: nothing is in flight, nothing
faults, and the kernels return.  The library must then report the timeout
(code 5, the quantize pass) through ``averis_last_device_error``, and the next
ordinary call on the same workspace -- or on the allocation-free call's
library-owned scratch -- must give the same bits as before the timeout (the
control block at the head of the workspace is back to zero).
"""

import numpy as np
import pytest

import workloads
from tests.gpu_util import to_dev_bf16

pytestmark = pytest.mark.gpu

WAIT = 200_000          # SM cycles (about 0.1 ms) per starved wait


def _same(a, b):
    import torch

    for k in ("row", "col", "mu_q"):
        assert torch.equal(a[k].codes, b[k].codes), k
        assert torch.equal(a[k].scales, b[k].scales), k
        assert torch.equal(a[k].tensor_scale, b[k].tensor_scale), k
    assert torch.equal(a["mu"], b["mu"]) and torch.equal(a["mu_hat"], b["mu_hat"])


@pytest.mark.parametrize("noalloc", [False, True])
def test_starved_stats_pass_reports_timeout_and_recovers(cuda_lib, noalloc):
    import torch
    from mean_residual_gemm_col_b300 import capi

    quant = capi.averis_quantize_noalloc if noalloc else capi.averis_quantize
    x = to_dev_bf16(workloads.activation(workloads.rng(91), 4096, 512, spike=50.0))
    want = quant(x, capi.AVERIS_MEAN_SPLIT)
    torch.cuda.synchronize()
    assert capi.averis_last_device_error() == 0

    capi.debug_starve_next_quantize(WAIT)
    quant(x, capi.AVERIS_MEAN_SPLIT)                 # results invalid by design
    assert capi.averis_last_device_error() == 5      # the quantize pass's wait gave up
    assert capi.averis_last_device_error() == 0      # reading clears the word

    for _ in range(2):
        got = quant(x, capi.AVERIS_MEAN_SPLIT)
        torch.cuda.synchronize()
        assert capi.averis_last_device_error() == 0
        _same(got, want)


def test_starve_switch_rejects_out_of_range_limits(cuda_lib):
    assert cuda_lib.averis_debug_starve_next_quantize(10) == 1
    assert cuda_lib.averis_debug_starve_next_quantize(1 << 40) == 1

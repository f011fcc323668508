"""The allocation-free quantize entry point, checked against the ordinary one.

``averis_quantize_noalloc`` serves callers that cannot allocate device
memory (a plugin host that passes an operator only its inputs and outputs,
or code where cudaMalloc's implicit device synchronisation is not allowed):
it takes no workspace and runs on a scratch array inside the library.  Its
results must equal those of ``averis_quantize`` on the same input: every
code, block scale and tensor scale bit for bit, the mean within the 1e-6
bound used elsewhere.  Two different inputs are quantized back to back, so
a call that inherited the previous call's scratch contents would show up in
the second comparison.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""

import ctypes

import numpy as np
import pytest

import workloads
from tests.gpu_util import to_dev_bf16, mu_close

pytestmark = pytest.mark.gpu


def _same_nvfp4(a, b, what):
    ca, sa, ga = a.canonical()
    cb, sb, gb = b.canonical()
    assert ga == gb, f"{what}: tensor scale {ga} vs {gb}"
    assert np.array_equal(ca, cb), f"{what}: {int((ca != cb).sum())} code mismatches"
    assert np.array_equal(sa, sb), f"{what}: {int((sa != sb).sum())} block-scale mismatches"


@pytest.mark.parametrize("flags_name", ["split", "split_h16"])
def test_noalloc_matches_workspace_entry_point_twice(cuda_lib, flags_name):
    import torch
    from mean_residual_gemm_col_b300 import capi

    flags = capi.AVERIS_MEAN_SPLIT | (capi.AVERIS_HADAMARD16 if flags_name == "split_h16" else 0)
    # two calls in a row on different inputs (different shapes, means and spikes)
    for seed, (rows, cols) in ((1, (2048, 1024)), (2, (1000, 512))):
        x32 = workloads.activation(workloads.rng(seed), rows, cols, spike=50.0)
        x = to_dev_bf16(x32)
        got = capi.averis_quantize_noalloc(x, flags)
        torch.cuda.synchronize()
        want = capi.averis_quantize(x, flags)
        torch.cuda.synchronize()
        assert capi.averis_last_device_error() == 0
        ok, worst = mu_close(got["mu"].cpu().numpy(), x32.astype(np.float64),
                             want["mu"].cpu().numpy().astype(np.float64))
        assert ok, f"call {seed}: mean off by {worst:.3g} (relative)"
        _same_nvfp4(got["row"], want["row"], f"call {seed} row layout")
        _same_nvfp4(got["col"], want["col"], f"call {seed} column layout")
        _same_nvfp4(got["mu_q"], want["mu_q"], f"call {seed} mean")
        assert torch.equal(got["mu_hat"], want["mu_hat"])


def test_noalloc_vanilla_matches(cuda_lib):
    import torch
    from mean_residual_gemm_col_b300 import capi

    x = to_dev_bf16(workloads.activation(workloads.rng(3), 512, 768, spike=30.0))
    got = capi.averis_quantize_noalloc(x, 0)
    want = capi.averis_quantize(x, 0)
    torch.cuda.synchronize()
    _same_nvfp4(got["row"], want["row"], "row layout")
    _same_nvfp4(got["col"], want["col"], "column layout")


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_lib):
    from mean_residual_gemm_col_b300 import capi

    lib = cuda_lib
    cap = 8 << 20
    rows, cols = 64, 1024
    for _ in range(40):                  # bounded: the need grows with the column count
        if lib.averis_quantize_workspace_bytes(rows, cols, 1) > cap:
            break
        cols *= 2
    else:
        pytest.skip("the quantize workspace never exceeds the no-alloc scratch")
    fake = ctypes.c_void_p(256)          # never dereferenced: the size check comes first
    nv_row = capi.NVFP4Struct(256, 256, 256, rows, cols)
    st = lib.averis_quantize_noalloc(fake, rows, cols, 0, None, None, None, ctypes.byref(nv_row), None, None)
    assert st == 4, capi.status_string(st)          # AVERIS_ERR_WORKSPACE_TOO_SMALL

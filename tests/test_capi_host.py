"""Host-side checks of the C-ABI library (no GPU needed)."""

import ctypes
import os
import re

import numpy as np
import pytest

from mean_residual_gemm_col_b300 import build, capi, layout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return capi.load()


def _header_functions():
    with open(os.path.join(ROOT, "include", "averis.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b((?:averis|nvfp4)_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _header_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(capi.EXPORTS) == names


def test_debug_build_exports_the_same_symbols():
    """The bounds-checked variant is the same C ABI (only its kernels check more)."""
    dbg = ctypes.CDLL(build.build(debug=True))
    for n in _header_functions():
        assert hasattr(dbg, n), n


def test_release_build_reports_no_bounds_checks(lib):
    # answered without touching a device: the checks are not compiled in
    assert lib.averis_debug_checks() == 0


def test_layout_helpers_agree_with_library(lib):
    for rows, cols in [(1, 16), (200, 272), (8192, 1024), (37, 4096)]:
        assert lib.averis_nvfp4_ld(cols) == layout.code_ld(cols)
        assert lib.averis_nvfp4_code_bytes(rows, cols) == rows * layout.code_ld(cols)
        assert lib.averis_nvfp4_scale_bytes(rows, cols) == layout.scale_bytes(rows, cols)


def test_scale_layout_is_a_bijection_onto_the_used_bytes():
    for rows, cols in [(128, 64), (200, 272), (1, 16), (300, 1024)]:
        off = layout.scale_offsets(rows, cols)
        assert len(np.unique(off)) == off.size
        assert off.max() < layout.scale_bytes(rows, cols)


def test_pack_unpack_roundtrip():
    rng = np.random.default_rng(0)
    for rows, cols in [(3, 16), (130, 272), (5, 1000 - 1000 % 16)]:
        codes = rng.integers(0, 16, (rows, layout.cdiv(cols, 16) * 16))
        scales = rng.integers(0, 127, (rows, layout.cdiv(cols, 16)))
        assert np.array_equal(layout.unpack_codes(layout.pack_codes(codes, rows, cols), rows, cols), codes)
        assert np.array_equal(layout.unpack_scales(layout.pack_scales(scales, rows, cols), rows, cols), scales)


def test_low_nibble_holds_the_even_element():
    b = layout.pack_codes(np.array([[1, 2] + [0] * 14]), 1, 16)
    assert b[0, 0] == 0x21


def test_workspace_sizes_positive(lib):
    assert lib.averis_quantize_workspace_bytes(8192, 1024, 1) > 0
    assert lib.averis_linear_fwd_workspace_bytes(8192, 1024, 4096, 1) > 0
    assert lib.averis_linear_bwd_workspace_bytes(8192, 1024, 4096, 1) > 0
    assert lib.averis_quantize_workspace_bytes(0, 16, 1) == 0


def test_invalid_arguments_rejected_before_any_device_work(lib):
    # null input, bad column count, missing workspace: INVALID_ARG (1), nothing launched
    assert lib.averis_quantize(None, 16, 16, 1, None, None, None, None, None, None, 0, None) == 1
    x = ctypes.c_void_p(256)
    assert lib.averis_quantize(x, 16, 24, 0, None, None, None, None, None, None, 0, None) == 1
    nv = capi.NVFP4Struct(256, 256, 256, 16, 16)
    assert lib.averis_quantize(x, 16, 16, 0, None, None, None, ctypes.byref(nv), None, None, 0, None) == 1
    assert lib.averis_quantize(x, 16, 16, 0, None, None, None, ctypes.byref(nv), None, ctypes.c_void_p(256), 1,
                               None) == 4
    # mismatched K
    a = capi.NVFP4Struct(256, 256, 256, 128, 64)
    b = capi.NVFP4Struct(256, 256, 256, 128, 80)
    assert lib.averis_gemm(ctypes.byref(a), ctypes.byref(b), None, None, None, 0.0, ctypes.c_void_p(256), 128, 0,
                           None) == 1
    # averis_linear_* require the mean split flag
    st = capi.FwdStateStruct()
    assert lib.averis_linear_fwd(x, 16, 16, 16, ctypes.byref(a), 0, x, ctypes.byref(st), x, 1 << 20, None) == 1


def test_grouped_weight_quantize_host_checks(lib):
    # sizes need no device; bad arguments are rejected before any device work
    assert lib.averis_quantize_weight_grouped_workspace_bytes(64, 2048, 1536) > \
        lib.averis_quantize_weight_grouped_workspace_bytes(1, 2048, 1536) > 0
    assert lib.averis_quantize_weight_grouped_workspace_bytes(0, 16, 16) == 0
    nv = (capi.NVFP4Struct * 2)(capi.NVFP4Struct(256, 256, 256, 16, 16), capi.NVFP4Struct(256, 256, 256, 16, 16))
    w = ctypes.c_void_p(256)
    assert lib.averis_quantize_weight_grouped(w, 0, 16, 16, 0, nv, None, w, 1 << 20, None) == 1  # no experts
    assert lib.averis_quantize_weight_grouped(w, 2, 16, 16, 0, None, None, w, 1 << 20, None) == 1  # no outputs
    assert lib.averis_quantize_weight_grouped(None, 2, 16, 16, 0, nv, None, w, 1 << 20, None) == 1  # no input
    assert lib.averis_quantize_weight_grouped(w, 2, 16, 24, 0, nv, None, w, 1 << 20, None) == 1  # n % 16


def test_status_strings(lib):
    for code in range(7):
        assert capi.status_string(code)
    assert b"debug" in lib.averis_status_string(6)

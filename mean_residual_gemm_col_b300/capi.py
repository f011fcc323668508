"""ctypes binding of libaveris.so (argument marshalling only).

Every function here takes torch tensors, allocates the outputs and the
workspace with torch on the tensors' device, and calls the C entry point of
the same name on the current torch stream.  No arithmetic of the method runs
in Python: if the shared library is missing or fails to load, ``load()``
raises, and nothing falls back to another implementation.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np

from . import layout

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libaveris.so")

AVERIS_MEAN_SPLIT = 1
AVERIS_HADAMARD16 = 2
AVERIS_OUT_BF16 = 4

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported architecture", 3: "CUDA error",
          4: "workspace too small", 5: "device-side wait timed out",
          6: "out-of-range access caught by a debug-build check"}

#: every function declared in include/averis.h
EXPORTS = (
    "averis_nvfp4_ld", "averis_nvfp4_code_bytes", "averis_nvfp4_scale_bytes",
    "averis_quantize_workspace_bytes", "averis_quantize", "averis_quantize_weight", "averis_rank1",
    "averis_gemm", "averis_linear_fwd_workspace_bytes", "averis_linear_bwd_workspace_bytes",
    "averis_linear_fwd", "averis_linear_bwd", "nvfp4_linear_fwd", "nvfp4_linear_bwd",
    "averis_status_string", "averis_last_device_error", "averis_version", "averis_quantize_noalloc",
    "averis_debug_checks", "averis_quantize_weight_grouped_workspace_bytes", "averis_quantize_weight_grouped",
    "averis_grouped_linear_fwd_workspace_bytes", "averis_grouped_linear_bwd_workspace_bytes",
    "averis_grouped_linear_fwd", "averis_grouped_linear_bwd", "averis_debug_starve_next_quantize",
)


class NVFP4Struct(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("tensor_scale", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class FwdStateStruct(ctypes.Structure):
    _fields_ = [("x_row", NVFP4Struct), ("x_col", NVFP4Struct), ("mu_q", NVFP4Struct),
                ("mu", ctypes.c_void_p), ("mu_hat", ctypes.c_void_p)]


class AverisError(RuntimeError):
    pass


_lib = None


def _declare(lib):
    P, I64, SZ, U, I, F = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_uint, ctypes.c_int,
                           ctypes.c_float)
    NP = ctypes.POINTER(NVFP4Struct)
    SP = ctypes.POINTER(FwdStateStruct)
    sig = {
        "averis_nvfp4_ld": (I64, [I64]),
        "averis_nvfp4_code_bytes": (SZ, [I64, I64]),
        "averis_nvfp4_scale_bytes": (SZ, [I64, I64]),
        "averis_quantize_workspace_bytes": (SZ, [I64, I64, U]),
        "averis_quantize": (I, [P, I64, I64, U, P, NP, P, NP, NP, P, SZ, P]),
        "averis_quantize_weight": (I, [P, I64, I64, U, NP, NP, P, SZ, P]),
        "averis_rank1": (I, [NP, NP, P, P]),
        "averis_gemm": (I, [NP, NP, P, P, P, F, P, I64, U, P]),
        "averis_linear_fwd_workspace_bytes": (SZ, [I64, I64, I64, U]),
        "averis_linear_bwd_workspace_bytes": (SZ, [I64, I64, I64, U]),
        "averis_linear_fwd": (I, [P, I64, I64, I64, NP, U, P, SP, P, SZ, P]),
        "averis_linear_bwd": (I, [P, I64, I64, I64, SP, NP, U, P, P, P, SZ, P]),
        "nvfp4_linear_fwd": (I, [P, I64, I64, I64, NP, U, P, SP, P, SZ, P]),
        "nvfp4_linear_bwd": (I, [P, I64, I64, I64, SP, NP, U, P, P, P, SZ, P]),
        "averis_status_string": (ctypes.c_char_p, [I]),
        "averis_last_device_error": (I, [P, ctypes.POINTER(I)]),
        "averis_version": (I, []),
        "averis_quantize_noalloc": (I, [P, I64, I64, U, P, NP, P, NP, NP, P]),
        "averis_grouped_linear_fwd_workspace_bytes": (SZ, [P, I64, I64, I64, U]),
        "averis_grouped_linear_bwd_workspace_bytes": (SZ, [P, I64, I64, I64, U]),
        "averis_grouped_linear_fwd": (I, [P, P, I64, I64, I64, P, U, P, P, P, SZ, P]),
        "averis_grouped_linear_bwd": (I, [P, P, I64, I64, I64, P, P, U, P, P, P, SZ, P]),
        "averis_debug_starve_next_quantize": (I, [ctypes.c_longlong]),
        "averis_debug_checks": (I, []),
        "averis_quantize_weight_grouped_workspace_bytes": (SZ, [I64, I64, I64]),
        "averis_quantize_weight_grouped": (I, [P, I64, I64, I64, U, NP, NP, P, SZ, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path: str = LIB_PATH):
    """Load (once) and return the C library; raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise AverisError(f"libaveris.so not built ({path}); run mean_residual_gemm_col_b300.build")
        _lib = _declare(ctypes.CDLL(path))
    return _lib


def _check(status: int, what: str):
    if status != 0:
        raise AverisError(f"{what}: {STATUS.get(status, status)}")


def _stream(device):
    import torch

    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


# ------------------------------------------------------------- tensors ----

@dataclass
class NVFP4Tensor:
    """Device NVFP4 tensor [rows, cols] blocked along cols (torch-owned buffers)."""

    codes: "object"          # torch.uint8 [rows, ld]
    scales: "object"         # torch.uint8 [scale_bytes]
    tensor_scale: "object"   # torch.float32 [1]
    rows: int
    cols: int

    @staticmethod
    def empty(rows: int, cols: int, device) -> "NVFP4Tensor":
        import torch

        return NVFP4Tensor(
            torch.empty((rows, layout.code_ld(cols)), dtype=torch.uint8, device=device),
            torch.zeros(layout.scale_bytes(rows, cols), dtype=torch.uint8, device=device),
            torch.zeros(1, dtype=torch.float32, device=device),
            rows, cols)

    @staticmethod
    def from_canonical(codes: np.ndarray, scales: np.ndarray, s_g: float, rows: int, cols: int,
                       device) -> "NVFP4Tensor":
        """Device tensor from canonical (unpacked) codes / scale codes / tensor scale."""
        import torch

        return NVFP4Tensor(
            torch.from_numpy(layout.pack_codes(codes, rows, cols)).to(device),
            torch.from_numpy(layout.pack_scales(scales, rows, cols)).to(device),
            torch.tensor([s_g], dtype=torch.float32, device=device),
            rows, cols)

    def struct(self) -> NVFP4Struct:
        return NVFP4Struct(self.codes.data_ptr(), self.scales.data_ptr(), self.tensor_scale.data_ptr(),
                           self.rows, self.cols)

    def canonical(self):
        """(codes int64 [rows, nb*16], scales int64 [rows, nb], s_g float) on the host."""
        codes = layout.unpack_codes(self.codes.cpu().numpy(), self.rows, self.cols)
        scales = layout.unpack_scales(self.scales.cpu().numpy(), self.rows, self.cols)
        return codes, scales, float(self.tensor_scale.cpu().item())


@dataclass
class FwdState:
    x_row: NVFP4Tensor
    x_col: NVFP4Tensor
    mu_q: NVFP4Tensor
    mu: "object"        # float32 [m]
    mu_hat: "object"    # float32 [m]

    @staticmethod
    def empty(l: int, m: int, device) -> "FwdState":
        import torch

        return FwdState(NVFP4Tensor.empty(l, m, device), NVFP4Tensor.empty(m, l, device),
                        NVFP4Tensor.empty(1, m, device),
                        torch.zeros(m, dtype=torch.float32, device=device),
                        torch.zeros(m, dtype=torch.float32, device=device))

    def struct(self) -> FwdStateStruct:
        return FwdStateStruct(self.x_row.struct(), self.x_col.struct(), self.mu_q.struct(),
                              self.mu.data_ptr(), self.mu_hat.data_ptr())


_ws_cache = {}


def workspace(nbytes: int, device, key: str = "default"):
    """A cached device workspace of at least ``nbytes`` (256-byte aligned).

    Allocated zero-filled: the library requires the control block at the head
    of a workspace to be zero before its first use and leaves it zero.
    """
    import torch

    k = (str(device), key)
    buf = _ws_cache.get(k)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[k] = buf
    return buf


def _check_bf16(t, name):
    import torch

    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise AverisError(f"{name} must be a contiguous CUDA bf16 tensor")


# ------------------------------------------------------------ functions ----

def averis_quantize(x, flags: int = AVERIS_MEAN_SPLIT, want_row=True, want_col=True):
    """Mean-split NVFP4 of x [rows, cols]; returns dict(mu, mu_q, mu_hat, row, col)."""
    import torch

    lib = load()
    _check_bf16(x, "x")
    R, C = x.shape
    dev = x.device
    split = bool(flags & AVERIS_MEAN_SPLIT)
    row = NVFP4Tensor.empty(R, C, dev) if want_row else None
    col = NVFP4Tensor.empty(C, R, dev) if want_col else None
    mu = torch.zeros(C, dtype=torch.float32, device=dev) if split else None
    mu_hat = torch.zeros(C, dtype=torch.float32, device=dev) if split else None
    mu_q = NVFP4Tensor.empty(1, C, dev) if split else None
    nbytes = lib.averis_quantize_workspace_bytes(R, C, flags)
    ws = workspace(nbytes, dev)
    rs = row.struct() if row else None
    cs = col.struct() if col else None
    ms = mu_q.struct() if mu_q else None
    st = lib.averis_quantize(_ptr(x), R, C, flags, _ptr(mu), ctypes.byref(ms) if ms else None, _ptr(mu_hat),
                             ctypes.byref(rs) if rs else None, ctypes.byref(cs) if cs else None,
                             _ptr(ws), ws.numel(), _stream(dev))
    _check(st, "averis_quantize")
    return dict(mu=mu, mu_q=mu_q, mu_hat=mu_hat, row=row, col=col)


def averis_quantize_noalloc(x, flags: int = AVERIS_MEAN_SPLIT, want_row=True, want_col=True):
    """``averis_quantize`` through the entry point that takes no workspace.

    For callers that cannot allocate device scratch: the library's own
    file-scope scratch array is used instead (calls on one stream only; see
    include/averis.h).  Outputs are allocated here, as in ``averis_quantize``.
    """
    import torch

    lib = load()
    _check_bf16(x, "x")
    R, C = x.shape
    dev = x.device
    split = bool(flags & AVERIS_MEAN_SPLIT)
    row = NVFP4Tensor.empty(R, C, dev) if want_row else None
    col = NVFP4Tensor.empty(C, R, dev) if want_col else None
    mu = torch.zeros(C, dtype=torch.float32, device=dev) if split else None
    mu_hat = torch.zeros(C, dtype=torch.float32, device=dev) if split else None
    mu_q = NVFP4Tensor.empty(1, C, dev) if split else None
    rs = row.struct() if row else None
    cs = col.struct() if col else None
    ms = mu_q.struct() if mu_q else None
    st = lib.averis_quantize_noalloc(_ptr(x), R, C, flags, _ptr(mu), ctypes.byref(ms) if ms else None,
                                     _ptr(mu_hat), ctypes.byref(rs) if rs else None,
                                     ctypes.byref(cs) if cs else None, _stream(dev))
    _check(st, "averis_quantize_noalloc")
    return dict(mu=mu, mu_q=mu_q, mu_hat=mu_hat, row=row, col=col)


def averis_quantize_weight(w, flags: int = 0):
    """(w_n [m, n] blocked along n, w_m [n, m] blocked along m) of W [m, n]."""
    lib = load()
    _check_bf16(w, "w")
    m, n = w.shape
    dev = w.device
    w_n = NVFP4Tensor.empty(m, n, dev)
    w_m = NVFP4Tensor.empty(n, m, dev)
    ws = workspace(lib.averis_quantize_workspace_bytes(m, n, flags), dev)
    a, b = w_n.struct(), w_m.struct()
    _check(lib.averis_quantize_weight(_ptr(w), m, n, flags, ctypes.byref(a), ctypes.byref(b), _ptr(ws), ws.numel(),
                                      _stream(dev)), "averis_quantize_weight")
    return w_n, w_m


def averis_quantize_weight_grouped(w, flags: int = 0, w_n=None, w_m=None):
    """Per expert e of the stacked W [E, m, n]: (w_n[e] [m, n] blocked along n,
    w_m[e] [n, m] blocked along m), as averis_quantize_weight gives, from one
    launch chain.  Preallocated output lists may be passed in (then filled)."""
    lib = load()
    _check_bf16(w, "w")
    if w.dim() != 3:
        raise AverisError("w must be [E, m, n]")
    E, m, n = w.shape
    dev = w.device
    if w_n is None:
        w_n = [NVFP4Tensor.empty(m, n, dev) for _ in range(E)]
    if w_m is None:
        w_m = [NVFP4Tensor.empty(n, m, dev) for _ in range(E)]
    ws = workspace(lib.averis_quantize_weight_grouped_workspace_bytes(E, m, n), dev, "grouped_wq")
    a = (NVFP4Struct * E)(*[t.struct() for t in w_n])
    b = (NVFP4Struct * E)(*[t.struct() for t in w_m])
    _check(lib.averis_quantize_weight_grouped(_ptr(w), E, m, n, flags, a, b, _ptr(ws), ws.numel(), _stream(dev)),
           "averis_quantize_weight_grouped")
    return w_n, w_m


def averis_rank1(mu_q: NVFP4Tensor, w: NVFP4Tensor):
    import torch

    lib = load()
    out = torch.empty(w.rows, dtype=torch.float32, device=w.codes.device)
    a, b = mu_q.struct(), w.struct()
    _check(lib.averis_rank1(ctypes.byref(a), ctypes.byref(b), _ptr(out), _stream(out.device)), "averis_rank1")
    return out


def averis_gemm(a: NVFP4Tensor, b: NVFP4Tensor, col_add=None, row_vec=None, col_vec=None, outer: float = 0.0,
                out_bf16: bool = False, out=None):
    import torch

    lib = load()
    dev = a.codes.device
    if out is None:
        out = torch.empty((a.rows, b.rows), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=dev)
    sa, sb = a.struct(), b.struct()
    _check(lib.averis_gemm(ctypes.byref(sa), ctypes.byref(sb), _ptr(col_add), _ptr(row_vec), _ptr(col_vec),
                           float(outer), _ptr(out), out.stride(0), AVERIS_OUT_BF16 if out_bf16 else 0,
                           _stream(dev)), "averis_gemm")
    return out


def _linear_fwd(name, x, w_m: NVFP4Tensor, flags, out_bf16, state=None, y=None):
    import torch

    lib = load()
    _check_bf16(x, "x")
    l, m = x.shape
    n = w_m.rows
    dev = x.device
    if state is None:
        state = FwdState.empty(l, m, dev)
    if y is None:
        y = torch.empty((l, n), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=dev)
    f = flags | (AVERIS_OUT_BF16 if out_bf16 else 0)
    ws = workspace(lib.averis_linear_fwd_workspace_bytes(l, m, n, f), dev, "fwd")
    ss, wsm = state.struct(), w_m.struct()
    _check(getattr(lib, name)(_ptr(x), l, m, n, ctypes.byref(wsm), f, _ptr(y), ctypes.byref(ss), _ptr(ws),
                              ws.numel(), _stream(dev)), name)
    return y, state


def _linear_bwd(name, d, state: FwdState, w_n: NVFP4Tensor, flags, out_bf16, dx=None, dw=None):
    import torch

    lib = load()
    _check_bf16(d, "d")
    l, n = d.shape
    m = w_n.rows
    dev = d.device
    if dx is None:
        dx = torch.empty((l, m), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=dev)
    if dw is None:
        dw = torch.empty((m, n), dtype=torch.float32, device=dev)
    f = flags | (AVERIS_OUT_BF16 if out_bf16 else 0)
    ws = workspace(lib.averis_linear_bwd_workspace_bytes(l, m, n, f), dev, "bwd")
    ss, wsn = state.struct(), w_n.struct()
    _check(getattr(lib, name)(_ptr(d), l, m, n, ctypes.byref(ss), ctypes.byref(wsn), f, _ptr(dx), _ptr(dw),
                              _ptr(ws), ws.numel(), _stream(dev)), name)
    return dx, dw


def averis_linear_fwd(x, w_m, flags=AVERIS_MEAN_SPLIT, out_bf16=False, state=None, y=None):
    return _linear_fwd("averis_linear_fwd", x, w_m, flags | AVERIS_MEAN_SPLIT, out_bf16, state, y)


def averis_linear_bwd(d, state, w_n, flags=AVERIS_MEAN_SPLIT, out_bf16=False, dx=None, dw=None):
    return _linear_bwd("averis_linear_bwd", d, state, w_n, flags | AVERIS_MEAN_SPLIT, out_bf16, dx, dw)


def nvfp4_linear_fwd(x, w_m, flags=0, out_bf16=False, state=None, y=None):
    return _linear_fwd("nvfp4_linear_fwd", x, w_m, flags, out_bf16, state, y)


def nvfp4_linear_bwd(d, state, w_n, flags=0, out_bf16=False, dx=None, dw=None):
    return _linear_bwd("nvfp4_linear_bwd", d, state, w_n, flags, out_bf16, dx, dw)


class GroupedLinear:
    """Per-expert buffers of a grouped (mixture-of-experts) linear layer.

    ``offsets`` (E+1 ints) split the expert-grouped rows of x [L, m]; weights
    are per expert.  The host arrays the C entry points take (offsets, weight
    descriptors, forward states, dW pointers) are built once here.
    """

    def __init__(self, offsets, m, n, w_m, w_n, device):
        import torch

        self.offsets = [int(o) for o in offsets]
        self.E, self.m, self.n = len(self.offsets) - 1, m, n
        self._off = (ctypes.c_int64 * (self.E + 1))(*self.offsets)
        self.w_m, self.w_n = w_m, w_n
        self._wm = (NVFP4Struct * self.E)(*[w.struct() for w in w_m])
        self._wn = (NVFP4Struct * self.E)(*[w.struct() for w in w_n])
        self.states = [FwdState.empty(max(1, b - a), m, device) for a, b in zip(self.offsets, self.offsets[1:])]
        self._st = (FwdStateStruct * self.E)(*[st.struct() for st in self.states])
        self.dw = [torch.zeros(m, n, dtype=torch.float32, device=device) for _ in range(self.E)]
        self._dw = (ctypes.c_void_p * self.E)(*[t.data_ptr() for t in self.dw])

    def fwd(self, x, flags=AVERIS_MEAN_SPLIT, out_bf16=False, y=None):
        import torch

        lib = load()
        _check_bf16(x, "x")
        dev = x.device
        f = flags | (AVERIS_OUT_BF16 if out_bf16 else 0)
        if y is None:
            y = torch.empty((self.offsets[-1], self.n), dtype=torch.bfloat16 if out_bf16 else torch.float32,
                            device=dev)
        ws = workspace(lib.averis_grouped_linear_fwd_workspace_bytes(self._off, self.E, self.m, self.n, f), dev,
                       "gfwd")
        _check(lib.averis_grouped_linear_fwd(_ptr(x), self._off, self.E, self.m, self.n, self._wm, f, _ptr(y),
                                             self._st, _ptr(ws), ws.numel(), _stream(dev)),
               "averis_grouped_linear_fwd")
        return y

    def bwd(self, d, flags=AVERIS_MEAN_SPLIT, out_bf16=False, dx=None):
        import torch

        lib = load()
        _check_bf16(d, "d")
        dev = d.device
        f = flags | (AVERIS_OUT_BF16 if out_bf16 else 0)
        if dx is None:
            dx = torch.empty((self.offsets[-1], self.m), dtype=torch.bfloat16 if out_bf16 else torch.float32,
                             device=dev)
        ws = workspace(lib.averis_grouped_linear_bwd_workspace_bytes(self._off, self.E, self.m, self.n, f), dev,
                       "gbwd")
        _check(lib.averis_grouped_linear_bwd(_ptr(d), self._off, self.E, self.m, self.n, self._st, self._wn, f,
                                             _ptr(dx), self._dw, _ptr(ws), ws.numel(), _stream(dev)),
               "averis_grouped_linear_bwd")
        return dx, self.dw


def averis_last_device_error(device=None) -> int:
    """0, or the code of the device-side wait that gave up, or (debug build)
    100 + the site of a bounds check that caught an access; then clears it."""
    import torch

    lib = load()
    where = ctypes.c_int(0)
    st = lib.averis_last_device_error(_stream(device or torch.cuda.current_device()), ctypes.byref(where))
    if st not in (0, 5, 6):
        _check(st, "averis_last_device_error")
    return where.value


def debug_starve_next_quantize(wait_cycles: int) -> None:
    """Make the next quantize call's waits for its input run out (timeout-path diagnostics)."""
    _check(load().averis_debug_starve_next_quantize(int(wait_cycles)), "averis_debug_starve_next_quantize")


def status_string(code: int) -> str:
    return load().averis_status_string(code).decode()

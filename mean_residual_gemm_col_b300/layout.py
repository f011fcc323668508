"""Index maps of the library's NVFP4 storage layout (pure layout, no arithmetic).

Codes: row-major bytes, ``ld(cols) = round_up(cols, 64) / 2`` per row; byte j
holds element 2j in its low nibble and 2j+1 in its high nibble.
Scales: E4M3 bytes in 512-byte tiles of 128 rows x 4 blocks; tile (rb, kc) at
``512 * (rb * ceil(cols/64) + kc)``, entry (r, k) at
``16*(r%32) + 4*((r%128)//32) + k%4`` inside it (the operand layout the
tcgen05 block-scaled MMA reads after a 32x128b warpx4 copy to TMEM).
"""

from __future__ import annotations

import numpy as np


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


def code_ld(cols: int) -> int:
    return cdiv(cols, 64) * 32


def scale_bytes(rows: int, cols: int) -> int:
    return 512 * cdiv(rows, 128) * cdiv(cols, 64)


def scale_offsets(rows: int, cols: int, row_idx=None) -> np.ndarray:
    """int64 [rows, ceil(cols/16)]: byte offset of each block scale (only the rows ``row_idx`` if given)."""
    kc = cdiv(cols, 64)
    r = (np.arange(rows, dtype=np.int64) if row_idx is None else np.asarray(row_idx, dtype=np.int64))[:, None]
    k = np.arange(cdiv(cols, 16), dtype=np.int64)[None, :]
    return ((r // 128) * kc + k // 4) * 512 + 16 * (r % 32) + 4 * ((r % 128) // 32) + (k % 4)


def unpack_codes(codes_bytes: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """uint8 [rows, ld] -> int64 [rows, ceil(cols/16)*16] codes 0..15."""
    b = np.asarray(codes_bytes, dtype=np.uint8).reshape(rows, code_ld(cols)).astype(np.int64)
    out = np.empty((rows, 2 * b.shape[1]), dtype=np.int64)
    out[:, 0::2] = b & 15
    out[:, 1::2] = b >> 4
    return out[:, : cdiv(cols, 16) * 16]


def pack_codes(codes: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """int [rows, >= cols] codes -> uint8 [rows, ld] (zero padding)."""
    full = np.zeros((rows, 2 * code_ld(cols)), dtype=np.int64)
    c = np.asarray(codes, dtype=np.int64)
    full[:, : c.shape[1]] = c
    return (full[:, 0::2] | (full[:, 1::2] << 4)).astype(np.uint8)


def unpack_scales(scale_bytes_arr: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """tiled uint8 -> int64 [rows, ceil(cols/16)] E4M3 codes."""
    flat = np.asarray(scale_bytes_arr, dtype=np.uint8).reshape(-1)
    return flat[scale_offsets(rows, cols)].astype(np.int64)


def pack_scales(scales: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """int [rows, ceil(cols/16)] E4M3 codes -> tiled uint8 (padding zero)."""
    out = np.zeros(scale_bytes(rows, cols), dtype=np.uint8)
    out[scale_offsets(rows, cols)] = np.asarray(scales, dtype=np.int64).astype(np.uint8)
    return out

"""The 128x4 swizzled block-scale layout.

Source: [vLLM-SM103] nvfp4_quant_kernels.cu, "Scale factor layout conversion:
SM100 <-> SM103" (the SM100 in-tile offset outerM*16 + innerM*4 + innerK with
outerM = m%32, innerM = (m/32)%4), nvfp4_utils.cuh (tile base
(mTile*numKTiles + kTile)*512, 128 rows x 4 scale columns per 512-byte tile),
and the GEMM entry "SM103 Entry Point" (scale tensors padded to
[round_up(rows,128), round_up(K/16,4)]).

A scale matrix with ``rows`` rows and ``cols`` scale columns (K/16 for NVFP4,
K/32 for MXFP4) is padded to Rp = round_up(rows, 128), Cp = round_up(cols, 4)
and stored as Rp*Cp bytes; padding bytes are 0x00.
"""
from __future__ import annotations

import numpy as np


def round_up(x: int, y: int) -> int:
    return (x + y - 1) // y * y


def padded_shape(rows: int, cols: int) -> tuple[int, int]:
    """(round_up(rows,128), round_up(cols,4)) -- the stored scale matrix shape."""
    return round_up(rows, 128), round_up(cols, 4)


def sf_offset(r, j, cols_padded: int):
    """Byte offset of scale (row r, scale column j) in the swizzled buffer.

    Tile (r // 128, j // 4) sits at (mTile * (Cp/4) + kTile) * 512; inside the
    tile, row r%128 splits into outer index r%32 (stride 16) and inner index
    (r//32)%4 (stride 4), and the scale column j%4 has stride 1.
    """
    r = np.asarray(r, dtype=np.int64)
    j = np.asarray(j, dtype=np.int64)
    k_tiles = cols_padded // 4
    tile = (r // 128) * k_tiles + (j // 4)
    inner = (r % 32) * 16 + ((r // 32) % 4) * 4 + (j % 4)
    return tile * 512 + inner


def swizzle(linear: np.ndarray) -> np.ndarray:
    """Row-major scale bytes [rows, cols] -> swizzled, zero-padded buffer of Rp*Cp bytes."""
    linear = np.asarray(linear, dtype=np.uint8)
    rows, cols = linear.shape
    rp, cp = padded_shape(rows, cols)
    out = np.zeros(rp * cp, dtype=np.uint8)
    rr, jj = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    out[sf_offset(rr, jj, cp)] = linear
    return out


def unswizzle(buf: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Swizzled buffer -> row-major scale bytes [rows, cols] (drops the padding)."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    _, cp = padded_shape(rows, cols)
    rr, jj = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    return buf[sf_offset(rr, jj, cp)]


def unswizzle_padded(buf: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Swizzled buffer -> the full padded matrix [Rp, Cp] (padding included)."""
    rp, cp = padded_shape(rows, cols)
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    rr, jj = np.meshgrid(np.arange(rp), np.arange(cp), indexing="ij")
    return buf[sf_offset(rr, jj, cp)]

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

The SM103 layout (same page, same section, and nvfp4_utils.cuh "SM103 swizzled
SF offset"; nvfp4_utils.py swizzle_blockscale_sm103) keeps the 512-byte tiles
and their order but arranges the bytes of a tile differently: row m of the tile
splits as m = m4b + 4*m4a + 16*m8 and lands at m8*16 + m4a*128 + m4b*4 + k.
(The page's CuTe atom comment, Shape <8,4,4> with Stride <16,128,4>, would read
m = i0 + 8*i1 + 32*i2 in CuTe's column-major mode order; the three code
passages agree with each other on the decomposition above, which is used here.)
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


def sf_offset_sm103(r, j, cols_padded: int):
    """Byte offset of scale (row r, scale column j) in the SM103 layout.

    Same tile base as sf_offset; inside the tile, row m = r%128 splits into
    m4b = m%4 (stride 4), m4a = (m//4)%4 (stride 128), m8 = (m//16)%8 (stride 16),
    and the scale column j%4 has stride 1.
    """
    r = np.asarray(r, dtype=np.int64)
    j = np.asarray(j, dtype=np.int64)
    k_tiles = cols_padded // 4
    tile = (r // 128) * k_tiles + (j // 4)
    m = r % 128
    inner = ((m // 16) % 8) * 16 + ((m // 4) % 4) * 128 + (m % 4) * 4 + (j % 4)
    return tile * 512 + inner


def swizzle_sm103(linear: np.ndarray) -> np.ndarray:
    """Row-major scale bytes [rows, cols] -> SM103-layout, zero-padded buffer of Rp*Cp bytes."""
    linear = np.asarray(linear, dtype=np.uint8)
    rows, cols = linear.shape
    rp, cp = padded_shape(rows, cols)
    out = np.zeros(rp * cp, dtype=np.uint8)
    rr, jj = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    out[sf_offset_sm103(rr, jj, cp)] = linear
    return out


def unswizzle_sm103(buf: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """SM103-layout buffer -> row-major scale bytes [rows, cols] (drops the padding)."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    _, cp = padded_shape(rows, cols)
    rr, jj = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    return buf[sf_offset_sm103(rr, jj, cp)]


def convert_layout(buf: np.ndarray, rows: int, cols: int, to_sm103: bool) -> np.ndarray:
    """Re-arrange a whole swizzled buffer between the two layouts (page section "Scale factor
    layout conversion: SM100 <-> SM103"): every byte of the padded [Rp, Cp] matrix, padding
    included, moves from its offset in one layout to its offset in the other."""
    rp, cp = padded_shape(rows, cols)
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    rr, jj = np.meshgrid(np.arange(rp), np.arange(cp), indexing="ij")
    src, dst = (sf_offset(rr, jj, cp), sf_offset_sm103(rr, jj, cp))
    if not to_sm103:
        src, dst = dst, src
    out = np.zeros(rp * cp, dtype=np.uint8)
    out[dst] = buf[src]
    return out

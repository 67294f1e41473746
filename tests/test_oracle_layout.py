"""Pins for oracle/layout.py: hand-worked offsets, bijection, and an independent
reshape/permute construction of the 128x4 layout."""
import os

import numpy as np
import pytest
import torch

from oracle import layout

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _golden_offsets():
    rows = []
    with open(os.path.join(GOLD, "sf_offsets_128x4.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            rows.append(tuple(int(v) for v in line.split()))
    return rows


def test_offsets_match_hand_worked_values():
    for R, C, r, j, off in _golden_offsets():
        _, cp = layout.padded_shape(R, C)
        assert int(layout.sf_offset(r, j, cp)) == off, (R, C, r, j)


def _permute_construction(mat: np.ndarray) -> np.ndarray:
    """128x4 layout built from the physical order (m_tile, k_tile, 32, 4, 4): the row
    index inside a tile is m = inner_m * 32 + outer_m, outer_m is the 16-byte stride
    axis, inner_m the 4-byte one, inner_k the byte axis (FlashInfer PR 4620 text)."""
    rows, cols = mat.shape
    rp, cp = layout.padded_shape(rows, cols)
    pad = torch.zeros(rp, cp, dtype=torch.int64)
    pad[:rows, :cols] = torch.from_numpy(mat.astype(np.int64))
    v = pad.reshape(rp // 128, 4, 32, cp // 4, 4)         # (m_tile, inner_m, outer_m, k_tile, inner_k)
    return v.permute(0, 3, 2, 1, 4).contiguous().reshape(-1).numpy()


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 5), (128, 4), (129, 4), (256, 448), (300, 37), (1000, 64)])
def test_swizzle_equals_permute_construction(rows, cols):
    rng = np.random.default_rng(rows * 1000 + cols)
    mat = rng.integers(1, 256, size=(rows, cols)).astype(np.uint8)
    assert np.array_equal(layout.swizzle(mat), _permute_construction(mat).astype(np.uint8))


@pytest.mark.parametrize("rows,cols", [(1, 1), (130, 9), (384, 448)])
def test_swizzle_is_bijection_with_zero_padding(rows, cols):
    rp, cp = layout.padded_shape(rows, cols)
    rr, jj = np.meshgrid(np.arange(rp), np.arange(cp), indexing="ij")
    offs = layout.sf_offset(rr, jj, cp).reshape(-1)
    assert np.array_equal(np.sort(offs), np.arange(rp * cp))
    mat = np.random.default_rng(0).integers(1, 256, size=(rows, cols)).astype(np.uint8)
    buf = layout.swizzle(mat)
    assert buf.size == rp * cp
    assert np.array_equal(layout.unswizzle(buf, rows, cols), mat)
    full = layout.unswizzle_padded(buf, rows, cols)
    assert np.all(full[rows:, :] == 0) and np.all(full[:, cols:] == 0)
    assert np.count_nonzero(buf) == rows * cols


def test_tiles_are_contiguous_512_byte_blocks():
    # all 512 bytes of tile (mt, kt) hold rows mt*128.. and columns kt*4..
    rows, cols = 256, 12
    _, cp = layout.padded_shape(rows, cols)
    for mt in range(2):
        for kt in range(3):
            rr, jj = np.meshgrid(np.arange(mt * 128, mt * 128 + 128), np.arange(kt * 4, kt * 4 + 4), indexing="ij")
            offs = np.sort(layout.sf_offset(rr, jj, cp).reshape(-1))
            base = (mt * (cp // 4) + kt) * 512
            assert np.array_equal(offs, np.arange(base, base + 512))


# ---------------------------------------------------------------- SM103 layout
def _golden_offsets_sm103():
    rows = []
    with open(os.path.join(GOLD, "sf_offsets_sm103.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            rows.append(tuple(int(v) for v in line.split()))
    return rows


def test_sm103_offsets_match_hand_worked_values():
    for R, C, r, j, off in _golden_offsets_sm103():
        _, cp = layout.padded_shape(R, C)
        assert int(layout.sf_offset_sm103(r, j, cp)) == off, (R, C, r, j)


def _permute_construction_sm103(mat: np.ndarray) -> np.ndarray:
    """SM103 layout built by reshaping: a tile row m = 16*m8 + 4*m4a + m4b, and the bytes of a
    tile are ordered (m4a, m8, m4b, k) from outermost to innermost (strides 128, 16, 4, 1)."""
    rows, cols = mat.shape
    rp, cp = layout.padded_shape(rows, cols)
    pad = torch.zeros(rp, cp, dtype=torch.int64)
    pad[:rows, :cols] = torch.from_numpy(mat.astype(np.int64))
    v = pad.reshape(rp // 128, 8, 4, 4, cp // 4, 4)      # (m_tile, m8, m4a, m4b, k_tile, k)
    return v.permute(0, 4, 2, 1, 3, 5).contiguous().reshape(-1).numpy()


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 5), (128, 4), (129, 4), (256, 448), (300, 37)])
def test_sm103_swizzle_equals_permute_construction(rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    mat = rng.integers(1, 256, size=(rows, cols)).astype(np.uint8)
    assert np.array_equal(layout.swizzle_sm103(mat), _permute_construction_sm103(mat).astype(np.uint8))


@pytest.mark.parametrize("rows,cols", [(1, 1), (130, 9), (384, 448)])
def test_sm103_is_bijection_with_zero_padding(rows, cols):
    rp, cp = layout.padded_shape(rows, cols)
    rr, jj = np.meshgrid(np.arange(rp), np.arange(cp), indexing="ij")
    offs = layout.sf_offset_sm103(rr, jj, cp).reshape(-1)
    assert np.array_equal(np.sort(offs), np.arange(rp * cp))
    # the same 512-byte tiles as the SM100 layout, only the bytes inside a tile move
    assert np.array_equal(offs // 512, layout.sf_offset(rr, jj, cp).reshape(-1) // 512)
    mat = np.random.default_rng(1).integers(1, 256, size=(rows, cols)).astype(np.uint8)
    buf = layout.swizzle_sm103(mat)
    assert np.array_equal(layout.unswizzle_sm103(buf, rows, cols), mat)
    assert np.count_nonzero(buf) == rows * cols


@pytest.mark.parametrize("rows,cols", [(5, 3), (128, 112), (257, 448)])
def test_layout_conversion_round_trip(rows, cols):
    mat = np.random.default_rng(2).integers(1, 256, size=(rows, cols)).astype(np.uint8)
    a = layout.swizzle(mat)
    b = layout.convert_layout(a, rows, cols, to_sm103=True)
    assert np.array_equal(b, layout.swizzle_sm103(mat))
    assert np.array_equal(layout.convert_layout(b, rows, cols, to_sm103=False), a)
    # padding bytes carry over too: non-zero padding survives the round trip
    a2 = a.copy()
    a2[a2 == 0] = 7
    assert np.array_equal(layout.convert_layout(layout.convert_layout(a2, rows, cols, True), rows, cols, False), a2)

"""Pins for oracle/quant.py: lossless round trips, the global-scale property, zero
blocks, an independent scalar re-derivation on tiny inputs, and the grouped layout."""
import struct

import numpy as np
import pytest
import torch

import synth
from oracle import formats, layout, quant


def f32(v: float) -> float:
    """Round a double to the nearest fp32 (ties to even) and return it as a double."""
    return struct.unpack("<f", struct.pack("<f", v))[0]


def _bf16(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def test_nvfp4_lossless_round_trip():
    rng = np.random.default_rng(0)
    e2m1 = formats.e2m1_decode(np.arange(16))
    e4m3 = formats.e4m3_decode(np.arange(1, 0x7F))
    for gs in (1.0, 2.0 ** 5, 2.0 ** -3):
        m, k = 16, 64
        codes = rng.integers(0, 16, size=(m, k))
        codes[:, ::16] = 7                                  # every block holds |6|
        sd_codes = rng.choice(np.nonzero((e4m3 <= 74) & (e4m3 >= 2.0 ** -6))[0] + 1, size=(m, k // 16))
        sd = formats.e4m3_decode(sd_codes)
        x = e2m1[codes] * np.repeat(sd, 16, axis=1) / gs
        assert np.array_equal(_bf16(x), x)                   # exactly representable
        got_codes, got_sc = quant.nvfp4_block_codes(x.astype(np.float32), gs)
        assert np.array_equal(got_sc, sd_codes)
        # the sign of zero is kept, so compare codes exactly
        assert np.array_equal(got_codes, codes)


def test_nvfp4_block_with_tensor_amax_gets_448():
    x = synth.activation(3, 64, 256).float().numpy()
    amax = np.float32(np.abs(x).max())
    gs = np.float32(2688.0) / amax
    codes, sc = quant.nvfp4_block_codes(x, gs)
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert sc[r, c // 16] == 0x7E
    assert np.all(sc <= 0x7E)
    # the amax element itself maps to +-6
    assert codes[r, c] & 7 == 7


def test_nvfp4_zero_blocks():
    x = np.zeros((4, 32), dtype=np.float32)
    x[1, :16] = -0.0
    x[2, 16:] = 1.0
    codes, sc = quant.nvfp4_block_codes(x, 1.0)
    assert np.all(sc[0] == 0) and sc[1, 0] == 0 and sc[2, 0] == 0 and sc[2, 1] != 0
    assert np.all(codes[0] == 0)
    assert np.all(codes[1, :16] == 8)                       # -0.0 keeps its sign
    q, sf = quant.nvfp4_quantize(x, 1.0)
    assert sf.size == 128 * 4
    assert np.count_nonzero(sf) == 1                        # padding rows/cols are 0x00


def _scalar_nvfp4(x: np.ndarray, gs: float):
    """Independent scalar derivation: doubles rounded to fp32 after every operation
    (exact for products of fp32s; double rounding is innocuous for / at these widths),
    e4m3/e2m1 by nearest-grid search with ties to the even code."""
    e4 = [(float(v), c) for c, v in enumerate(formats.e4m3_decode(np.arange(0x7F)))]
    e2 = [(float(v), c) for c, v in enumerate(formats.e2m1_decode(np.arange(8)))]

    def nearest(grid, v):
        best = min(abs(g - v) for g, _ in grid)
        cs = [c for g, c in grid if abs(g - v) == best]
        ev = [c for c in cs if c % 2 == 0]
        return ev[0] if ev else cs[0]

    m, k = x.shape
    codes = np.zeros((m, k), dtype=np.int64)
    scs = np.zeros((m, k // 16), dtype=np.int64)
    for r in range(m):
        for b in range(k // 16):
            blk = [float(v) for v in x[r, 16 * b: 16 * b + 16]]
            amax = max(abs(v) for v in blk)
            s = f32(f32(gs * amax) / 6.0)
            sc = 0x7E if s >= 448 else nearest(e4, s)
            sd = e4[sc][0]
            inv = 0.0 if sd == 0 else f32(gs / sd)
            scs[r, b] = sc
            for i, v in enumerate(blk):
                y = f32(v * inv)
                c = nearest(e2, min(abs(y), 6.0))
                codes[r, 16 * b + i] = c | (8 if np.signbit(y) else 0)
    return codes, scs


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_nvfp4_matches_scalar_derivation(seed):
    x = synth.activation(seed, 6, 64).float().numpy()
    x[0, :16] = 0.0
    x[1, 16:32] *= 1e-3
    gs = float(np.float32(2688.0) / np.float32(np.abs(x).max()))
    want_codes, want_sc = _scalar_nvfp4(x, gs)
    codes, sc = quant.nvfp4_block_codes(x, gs)
    assert np.array_equal(sc, want_sc)
    assert np.array_equal(codes, want_codes)


def test_pack_order_and_layout_independence():
    x = synth.activation(5, 130, 96).float().numpy()
    gs = np.float32(2688.0) / np.float32(np.abs(x).max())
    codes, sc = quant.nvfp4_block_codes(x, gs)
    q, sf = quant.nvfp4_quantize(x, gs)
    assert q.shape == (130, 48)
    assert np.array_equal(q & 0xF, codes[:, 0::2]) and np.array_equal(q >> 4, codes[:, 1::2])
    assert np.array_equal(layout.unswizzle(sf, 130, 6), sc)
    assert sf.size == 256 * 8


def test_mxfp4_scale_is_smallest_power_of_two_covering_amax():
    x = synth.activation(7, 32, 256).float().numpy()
    x[0, :32] = 6.0 * 2.0 ** -3                     # amax exactly 6 * 2^e: lossless
    x[1, :32] = 0.0
    codes, sc = quant.mxfp4_block_codes(x)
    amax = np.abs(x.reshape(32, 8, 32)).max(axis=2)
    s = (amax / np.float32(6.0)).astype(np.float32)
    for (r, b), c in np.ndenumerate(sc):
        if s[r, b] == 0:
            assert c == 0
            continue
        ok = [e for e in range(255) if 2.0 ** (e - 127) >= float(s[r, b])]
        assert c == ok[0]
    assert sc[0, 0] == 127 - 3 and np.all(codes[0, :32] == 7)
    vals = formats.e2m1_decode(codes) * np.repeat(formats.ue8m0_decode(sc), 32, axis=1)
    # round-up scale: decoded magnitude never exceeds the block amax by more than one
    # e2m1 rounding step, and no element needs saturation beyond 6
    assert np.all(np.abs(x * np.repeat(np.exp2(127.0 - sc), 32, axis=1)) <= 6.0 * (1 + 2 ** -22))
    assert np.all(np.abs(vals) <= np.repeat(amax, 32, axis=1) * 1.3334 + 1e-30)


def test_mxfp4_grouped_blocks():
    counts = np.array([0, 1, 127, 128, 129, 5])
    ro = np.concatenate([[0], np.cumsum(counts)])
    x = synth.activation(9, int(ro[-1]), 64).float().numpy()
    q, sf = quant.mxfp4_quantize(x, ro)
    sfr = quant.expert_sf_rows(ro)
    assert list(sfr) == [0, 0, 128, 256, 384, 640, 768]
    assert sf.size == 768 * 4
    dq, dsf = quant.mxfp4_quantize(x)
    assert np.array_equal(q, dq)
    for e in range(len(counts)):
        r0, r1 = ro[e], ro[e + 1]
        if r1 == r0:
            continue
        _, blk = quant.mxfp4_quantize(x[r0:r1])
        assert np.array_equal(sf[sfr[e] * 4: sfr[e] * 4 + blk.size], blk)

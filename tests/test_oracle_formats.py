"""Pins for oracle/formats.py: decoders against library casts and the format table,
encoders against brute-force nearest-value search (ties to the even code)."""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _golden_e2m1():
    vals = {}
    with open(os.path.join(GOLD, "e2m1_values.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            c, v = line.split()
            vals[int(c, 16)] = float(v)
    return vals


def test_e2m1_decode_matches_spec_table():
    gold = _golden_e2m1()
    assert len(gold) == 16
    got = formats.e2m1_decode(np.arange(16))
    for c in range(16):
        assert got[c] == gold[c]
        assert np.signbit(got[c]) == np.signbit(gold[c]), c
    assert got.max() == 6.0  # FLOAT4_E2M1_MAX


def test_e4m3_decode_matches_torch_all_codes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = formats.e4m3_decode(np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.nanmax(got) == 448.0  # FLOAT8_E4M3_MAX


def test_ue8m0_decode_matches_torch_all_codes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    got = formats.ue8m0_decode(np.arange(256))
    assert np.isnan(ref[255]) and np.isnan(got[255])
    assert np.array_equal(ref[:255], got[:255])


def _nearest_even(grid_vals, grid_codes, x):
    """Brute force: the grid value nearest to x; on a tie the candidate whose code is even."""
    d = np.abs(grid_vals[None, :] - x[:, None])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    out = np.empty(len(x), dtype=np.int64)
    for i in range(len(x)):
        cs = grid_codes[cand[i]]
        even = cs[cs % 2 == 0]
        out[i] = even[0] if len(even) else cs[0]
    return out


def _f32_neighbourhood(points):
    """Each point, and the fp32 values one ulp either side of it."""
    p = np.asarray(points, dtype=np.float32)
    return np.unique(np.concatenate([p, np.nextafter(p, np.float32(np.inf)),
                                     np.nextafter(p, np.float32(0))]))


def _e4m3_sweep():
    grid = formats.e4m3_decode(np.arange(0x7F))           # all non-negative finite codes
    mids = (grid[1:] + grid[:-1]) / 2
    rng = np.random.default_rng(0)
    rand = np.exp2(rng.uniform(-12, 9, 20000)).astype(np.float32)
    return _f32_neighbourhood(np.concatenate([grid, mids, rand, [2.0 ** -10, 1e-30]]))


def test_e4m3_encode_brute_force_nearest():
    x = _e4m3_sweep()
    x = x[(x >= 0) & (x < 448)]
    codes = np.arange(0x7F)
    grid = formats.e4m3_decode(codes)
    want = _nearest_even(grid, codes, x.astype(np.float64))
    got = formats.e4m3_encode(x)
    assert np.array_equal(got, want)


def test_e4m3_encode_matches_torch_cast():
    x = _e4m3_sweep()
    x = x[(x >= 0) & (x < 464)]  # torch's cast is not saturating above 464
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(formats.e4m3_encode(x), ref)


def test_e4m3_encode_saturates():
    x = np.array([448.0, 448.5, 464.0, 480.0, 1e6, 3.4e38, np.inf], dtype=np.float32)
    assert np.all(formats.e4m3_encode(x) == 0x7E)
    assert formats.e4m3_encode(np.float32(0.0)) == 0


def test_e2m1_encode_brute_force_nearest():
    codes = np.arange(8)
    grid = formats.e2m1_decode(codes)
    mids = (grid[1:] + grid[:-1]) / 2
    rng = np.random.default_rng(1)
    pts = np.concatenate([grid, mids, rng.uniform(0, 8, 20000), [7.0, 8.0, 1e30, 1e-30]])
    mag = _f32_neighbourhood(pts)
    mag = mag[mag >= 0]
    want = _nearest_even(np.concatenate([grid, [6.0]]), np.concatenate([codes, [7]]), np.minimum(mag, 6.0))
    assert np.array_equal(formats.e2m1_encode(mag), want)
    # negative inputs: same magnitude code with the sign bit set
    assert np.array_equal(formats.e2m1_encode(-mag), want | 8)


def test_e2m1_sign_of_zero():
    assert formats.e2m1_encode(np.float32(-0.0)) == 0x8
    assert formats.e2m1_encode(np.float32(-0.1)) == 0x8
    assert formats.e2m1_encode(np.float32(0.0)) == 0x0
    assert formats.e2m1_encode(np.float32(0.25)) == 0x0   # tie -> even code 0
    assert formats.e2m1_encode(np.float32(-0.25)) == 0x8


def test_encoders_are_idempotent_on_codes():
    c2 = np.arange(16)
    assert np.array_equal(formats.e2m1_encode(formats.e2m1_decode(c2).astype(np.float32)), c2)
    c8 = np.arange(0x7F)
    assert np.array_equal(formats.e4m3_encode(formats.e4m3_decode(c8).astype(np.float32)), c8)


def test_ue8m0_round_up_brute_force():
    rng = np.random.default_rng(2)
    s = np.concatenate([np.exp2(rng.uniform(-130, 127, 5000)), np.exp2(np.arange(-126, 127)),
                        [0.0, 1e-45, 2.0 ** -127, 2.0 ** -127 * 1.5]]).astype(np.float32)
    s = _f32_neighbourhood(s)
    s = s[np.isfinite(s) & (s >= 0)]
    got = formats.ue8m0_encode_up(s)
    for v, c in zip(s[::7], got[::7]):
        fv = Fraction(float(v))
        cands = [k for k in range(255) if Fraction(2) ** (k - 127) >= fv]
        want = cands[0] if (cands and v != 0) else (0 if v == 0 else 254)
        assert c == want, (v, c, want)

"""Pins for oracle/gemm.py: exact integer GEMM, brute force with exact rationals on tiny
shapes (decoding through library casts and the permute construction, not the oracle's
own decoders), one-hot probes, alpha linearity and zero-scale blocks."""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import synth
from oracle import gemm, layout, quant

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _e2m1_table():
    vals = {}
    with open(os.path.join(GOLD, "e2m1_values.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            c, v = line.split()
            vals[int(c, 16)] = Fraction(float(v))
    return vals


def _random_operands(seed, rows, k):
    """Random packed codes and random finite e4m3 scales, as raw bytes."""
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 256, size=(rows, k // 2)).astype(np.uint8)
    sc = rng.integers(0, 0x7F, size=(rows, k // 16)).astype(np.uint8)   # finite, non-negative
    return q, layout.swizzle(sc), sc


def _brute_force(qa, sca, qb, scb, alpha, m, n, k):
    """Exact rationals; e4m3 via torch's cast, e2m1 via the spec table, row-major scales."""
    e2 = _e2m1_table()
    e4a = torch.from_numpy(sca).view(torch.float8_e4m3fn).double().numpy()
    e4b = torch.from_numpy(scb).view(torch.float8_e4m3fn).double().numpy()

    def nib(q, r, kk):
        byte = int(q[r, kk // 2])
        return byte & 0xF if kk % 2 == 0 else byte >> 4

    out = [[Fraction(0)] * n for _ in range(m)]
    for i in range(m):
        for j in range(n):
            s = Fraction(0)
            for kk in range(k):
                a = e2[nib(qa, i, kk)] * Fraction(float(e4a[i, kk // 16]))
                b = e2[nib(qb, j, kk)] * Fraction(float(e4b[j, kk // 16]))
                s += a * b
            out[i][j] = Fraction(float(np.float32(alpha))) * s
    return out


@pytest.mark.parametrize("m,n,k", [(3, 5, 32), (8, 8, 64), (1, 2, 96)])
def test_brute_force_tiny(m, n, k):
    qa, sfa, sca = _random_operands(m * 7 + k, m, k)
    qb, sfb, scb = _random_operands(n * 11 + k, n, k)
    alpha = 0.37
    want = _brute_force(qa, sca, qb, scb, alpha, m, n, k)
    got = gemm.nvfp4_gemm(qa, sfa, qb, sfb, alpha, m, n, k)
    for i in range(m):
        for j in range(n):
            assert Fraction(float(got[i, j])) == want[i][j] or \
                abs(float(got[i, j]) - float(want[i][j])) <= 1e-15 * abs(float(want[i][j]))


def _exact_int(q, sf, rows, k):
    """Dequantised values times 2^10 as exact int64 (e2m1 in halves, e4m3 in 2^-9 units)."""
    codes = quant.unpack_nibbles(q).astype(np.int64)
    half = np.array([0, 1, 2, 3, 4, 6, 8, 12], dtype=np.int64)      # e2m1 magnitude * 2
    a = np.where(codes & 8, -1, 1) * half[codes & 7]
    sc = layout.unswizzle(sf, rows, k // 16).astype(np.int64)
    e, mm = (sc >> 3) & 15, sc & 7
    units = np.where(e == 0, mm, (8 + mm) << np.maximum(e - 1, 0))   # e4m3 * 2^9
    return a * np.repeat(units, 16, axis=1)


def test_fp64_equals_exact_integer_gemm_pr1():
    """PR1 shapes: A 32x1024 ~N(0,1), B 1024x1024 ~N(0,0.02), quantised by the oracle."""
    m, n, k = 32, 1024, 1024
    xa = synth.activation(0, m, k, outliers=False).float().numpy()
    xb = synth.weight(0, n, k).float().numpy()
    gsa = np.float32(2688.0) / np.float32(np.abs(xa).max())
    gsb = np.float32(2688.0) / np.float32(np.abs(xb).max())
    qa, sfa = quant.nvfp4_quantize(xa, gsa)
    qb, sfb = quant.nvfp4_quantize(xb, gsb)
    ia, ib = _exact_int(qa, sfa, m, k), _exact_int(qb, sfb, n, k)
    exact = ia @ ib.T                                                 # int64, units of 2^-20
    assert np.abs(exact).max() < 2 ** 53
    got = gemm.nvfp4_gemm(qa, sfa, qb, sfb, 1.0, m, n, k)
    assert np.array_equal(got, exact.astype(np.float64) * 2.0 ** -20)


def test_one_hot_probes_pin_nibble_and_scale_placement():
    m, n, k = 4, 3, 128
    qb = np.full((n, k // 2), 0x22, dtype=np.uint8)                   # every b = 1.0
    scb = np.full((n, k // 16), 0x38, dtype=np.uint8)                 # scale 1.0
    sfb = layout.swizzle(scb)
    for (r, kk) in [(0, 0), (1, 1), (2, 17), (3, 126), (3, 127)]:
        qa = np.zeros((m, k // 2), dtype=np.uint8)
        qa[r, kk // 2] = 0x5 if kk % 2 == 0 else 0x50                 # value 3.0 at (r, kk)
        sca = np.full((m, k // 16), 0x38, dtype=np.uint8)
        sca[r, kk // 16] = 0x40                                       # scale 2.0 on its block
        R = gemm.nvfp4_gemm(qa, layout.swizzle(sca), qb, sfb, 1.0, m, n, k)
        want = np.zeros((m, n))
        want[r, :] = 6.0
        assert np.array_equal(R, want), (r, kk)


def test_alpha_linearity_and_zero_scale_blocks():
    m, n, k = 16, 24, 256
    qa, sfa, sca = _random_operands(1, m, k)
    qb, sfb, scb = _random_operands(2, n, k)
    r1 = gemm.nvfp4_gemm(qa, sfa, qb, sfb, 0.5, m, n, k)
    r2 = gemm.nvfp4_gemm(qa, sfa, qb, sfb, 1.0, m, n, k)
    assert np.array_equal(2 * r1, r2)
    sca0 = sca.copy()
    sca0[:, 3] = 0
    qa0 = qa.copy()
    qa0[:, 24:32] = 0                                                 # same block's data zeroed
    ra = gemm.nvfp4_gemm(qa, layout.swizzle(sca0), qb, sfb, 1.0, m, n, k)
    rb = gemm.nvfp4_gemm(qa0, sfa, qb, sfb, 1.0, m, n, k)
    assert np.array_equal(ra, rb)


def test_transposed_operand_is_caught():
    m, n, k = 8, 8, 64
    qa, sfa, _ = _random_operands(3, m, k)
    qb, sfb, _ = _random_operands(4, n, k)
    R = gemm.nvfp4_gemm(qa, sfa, qb, sfb, 1.0, m, n, k)
    Rt = gemm.nvfp4_gemm(qb, sfb, qa, sfa, 1.0, n, m, k)
    assert np.array_equal(R, Rt.T)
    assert not np.array_equal(R, Rt)


def test_ulp_and_rounding_helpers():
    assert gemm.ulp_bf16(1.0) == 2.0 ** -7
    assert gemm.ulp_bf16(3.0) == 2.0 ** -6
    assert gemm.ulp_bf16(-0.75) == 2.0 ** -8
    assert gemm.ulp_bf16(0.0) == 0.0
    x = np.random.default_rng(0).normal(size=1000) * 100
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(gemm.bf16_round(x), ref)


def test_grouped_equals_per_expert_dense():
    counts = np.array([3, 0, 130, 1])
    ro = np.concatenate([[0], np.cumsum(counts)])
    E, n, k = len(counts), 32, 64
    xa = synth.activation(1, int(ro[-1]), k).float().numpy()
    qa, sfa = quant.mxfp4_quantize(xa, ro)
    xb = synth.weight(1, n, k, experts=E).float().numpy()
    qb = np.stack([quant.mxfp4_quantize(xb[e])[0] for e in range(E)])
    sfb = np.stack([quant.mxfp4_quantize(xb[e])[1] for e in range(E)])
    out = gemm.mxfp4_grouped_gemm(qa, sfa, ro, qb, sfb, None, n, k)
    codes_a, sca = quant.mxfp4_block_codes(xa)
    from oracle import formats
    A = formats.e2m1_decode(codes_a) * np.repeat(formats.ue8m0_decode(sca), 32, axis=1)
    for e in range(E):
        cb, scb = quant.mxfp4_block_codes(xb[e])
        B = formats.e2m1_decode(cb) * np.repeat(formats.ue8m0_decode(scb), 32, axis=1)
        assert np.array_equal(out[e][2], A[ro[e]:ro[e + 1]] @ B.T)


def test_dequantize_matches_exact_rationals():
    """deq(q, sf)[r, k] = e2m1(nibble) * e4m3(scale of block k/16), decoded through the spec
    table and torch's e4m3 cast with the row-major scale matrix (not the oracle's decoders)."""
    rows, k = 5, 64
    q, sf, sc = _random_operands(9, rows, k)
    got = gemm.dequantize(q, sf, rows, k, 16, "e4m3")
    e2 = _e2m1_table()
    e4 = torch.from_numpy(sc).view(torch.float8_e4m3fn).double().numpy()
    for r in range(rows):
        for kk in range(k):
            byte = int(q[r, kk // 2])
            nib = byte & 0xF if kk % 2 == 0 else byte >> 4
            assert Fraction(float(got[r, kk])) == e2[nib] * Fraction(float(e4[r, kk // 16])), (r, kk)


def test_abs_product_sum_and_tolerance_by_hand():
    """sum_k |alpha a b| by explicit loops in exact rationals, and the acceptance bound on
    hand-worked values: ulp_bf16(3) = 2^-6, so |R| = 3 with abs-sum 100 allows 2^-6 + 1e-3."""
    rng = np.random.default_rng(5)
    A = rng.normal(size=(3, 7))
    B = rng.normal(size=(4, 7))
    alpha = -0.625
    got = gemm.abs_product_sum(A, B, alpha)
    for i in range(3):
        for j in range(4):
            s = sum(abs(Fraction(alpha) * Fraction(A[i, kk]) * Fraction(B[j, kk])) for kk in range(7))
            assert abs(Fraction(float(got[i, j])) - s) <= Fraction(1, 10 ** 12) * s
    tol = gemm.tolerance(np.array([3.0, -3.0, 0.0, 1.0]), np.array([100.0, 100.0, 0.0, 0.0]))
    assert np.array_equal(tol, np.array([2.0 ** -6 + 1e-3, 2.0 ** -6 + 1e-3, 0.0, 2.0 ** -7]))

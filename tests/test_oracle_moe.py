"""Pins for oracle/moe.py: the fp32 exp against fp64 exp, silu limits, bf16 rounding against
torch, the routing sort against numpy's stable argsort, per-expert quantisation against the
dense quantiser, combine against fp64 sums and hand-worked values, the grouped GEMM against the
dense oracle GEMM."""
import numpy as np
import pytest
import torch

from oracle import gemm as ogemm
from oracle import layout, moe
from oracle import quant as oquant

F32 = np.float32


def _ulp32(x):
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 2.0 ** (e - 23)


def test_exp_close_to_fp64_exp():
    rng = np.random.default_rng(0)
    t = np.concatenate([np.linspace(-87, 88, 200001), rng.uniform(-87, 88, 200000),
                        rng.uniform(-1, 1, 100000)]).astype(F32)
    e = moe.exp_f32(t).astype(np.float64)
    ref = np.exp(t.astype(np.float64))
    err_ulp = np.abs(e - ref) / _ulp32(ref)
    assert err_ulp.max() <= 4.0, err_ulp.max()
    assert moe.exp_f32(F32(0.0)) == F32(1.0)
    assert np.isinf(moe.exp_f32(F32(88.5))) and moe.exp_f32(F32(-87.5)) == 0.0


def test_exp_steps_are_the_documented_ones():
    # r = 0 exactly at t = n*ln2 split points: exp(t) = 2^n * p(r) with p(0) = 1
    for n in (-20, -1, 0, 1, 5, 40):
        t = F32(np.float32(n) * moe.LN2_HI)   # exact product (16-bit constant)
        e = moe.exp_f32(t)
        r = (t - F32(n) * moe.LN2_HI) - F32(n) * moe.LN2_LO
        p = moe.TAYLOR[0]
        for c in moe.TAYLOR[1:]:
            p = F32(F32(r * p) + c)
        assert e == F32(p * F32(2.0 ** n))


def test_silu_limits_and_fp64():
    g = np.linspace(-20, 20, 40001).astype(F32)
    s = moe.silu_f32(g).astype(np.float64)
    ref = g.astype(np.float64) / (1.0 + np.exp(-g.astype(np.float64)))
    assert np.all(np.abs(s - ref) <= 8 * _ulp32(ref) + 1e-38)
    assert moe.silu_f32(F32(0.0)) == 0.0
    assert moe.silu_f32(F32(30.0)) == F32(30.0)
    assert np.all(moe.silu_f32(g[g < 0]) <= 0)
    assert moe.silu_f32(F32(-100.0)) == 0.0 and np.signbit(moe.silu_f32(F32(-100.0)))


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(1).standard_normal(100000).astype(F32) * F32(3.0)
    x[:5] = [1.00390625, 1.01171875, -2.0078125, 0.0, 65504.0]   # ties to even among them
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(moe.bf16_rne(x), want)


def test_silu_and_mul_is_bf16_of_fp32_product():
    rng = np.random.default_rng(2)
    x = torch.from_numpy(rng.standard_normal((7, 64)).astype(F32)).to(torch.bfloat16)
    h = moe.silu_and_mul(x)
    xf = x.float().numpy()
    want = moe.bf16_rne(moe.silu_f32(xf[:, :32]) * xf[:, 32:])
    assert np.array_equal(h, want)
    ref = xf[:, :32].astype(np.float64) / (1 + np.exp(-xf[:, :32].astype(np.float64))) * xf[:, 32:]
    assert np.all(np.abs(h - ref) <= 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7) + 1e-30)


@pytest.mark.parametrize("T,topk,E", [(1, 1, 1), (5, 2, 4), (64, 8, 16), (300, 8, 128)])
def test_sort_matches_stable_argsort(T, topk, E):
    rng = np.random.default_rng(T + E)
    ids = np.stack([rng.permutation(E)[:topk] for _ in range(T)]) if topk <= E else rng.integers(0, E, (T, topk))
    ro, src, pos = moe.sort_by_expert(ids, E)
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")
    assert np.array_equal(src, order // topk)
    assert np.array_equal(ro, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    inv = np.empty_like(order)
    inv[order] = np.arange(order.size)
    assert np.array_equal(pos.reshape(-1), inv)
    for e in range(E):   # rows of expert e carry expert e
        assert np.all(flat[order[ro[e]:ro[e + 1]]] == e)


def test_sort_edge_cases():
    ro, src, pos = moe.sort_by_expert(np.zeros((6, 2), dtype=np.int64), 3)   # everything to expert 0
    assert list(ro) == [0, 12, 12, 12] and list(src) == [0, 0, 1, 1, 2, 2, 3, 3, 4, 4, 5, 5]
    with pytest.raises(ValueError):
        moe.sort_by_expert(np.array([[3]]), 3)


def test_expert_quantisation_equals_dense_per_expert():
    rng = np.random.default_rng(3)
    counts = [0, 5, 130, 1, 0, 64]
    ro = np.concatenate([[0], np.cumsum(counts)])
    T, K = int(ro[-1]), 96
    x = torch.from_numpy(rng.standard_normal((T, K)).astype(F32)).to(torch.bfloat16)
    gs = np.array([1.0, 2.0, 300.0, 0.5, 7.0, 1024.0], dtype=F32)
    q, sf = moe.nvfp4_quantize_experts(x, ro, gs)
    sfr = oquant.expert_sf_rows(ro)
    cp = layout.round_up(K // 16, 4)
    assert sf.size == int(sfr[-1]) * cp <= moe.grouped_sf_bytes(T, len(counts), K)
    for e in range(len(counts)):
        r0, r1 = int(ro[e]), int(ro[e + 1])
        if r1 == r0:
            continue
        qe, sfe = oquant.nvfp4_quantize(x[r0:r1], gs[e])
        assert np.array_equal(q[r0:r1], qe)
        assert np.array_equal(sf[int(sfr[e]) * cp: int(sfr[e]) * cp + sfe.size], sfe)


def test_combine_hand_worked_and_identity():
    y = np.array([[1.0, 2.0], [4.0, -8.0], [0.5, 0.25]], dtype=F32)
    pos = np.array([[1, 2], [0, 1]])
    w = np.array([[0.5, 2.0], [1.0, 0.25]], dtype=F32)
    out = moe.combine(y, pos, w)
    assert np.array_equal(out, np.array([[0.5 * 4 + 2 * 0.5, 0.5 * -8 + 2 * 0.25], [1 + 1, 2 - 2]], dtype=F32))
    # top-1 with unit weights is a permutation
    rng = np.random.default_rng(4)
    yy = moe.bf16_rne(rng.standard_normal((10, 16)).astype(F32))
    p1 = rng.permutation(10).reshape(10, 1)
    assert np.array_equal(moe.combine(yy, p1, np.ones((10, 1), F32)), yy[p1[:, 0]])


def test_combine_close_to_fp64():
    rng = np.random.default_rng(5)
    y = moe.bf16_rne(rng.standard_normal((64, 32)).astype(F32))
    pos = np.stack([rng.permutation(64)[:8] for _ in range(20)])
    w = rng.uniform(0, 1, (20, 8)).astype(F32)
    out = moe.combine(y, pos, w)
    ref = np.einsum("tj,tjh->th", w.astype(np.float64), y[pos].astype(np.float64))
    bound = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7) + 8 * 2.0 ** -23 * np.einsum(
        "tj,tjh->th", w.astype(np.float64), np.abs(y[pos]).astype(np.float64))
    assert np.all(np.abs(out - ref) <= bound)


def test_grouped_gemm_equals_dense_oracle_per_expert():
    rng = np.random.default_rng(6)
    counts = [3, 0, 40]
    ro = np.concatenate([[0], np.cumsum(counts)])
    T, N, K, E = int(ro[-1]), 64, 128, 3
    x = torch.from_numpy(rng.standard_normal((T, K)).astype(F32)).to(torch.bfloat16)
    gsa = np.array([100.0, 1.0, 50.0], dtype=F32)
    qa, sfa = moe.nvfp4_quantize_experts(x, ro, gsa)
    qb, sfb, gsb = [], [], []
    for e in range(E):
        w = torch.from_numpy(rng.standard_normal((N, K)).astype(F32) * F32(0.02)).to(torch.bfloat16)
        g = F32(2688.0) / F32(w.float().abs().max().item())
        q_, s_ = oquant.nvfp4_quantize(w, g)
        qb.append(q_), sfb.append(s_), gsb.append(g)
    alpha = F32(1.0) / (gsa * np.array(gsb, dtype=F32))
    res = moe.nvfp4_grouped_gemm(qa, sfa, ro, np.stack(qb), np.stack(sfb), alpha, N, K)
    sfr = oquant.expert_sf_rows(ro)
    cp = layout.round_up(K // 16, 4)
    for e in range(E):
        r0, r1 = int(ro[e]), int(ro[e + 1])
        if r1 == r0:
            assert res[e][2].shape == (0, N)
            continue
        rp = layout.round_up(r1 - r0, 128)
        seg = sfa[int(sfr[e]) * cp: int(sfr[e]) * cp + rp * cp]
        want = ogemm.nvfp4_gemm(qa[r0:r1], seg, qb[e], sfb[e], alpha[e], r1 - r0, N, K)
        assert np.array_equal(res[e][2], want)

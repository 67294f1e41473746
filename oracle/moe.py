"""The MoE steps around the grouped GEMMs, NVFP4 flavour (test infrastructure only).

Sources: vLLM fork compare view "add pdl", ops.h / torch_bindings.cpp (the op names
scaled_fp4_experts_quant, silu_and_mul_scaled_fp4_experts_quant with the arguments
input_offset_by_experts and output_scale_offset_by_experts, and cutlass_fp4_group_mm);
vLLM PR 51158 "Enable CUTLASS MXFP4 W4A4 MoE on SM12x", "Changes" (experts quantise, grouped
GEMM, CutlassExpertsMxfp4 around them).  The pages give names and arguments only; the readings
taken here:

* routing order: rows are grouped by expert; inside an expert, (token, slot) pairs keep their
  row-major order (a stable counting sort of the flattened top-k ids);
* gather: permuted row r is token src[r];
* per-expert NVFP4 quantisation: expert e's rows use its own fp32 global scale gs[e]; its scales
  form their own zero-padded 128-row block (as the MXFP4 grouped path);
* SiLU-and-mul: input [T, 2I] = [gate | up]; h = bf16(silu(gate) * up) with silu(g) =
  g * (1 / (1 + exp(-g))) in fp32, exp as defined below; h is then quantised as above, so the
  fused kernel equals "silu_and_mul to bf16, then quantise";
* grouped GEMM: D_e = alpha[e] * deq(A_e) deq(B_e)^T, one fp32 alpha per expert;
* combine: out[t] = bf16(sum_j w[t, j] * y[pos[t, j]]) in fp32, j = 0 .. topk-1 in order, each
  product and sum rounded (no fused multiply-add), the first term w[t,0]*y[pos[t,0]].

exp (for the silu): Cody and Waite's range reduction followed by a Taylor polynomial, every
operation in fp32 with round-to-nearest-even and nothing fused, so that two implementations
following the same steps agree bit for bit:
  t  = -g;  t > 88 -> exp = +inf;  t < -87 -> exp = 0;
  n  = rint(t * LOG2E)                       (ties to even)
  r  = (t - n * LN2_HI) - n * LN2_LO          (LN2_HI has 16 significant bits: n * LN2_HI exact)
  p  = 1 + r*(1 + r*(1/2 + r*(1/6 + r*(1/24 + r*(1/120 + r*(1/720 + r*(1/5040)))))))
  exp = p * 2^n                               (exact scaling, -126 <= n <= 127 here)
with LOG2E = fp32(1/ln 2), LN2_HI = 0.693145751953125, LN2_LO = fp32(ln 2 - LN2_HI) and the
Taylor coefficients fp32(1/k!).  The truncation error of the degree-7 polynomial on
|r| <= ln2/2 is below 6e-9 relative; with the roundings the result stays within a few fp32 ulps
of exp (pinned in tests).
"""
from __future__ import annotations

import numpy as np

from . import formats, layout, quant

F32 = np.float32

LOG2E = F32(1.4426950408889634)
LN2_HI = F32(0.693145751953125)
LN2_LO = F32(0.6931471805599453 - 0.693145751953125)
TAYLOR = [F32(1.0 / v) for v in (5040.0, 720.0, 120.0, 24.0, 6.0, 2.0, 1.0, 1.0)]  # 1/7! .. 1/0!


def exp_f32(t) -> np.ndarray:
    """exp(t) in fp32 by the steps in the module docstring (elementwise)."""
    t = np.asarray(t, dtype=F32)
    big, small = t > F32(88.0), t < F32(-87.0)
    tt = np.where(big | small, F32(0.0), t).astype(F32)
    n = np.rint(tt * LOG2E).astype(F32)
    r = ((tt - n * LN2_HI).astype(F32) - (n * LN2_LO).astype(F32)).astype(F32)
    p = TAYLOR[0]
    for c in TAYLOR[1:]:
        p = (r * p).astype(F32)
        p = (p + c).astype(F32)
    e = (p * np.exp2(n.astype(np.float64)).astype(F32)).astype(F32)
    return np.where(big, F32(np.inf), np.where(small, F32(0.0), e)).astype(F32)


def silu_f32(g) -> np.ndarray:
    """silu(g) = g * (1 / (1 + exp(-g))) in fp32."""
    g = np.asarray(g, dtype=F32)
    e = exp_f32(-g)
    with np.errstate(over="ignore"):
        sig = (F32(1.0) / (F32(1.0) + e).astype(F32)).astype(F32)
    return (g * sig).astype(F32)


def bf16_rne(x) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even), returned as fp32 values."""
    f = np.asarray(x, dtype=F32).view(np.uint32).astype(np.uint64)
    lsb = (f >> 16) & 1
    f = (f + 0x7FFF + lsb) >> 16 << 16
    return f.astype(np.uint32).view(F32)


def silu_and_mul(x) -> np.ndarray:
    """[T, 2I] bf16 values -> h [T, I] = bf16(silu(gate) * up), gate = x[:, :I], up = x[:, I:]."""
    x = np.asarray(x.detach().cpu().float().numpy() if hasattr(x, "detach") else x, dtype=F32)
    i = x.shape[1] // 2
    return bf16_rne((silu_f32(x[:, :i]) * x[:, i:]).astype(F32))


def sort_by_expert(topk_ids, num_experts: int):
    """Stable counting sort of the flattened [T, topk] expert ids.

    Returns (row_offsets [E+1] int64, src [T*topk] int64 = token of each permuted row,
    pos [T, topk] int64 = permuted row of each (token, slot))."""
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, topk = ids.shape
    flat = ids.reshape(-1)
    if np.any(flat < 0) or np.any(flat >= num_experts):
        raise ValueError("expert id out of range")
    counts = np.zeros(num_experts, dtype=np.int64)
    for v in flat:
        counts[v] += 1
    row_offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    nxt = row_offsets[:-1].copy()
    src = np.empty(T * topk, dtype=np.int64)
    pos = np.empty(T * topk, dtype=np.int64)
    for idx, v in enumerate(flat):          # row-major (token, slot) order: stable
        pos[idx] = nxt[v]
        src[nxt[v]] = idx // topk
        nxt[v] += 1
    return row_offsets, src, pos.reshape(T, topk)


def nvfp4_quantize_experts(x, row_offsets, gs) -> tuple[np.ndarray, np.ndarray]:
    """bf16 [T, K] rows grouped by expert -> (packed e2m1 [T, K/2], grouped e4m3 scales).
    Expert e's rows use global scale gs[e]; its scales form their own 128-row block starting at
    scale row sum_{j<e} round_up(M_j, 128) of a round_up(K/16, 4)-column swizzled matrix."""
    x = quant._as_f32_matrix(x)
    t, k = x.shape
    ro = np.asarray(row_offsets, dtype=np.int64)
    if ro[0] != 0 or ro[-1] != t:
        raise ValueError("row offsets must start at 0 and end at T")
    gs = np.asarray(gs, dtype=F32)
    sfr = quant.expert_sf_rows(ro)
    cp = layout.round_up(k // 16, 4)
    codes = np.zeros((t, k), dtype=np.uint8)
    sf = np.zeros(int(sfr[-1]) * cp, dtype=np.uint8)
    for e in range(len(ro) - 1):
        r0, r1 = int(ro[e]), int(ro[e + 1])
        if r1 == r0:
            continue
        c, sc = quant.nvfp4_block_codes(x[r0:r1], gs[e])
        codes[r0:r1] = c
        blk = layout.swizzle(sc)
        base = int(sfr[e]) * cp
        sf[base: base + blk.size] = blk
    return quant.pack_nibbles(codes), sf


def grouped_sf_bytes(total_rows: int, num_experts: int, k: int, vec: int = 16) -> int:
    """Upper bound of the grouped scale buffer: (round_up(T,128) + 128 E) * round_up(K/vec, 4)."""
    return (layout.round_up(total_rows, 128) + 128 * num_experts) * layout.round_up(k // vec, 4)


def combine(y, pos, w) -> np.ndarray:
    """out[t] = bf16(sum_j w[t,j] * y[pos[t,j]]) with fp32 products and sums in slot order."""
    y = np.asarray(y.detach().cpu().float().numpy() if hasattr(y, "detach") else y, dtype=F32)
    pos = np.asarray(pos, dtype=np.int64)
    w = np.asarray(w, dtype=F32)
    T, topk = pos.shape
    acc = (w[:, 0:1] * y[pos[:, 0]]).astype(F32)
    for j in range(1, topk):
        acc = (acc + (w[:, j:j + 1] * y[pos[:, j]]).astype(F32)).astype(F32)
    return bf16_rne(acc)


def nvfp4_grouped_gemm(a, sfa, row_offsets, b, sfb, alpha, n: int, k: int, experts=None) -> dict:
    """Per-expert R_e = alpha[e] * deq(A_e) @ deq(B_e)^T in fp64 (NVFP4 operands).
    sfa: grouped scales as nvfp4_quantize_experts lays them out; b: [E, n, k/2];
    sfb: [E, round_up(n,128) * round_up(k/16,4)].  Returns {e: (A_e, B_e, R_e)}."""
    from . import gemm as ogemm
    ro = np.asarray(row_offsets, dtype=np.int64)
    E = len(ro) - 1
    a = np.asarray(a, dtype=np.uint8)
    b = np.asarray(b, dtype=np.uint8).reshape(E, n, k // 2)
    sfb = np.asarray(sfb, dtype=np.uint8).reshape(E, -1)
    sfa = np.asarray(sfa, dtype=np.uint8).reshape(-1)
    alpha = np.asarray(alpha, dtype=F32)
    sfr = quant.expert_sf_rows(ro)
    cp = layout.round_up(k // 16, 4)
    out = {}
    for e in (range(E) if experts is None else experts):
        r0, r1 = int(ro[e]), int(ro[e + 1])
        rows = r1 - r0
        Be = ogemm.dequantize(b[e], sfb[e], n, k, 16, "e4m3")
        if rows == 0:
            out[e] = (np.zeros((0, k)), Be, np.zeros((0, n)))
            continue
        rp = layout.round_up(rows, 128)
        seg = sfa[int(sfr[e]) * cp: int(sfr[e]) * cp + rp * cp]
        Ae = ogemm.dequantize(a[r0:r1], seg, rows, k, 16, "e4m3")
        out[e] = (Ae, Be, np.float64(alpha[e]) * (Ae @ Be.T))
    return out

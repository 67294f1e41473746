"""Block-scaled FP4 GEMM in fp64, and the tolerance the GPU result is held to.

Definition ([vLLM-SM103] "SM103 Entry Point": A is [M, K/2] packed e2m1,
B is [N, K/2] packed e2m1 stored K-major, scale_a / scale_b are e4m3 in the
128x4 layout, alpha is one fp32, D is bf16 [M, N]; [FI-4865] "2. Alpha
epilogue bug": alpha multiplies the fp32 accumulator before the single
conversion to the output type):

    R[m, n] = alpha * sum_k a(m, k) * b(n, k),
    a(m, k) = e2m1(A nibble (m, k)) * e4m3(scale_a[m, k // 16]),

computed here in fp64 with a library matmul over the dequantised operands.
Every dequantised NVFP4 value is an integer multiple of 2^-10, so the fp64
sum is exact whenever its magnitude stays below 2^43 (pinned against an exact
integer GEMM in the tests).

The MXFP4 grouped GEMM ([vLLM-51158], "Changes": grouped GEMM over experts)
is the same per expert with ue8m0 scales per 32 and alpha defaulting to 1.

Acceptance bound per element:
    |D - R| <= ulp_bf16(|R|) + 1e-5 * sum_k |alpha * a(m,k) * b(n,k)|,
ulp_bf16(x) = 2^(floor(log2 x) - 7), ulp_bf16(0) = 0.
"""
from __future__ import annotations

import numpy as np

from . import formats, layout
from .quant import expert_sf_rows, unpack_nibbles


def dequantize(q, sf, rows: int, k: int, vec: int, scale_kind: str) -> np.ndarray:
    """Packed FP4 bytes [rows, k/2] + swizzled scale bytes -> fp64 values [rows, k]."""
    q = np.asarray(q, dtype=np.uint8).reshape(rows, k // 2)
    vals = formats.e2m1_decode(unpack_nibbles(q))
    sc = layout.unswizzle(np.asarray(sf, dtype=np.uint8).reshape(-1), rows, k // vec)
    dec = formats.e4m3_decode if scale_kind == "e4m3" else formats.ue8m0_decode
    scales = np.repeat(dec(sc), vec, axis=1)
    return vals * scales


def nvfp4_gemm(a, sfa, b, sfb, alpha, m: int, n: int, k: int) -> np.ndarray:
    """R = alpha * deq(A) @ deq(B)^T in fp64, shape [m, n]."""
    A = dequantize(a, sfa, m, k, 16, "e4m3")
    B = dequantize(b, sfb, n, k, 16, "e4m3")
    return np.float64(np.float32(alpha)) * (A @ B.T)


def abs_product_sum(A: np.ndarray, B: np.ndarray, alpha) -> np.ndarray:
    """sum_k |alpha * a(m,k) * b(n,k)| for dequantised operands."""
    return abs(np.float64(np.float32(alpha))) * (np.abs(A) @ np.abs(B).T)


def ulp_bf16(x) -> np.ndarray:
    """bf16 unit in the last place of |x|: 2^(floor(log2|x|) - 7); 0 at 0."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(x)  # x = f * 2^e, f in [0.5, 1) -> floor(log2 x) = e - 1
    return np.where(x == 0, 0.0, np.exp2(e - 1.0 - 7.0))


def tolerance(R: np.ndarray, abs_sum: np.ndarray) -> np.ndarray:
    """Per-element acceptance bound: one bf16 ulp of |R| plus 1e-5 * sum_k |alpha a b|."""
    return ulp_bf16(R) + 1e-5 * abs_sum


def bf16_round(R: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 value (RNE, via fp32) as fp64; what an exact kernel would store."""
    f = np.asarray(R, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (f >> 16) & 1
    f = (f + 0x7FFF + lsb) >> 16 << 16
    return f.astype(np.uint32).view(np.float32).astype(np.float64)


def mxfp4_grouped_gemm(a, sfa, row_offsets, b, sfb, alpha, n: int, k: int,
                       experts=None) -> dict:
    """Per-expert R_e = alpha * deq(A_e) @ deq(B_e)^T in fp64.

    a: [T, k/2] bytes; sfa: grouped scales as mxfp4_quantize(..., row_offsets) lays them out;
    b: [E, n, k/2] bytes; sfb: [E, round_up(n,128) * round_up(k/32,4)] swizzled ue8m0 bytes.
    Returns {e: (A_e, B_e, R_e)} for the experts asked for (all by default).
    """
    ro = np.asarray(row_offsets, dtype=np.int64)
    E = len(ro) - 1
    a = np.asarray(a, dtype=np.uint8)
    b = np.asarray(b, dtype=np.uint8).reshape(E, n, k // 2)
    sfb = np.asarray(sfb, dtype=np.uint8).reshape(E, -1)
    sfa = np.asarray(sfa, dtype=np.uint8).reshape(-1)
    sfr = expert_sf_rows(ro)
    cp = layout.round_up(k // 32, 4)
    al = np.float64(1.0 if alpha is None else np.float32(alpha))
    out = {}
    for e in (range(E) if experts is None else experts):
        r0, r1 = int(ro[e]), int(ro[e + 1])
        rows = r1 - r0
        Be = dequantize(b[e], sfb[e], n, k, 32, "ue8m0")
        if rows == 0:
            out[e] = (np.zeros((0, k)), Be, np.zeros((0, n)))
            continue
        rp = layout.round_up(rows, 128)
        seg = sfa[int(sfr[e]) * cp: int(sfr[e]) * cp + rp * cp]
        Ae = dequantize(a[r0:r1], seg, rows, k, 32, "ue8m0")
        out[e] = (Ae, Be, al * (Ae @ Be.T))
    return out

"""Block quantisers: bf16 -> NVFP4 (e2m1 + e4m3 per 16) and bf16 -> MXFP4 (e2m1 + ue8m0 per 32).

NVFP4 follows the structure of [vLLM-SM103] nvfp4_quant_kernels.cu, "SM103
(B300) activation quantization kernel": one fp32 global scale for the tensor,
one scale per 16 consecutive K-elements of a row, packed e2m1 output, scales
written into the 128x4 swizzled layout, and padded scale rows and columns
quantised from zero input (so their scale bytes are 0x00).  The global scale
is defined in [vLLM-SM103] test_nvfp4_quant.py as
FLOAT8_E4M3_MAX * FLOAT4_E2M1_MAX / amax = 2688 / amax; it is an input here.

The arithmetic inside a block is not on the pages.  Reading (fp32, every
operation rounded to nearest even, nothing fused):
  1. amax = max |x_i| over the 16 values (exact);
  2. s = (gs * amax) / 6;
  3. sc = e4m3(s) (RNE, saturating), sd = its value;
  4. inv = gs / sd, or 0 when sd == 0;
  5. code_i = e2m1(x_i * inv) (RNE, saturating, sign kept);
  6. element 2t goes in the low nibble of byte t, element 2t+1 in the high one.

MXFP4 ("e2m1 data with e8m0 scale per 32 K-elements", [vLLM-51158] and the
grouped MoE workload) reading: no global scale; s = amax / 6 in fp32; the
scale is the smallest power of two >= s (round up, so no element clips beyond
the rounding of s), code clamped to [0, 254]; inv = 2^(127 - code) exactly;
code_i = e2m1(x_i * inv).  For grouped (MoE) input the rows of expert e are
rows row_offsets[e] .. row_offsets[e+1]-1, and its scale rows start at scale
row sum_{j<e} round_up(M_j, 128): every expert's scales form their own
128-row-padded block.
"""
from __future__ import annotations

import numpy as np

from . import formats, layout

F32 = np.float32


def _as_f32_matrix(x) -> np.ndarray:
    """Accept a torch bf16 tensor or an array of bf16-representable values; return fp32 [M, K]."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").float().numpy()
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    if x.ndim != 2:
        raise ValueError("expected a 2-D matrix")
    if not np.all(np.isfinite(x)):
        raise ValueError("inputs must be finite")
    return x


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """4-bit codes [M, K] -> bytes [M, K/2]: even element in the low nibble, odd in the high one."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] & 0xF) | ((codes[:, 1::2] & 0xF) << 4)


def unpack_nibbles(q: np.ndarray) -> np.ndarray:
    """Bytes [M, K/2] -> 4-bit codes [M, K] (inverse of pack_nibbles)."""
    q = np.asarray(q, dtype=np.uint8)
    out = np.empty((q.shape[0], q.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = q & 0xF
    out[:, 1::2] = q >> 4
    return out


def nvfp4_block_codes(x: np.ndarray, gs) -> tuple[np.ndarray, np.ndarray]:
    """Per-16 block quantisation in row-major form: (e2m1 codes [M, K], e4m3 scale codes [M, K/16])."""
    x = _as_f32_matrix(x)
    m, k = x.shape
    if k % 16:
        raise ValueError("K must be a multiple of 16")
    gs = F32(gs)
    if not (np.isfinite(gs) and gs > 0):
        raise ValueError("global scale must be a positive finite fp32")
    blocks = x.reshape(m, k // 16, 16)
    amax = np.max(np.abs(blocks), axis=2)                     # step 1
    s = (gs * amax) / F32(6.0)                                # step 2
    sc = formats.e4m3_encode(s)                               # step 3
    sd = formats.e4m3_decode(sc).astype(F32)
    safe = np.where(sd == 0, F32(1.0), sd)
    inv = np.where(sd == 0, F32(0.0), gs / safe).astype(F32)  # step 4
    y = blocks * inv[:, :, None]                              # step 5 (fp32 multiply)
    codes = formats.e2m1_encode(y).reshape(m, k)
    return codes, sc


def nvfp4_quantize(x, gs) -> tuple[np.ndarray, np.ndarray]:
    """bf16 [M, K] -> (packed e2m1 bytes [M, K/2], swizzled e4m3 scale bytes [Rp*Cp])."""
    codes, sc = nvfp4_block_codes(x, gs)
    return pack_nibbles(codes), layout.swizzle(sc)


def mxfp4_block_codes(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Per-32 block quantisation: (e2m1 codes [M, K], ue8m0 scale codes [M, K/32])."""
    x = _as_f32_matrix(x)
    m, k = x.shape
    if k % 32:
        raise ValueError("K must be a multiple of 32")
    blocks = x.reshape(m, k // 32, 32)
    amax = np.max(np.abs(blocks), axis=2)
    s = amax / F32(6.0)
    sc = formats.ue8m0_encode_up(s)
    inv = np.exp2(127.0 - sc.astype(np.float64)).astype(F32)  # exact power of two
    y = blocks * inv[:, :, None]
    codes = formats.e2m1_encode(y).reshape(m, k)
    return codes, sc


def expert_sf_rows(row_offsets) -> np.ndarray:
    """Scale-row start of every expert (length E+1): prefix sums of round_up(M_e, 128)."""
    ro = np.asarray(row_offsets, dtype=np.int64)
    counts = np.diff(ro)
    if np.any(counts < 0):
        raise ValueError("row offsets must be non-decreasing")
    padded = (counts + 127) // 128 * 128
    return np.concatenate([[0], np.cumsum(padded)]).astype(np.int64)


def mxfp4_quantize(x, row_offsets=None) -> tuple[np.ndarray, np.ndarray]:
    """bf16 [T, K] -> (packed e2m1 bytes [T, K/2], ue8m0 scales).

    Without ``row_offsets`` the scales are one swizzled [round_up(T,128), round_up(K/32,4)]
    block.  With ``row_offsets`` (E+1 non-decreasing row indices, last = T) each expert's
    scales are their own zero-padded block starting at scale row expert_sf_rows()[e].
    """
    codes, sc = mxfp4_block_codes(x)
    t, k = codes.shape
    q = pack_nibbles(codes)
    if row_offsets is None:
        return q, layout.swizzle(sc)
    ro = np.asarray(row_offsets, dtype=np.int64)
    if ro[0] != 0 or ro[-1] != t:
        raise ValueError("row offsets must start at 0 and end at T")
    sfr = expert_sf_rows(ro)
    cp = layout.round_up(k // 32, 4)
    sf = np.zeros(int(sfr[-1]) * cp, dtype=np.uint8)
    for e in range(len(ro) - 1):
        r0, r1 = int(ro[e]), int(ro[e + 1])
        if r1 == r0:
            continue
        blk = layout.swizzle(sc[r0:r1])
        base = int(sfr[e]) * cp
        sf[base: base + blk.size] = blk
    return q, sf

"""Element and scale formats: decoders and round-to-nearest-even encoders.

Formats (the pages name them; the bit layouts are the OCP Microscaling
Formats v1.0 definitions):

* e2m1 (FP4 data): 1 sign, 2 exponent bits (bias 1), 1 mantissa bit, no
  inf/NaN.  Largest magnitude 6 ([vLLM-SM103] test_nvfp4_quant.py uses
  FLOAT4_E2M1_MAX = 6 for the global scale).
* e4m3fn (NVFP4 block scale, "float8_e4m3fn" in the GEMM entry's SF dtype):
  1 sign, 4 exponent bits (bias 7), 3 mantissa bits; S.1111.111 is NaN, no
  inf; largest finite 448 (FLOAT8_E4M3_MAX in the same test).
* ue8m0 (MXFP4 block scale, "e8m0 scale per 32"): 8-bit biased exponent,
  value 2^(c-127); 0xFF is NaN.

Encoders (fp32 -> code).  The pages do not spell them out.  Reading: round to
nearest, ties to even, saturating to the largest finite value (what the
hardware ``.rn.satfinite`` conversions do); e2m1 keeps the sign of the
rounded value, so a negative input that rounds to zero gives code 0x8.
"""
from __future__ import annotations

import numpy as np


def e2m1_decode(codes) -> np.ndarray:
    """Value of each 4-bit e2m1 code (fp64), from its sign/exponent/mantissa fields."""
    c = np.asarray(codes, dtype=np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = c & 0x1
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e - 1.0))
    return sign * mag


def e4m3_decode(codes) -> np.ndarray:
    """Value of each e4m3fn byte (fp64); S.1111.111 decodes to NaN."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def ue8m0_decode(codes) -> np.ndarray:
    """Value of each ue8m0 byte (fp64): 2^(c-127), 0xFF is NaN."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    v = np.exp2(c - 127.0)
    return np.where(c == 255, np.nan, v)


def e4m3_encode(x) -> np.ndarray:
    """Non-negative fp32 scale -> e4m3fn code (uint8), RNE, saturating at 448 (0x7E).

    Subnormal range (x < 2^-6): q = rne(x * 2^9) is the code (q = 8 lands on
    the smallest normal 0x08).  Normal range: x = 2^e * (1 + f), mantissa
    m = rne(f * 8), a carry m == 8 moves to the next binade.
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    if np.any(x < 0) or np.any(np.isnan(x)):
        raise ValueError("e4m3_encode: scales are non-negative numbers")
    out = np.zeros(x.shape, dtype=np.int64)
    sat = x >= 448.0
    sub = (x < 2.0 ** -6) & ~sat
    nrm = ~sat & ~sub
    out[sub] = np.rint(x[sub] * 2.0 ** 9).astype(np.int64)
    if np.any(nrm):
        mant, exp = np.frexp(x[nrm])  # x = mant * 2^exp, mant in [0.5, 1)
        e = exp - 1                    # x = (2*mant) * 2^e, 2*mant in [1, 2)
        m = np.rint((2.0 * mant - 1.0) * 8.0).astype(np.int64)
        carry = m == 8
        e = np.where(carry, e + 1, e)
        m = np.where(carry, 0, m)
        out[nrm] = ((e + 7) << 3) | m
    out[sat] = 0x7E
    return out.astype(np.uint8)


# Magnitude thresholds of RNE onto {0, .5, 1, 1.5, 2, 3, 4, 6}: a value on a
# midpoint goes to the neighbour with the even code.
def e2m1_encode(y) -> np.ndarray:
    """fp32 value -> 4-bit e2m1 code (uint8 in 0..15), RNE with ties to even, saturating at 6.

    The sign bit is the sign bit of ``y`` (so -0.0 and small negatives give 0x8).
    """
    y = np.asarray(y, dtype=np.float32)
    a = np.abs(y).astype(np.float64)
    mag = np.select(
        [a <= 0.25, a < 0.75, a <= 1.25, a < 1.75, a <= 2.5, a < 3.5, a <= 5.0],
        [0, 1, 2, 3, 4, 5, 6],
        default=7,
    )
    sign = np.signbit(y).astype(np.int64) << 3
    return (sign | mag).astype(np.uint8)


def ue8m0_encode_up(s) -> np.ndarray:
    """Non-negative fp32 scale -> smallest power-of-two ue8m0 code with 2^(c-127) >= s, clamped to [0, 254]."""
    s = np.asarray(s, dtype=np.float32).astype(np.float64)
    mant, exp = np.frexp(s)            # s = mant * 2^exp, mant in [0.5, 1) or s == 0
    k = np.where(mant == 0.5, exp - 1, exp)  # exact powers of two need no rounding up
    code = np.where(s == 0.0, 0, k + 127)
    return np.clip(code, 0, 254).astype(np.uint8)

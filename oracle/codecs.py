"""Bit-level codecs used by the oracle (test infrastructure only).

bf16: 1 sign, 8 exponent, 7 mantissa bits; the upper half of an IEEE
binary32.  Decoding is exact in float64.  Encoding rounds to nearest, ties
to even.

e4m3 (OCP 8-bit floating point, "E4M3"): 1 sign, 4 exponent, 3 mantissa bits,
exponent bias 7, no infinities, S.1111.111 is NaN, largest finite magnitude
1.75 * 2^8 = 448, subnormals m/8 * 2^-6 (smallest 2^-9).  The encoder rounds
to nearest, ties to even, and saturates finite overflow to +-448 (the
``satfinite`` convention); the DCP + FP8 KV MLA decode digest
(§实现拆解 1, §关键源码片段 mla_attention.py) names the concat-quant step
but not its rounding, so this plain reading is taken.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_to_f64", "f64_to_bf16", "f32_to_bf16",
    "e4m3_to_f64", "f32_to_e4m3", "E4M3_MAX",
]

E4M3_MAX = 448.0


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16/int16) -> exact float64 values."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f32_to_bf16(x) -> np.ndarray:
    """float32 values -> bf16 bits, round to nearest even (NaN stays NaN)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lower = u & 0xFFFF
    upper = u >> 16
    # round half to even on the 16 dropped bits
    round_up = (lower > 0x8000) | ((lower == 0x8000) & ((upper & 1) == 1))
    out = (upper + round_up.astype(np.uint64)) & 0xFFFF
    nan = np.isnan(x)
    out = np.where(nan, (upper | 0x40) & 0xFFFF, out)   # quiet NaN, keep sign
    return out.astype(np.uint16)


def f64_to_bf16(x) -> np.ndarray:
    """float64 -> bf16 bits via the exact float32 value when it is one.

    Only used on values that are already float32-representable; a general
    double would need a single rounding, which the oracle never asks for."""
    x = np.asarray(x, dtype=np.float64)
    x32 = x.astype(np.float32)
    if not np.all((x32.astype(np.float64) == x) | np.isnan(x)):
        raise ValueError("f64_to_bf16 expects float32-representable values")
    return f32_to_bf16(x32)


def e4m3_to_f64(codes) -> np.ndarray:
    """e4m3 codes (uint8) -> float64 values from the format definition."""
    c = np.asarray(codes).astype(np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (8.0 + m) * np.exp2(e - 10.0)      # (1 + m/8) * 2^(e-7)
    sub = m * 2.0 ** -9                          # (m/8) * 2^-6
    mag = np.where(e == 0, sub, normal)
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def f32_to_e4m3(x) -> np.ndarray:
    """float32 values -> e4m3 codes: round to nearest even, satfinite.

    Arithmetic is exact: every float32 is exact in float64, the quantum is a
    power of two, so ``a / quantum`` is exact and ``np.rint`` (ties to even)
    performs the one rounding.  +-inf saturates to +-448; NaN -> 0x7F with
    its sign bit."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    sign = np.signbit(x).astype(np.int64) << 7
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    a = np.minimum(a, 1e30)  # inf -> large finite, saturates below
    # exponent of the binade; subnormal range shares the 2^-6 binade's quantum
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)
    # guard against log2 rounding at exact powers of two
    e = np.where(a >= np.exp2(e + 1), e + 1, e)
    e = np.where(a < np.exp2(e), e - 1, e)
    e = np.clip(e, -6, 8)
    quantum = np.exp2(e - 3)
    q = np.rint(a / quantum)                     # ties to even
    val = q * quantum
    val = np.minimum(val, E4M3_MAX)              # satfinite
    # re-derive fields from the rounded value
    with np.errstate(divide="ignore"):
        e2 = np.floor(np.log2(np.where(val > 0, val, 1.0)))
    e2 = np.clip(e2, -6, 8)
    e2 = np.where(val >= np.exp2(e2 + 1), e2 + 1, e2)
    e2 = np.where((val > 0) & (val < np.exp2(e2)), e2 - 1, e2)
    e2 = np.clip(e2, -6, 8)
    is_normal = val >= 2.0 ** -6
    mant_norm = np.rint(val / np.exp2(e2 - 3)) - 8
    code_norm = ((e2 + 7).astype(np.int64) << 3) | mant_norm.astype(np.int64)
    code_sub = np.rint(val / 2.0 ** -9).astype(np.int64)
    code = np.where(is_normal, code_norm, code_sub)
    code = np.where(nan, 0x7F, code)
    return (code | sign).astype(np.uint8)

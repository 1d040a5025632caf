"""bfloat16 decode / encode for the oracle (test infrastructure only).

bfloat16 is the top half of an IEEE-754 binary32 pattern: 1 sign bit, 8
exponent bits (bias 127), 7 fraction bits.  Every bf16 value is exactly
representable in float64, so decoding is exact.  Encoding rounds a float64
value directly to the nearest bf16 value, ties to even, without passing
through float32 (so there is no double rounding).
"""
from __future__ import annotations

import numpy as np

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127          # largest finite bf16
BF16_MIN_NORMAL_EXP = -126                          # 2^-126 smallest normal
BF16_SUBNORMAL_QUANTUM_EXP = -133                   # 2^-133 = spacing of subnormals


def decode(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values, exactly."""
    b = np.asarray(bits, dtype=np.uint16)
    f32 = (b.astype(np.uint32) << np.uint32(16)).view(np.float32)
    with np.errstate(invalid="ignore"):
        return f32.astype(np.float64)


def encode_rne(x) -> np.ndarray:
    """float64 -> bf16 bit patterns (uint16), round to nearest, ties to even.

    Overflow rounds to +-inf, NaN becomes the quiet NaN 0x7FC0 (sign kept),
    subnormals are kept (no flush to zero)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint16)
    sign = np.where(np.signbit(x), np.uint16(0x8000), np.uint16(0))
    a = np.abs(x)
    nan = np.isnan(x)
    fin = np.isfinite(x) & (a > 0)
    # a = m * 2^e with m in [0.5, 1): eight significant bits => quantum 2^(e-8),
    # but never finer than the subnormal spacing 2^-133.
    _, e = np.frexp(np.where(fin, a, 1.0))
    q_exp = np.maximum(e - 8, BF16_SUBNORMAL_QUANTUM_EXP)
    q = np.ldexp(1.0, q_exp)
    r = np.where(fin, np.rint(a / q) * q, 0.0)      # np.rint rounds half to even
    over = fin & (r > BF16_MAX)
    ok = fin & ~over
    # r now has at most eight significant bits: exactly a float32, then take the top half
    r32 = np.where(ok, r, 0.0).astype(np.float32)
    mag = (r32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    out = np.where(ok, mag, out)
    out = np.where(over | (np.isinf(x)), np.uint16(0x7F80), out)
    out = (out | sign).astype(np.uint16)
    out = np.where(nan, np.uint16(0x7FC0) | sign, out).astype(np.uint16)
    return out

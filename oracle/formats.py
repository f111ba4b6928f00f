"""E2M1 element codes and E4M3 block-scale bytes, decoded and encoded from their bit layouts.

[TRACE] "NVFP4 与 E2M1 码本": the NVFP4 element format is E2M1 -- 1 sign bit,
2 exponent bits, 1 mantissa bit -- so a value can only take one of a finite set
of codebook levels, and a real value is rounded to the nearest level.
[QUADS] section 1: the E2M1 grid has only 8 positive representable levels per
sign (counting zero).

The block scale is one byte per 16 elements (the 1.5 bit-per-value record cost
in [TRACE] "核心方法" is 1 mantissa bit + 8 scale bits / 16 values); the byte
is an unsigned OCP FP8 E4M3 value (4 exponent bits, bias 7, 3 mantissa bits,
subnormals, no infinities; 0x7F is NaN, the largest finite value 448).

Rounding is to nearest; an exact midpoint goes to the code whose lowest bit is
0 (the even mantissa bit), which is the IEEE round-half-to-even rule restated
on codes.  E4M3 encoding saturates at 448 and never produces NaN.
"""
from __future__ import annotations

import numpy as np

E2M1_EXP_BITS, E2M1_MAN_BITS, E2M1_BIAS = 2, 1, 1
E4M3_EXP_BITS, E4M3_MAN_BITS, E4M3_BIAS = 4, 3, 7


def e2m1_level(magnitude_code: int) -> float:
    """Value of a 3-bit E2M1 magnitude code (exponent e, mantissa m)."""
    e = magnitude_code >> E2M1_MAN_BITS
    m = magnitude_code & ((1 << E2M1_MAN_BITS) - 1)
    if e == 0:  # subnormal: m * 2^(1 - bias) / 2^man_bits
        return m * 2.0 ** (1 - E2M1_BIAS) / (1 << E2M1_MAN_BITS)
    return (1.0 + m / (1 << E2M1_MAN_BITS)) * 2.0 ** (e - E2M1_BIAS)


#: non-negative E2M1 levels in code order 0..7
E2M1_LEVELS = np.array([e2m1_level(c) for c in range(8)], dtype=np.float64)


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """4-bit codes (bit 3 = sign) -> float64 values (code 0x8 decodes to -0.0)."""
    codes = np.asarray(codes, dtype=np.uint8)
    mag = E2M1_LEVELS[codes & 7]
    return np.where(codes & 8, -mag, mag)


def _nearest_code(mag: np.ndarray, levels: np.ndarray) -> np.ndarray:
    """Index of the nearest entry of the ascending table ``levels``; a midpoint
    goes to the even index.  ``mag`` must be >= 0 and <= levels[-1]."""
    mag = np.asarray(mag, dtype=np.float64)
    hi = np.searchsorted(levels, mag, side="left")          # levels[hi] >= mag
    hi = np.minimum(hi, len(levels) - 1)
    lo = np.maximum(hi - 1, 0)
    mid = (levels[lo] + levels[hi]) * 0.5                   # exact: dyadic values
    pick_hi = (mag > mid) | ((mag == mid) & (hi % 2 == 0))
    pick = np.where(pick_hi, hi, lo)
    return np.where(levels[hi] == mag, hi, pick)


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """Round float32 values to E2M1 codes: nearest level, ties to even, |v| > 6 -> 6.

    The sign bit is the sign bit of v, so a negative value that rounds to zero
    (and -0.0) gives code 0x8.  NaN is outside the domain.
    """
    v = np.asarray(v, dtype=np.float32)
    mag = np.minimum(np.abs(v).astype(np.float64), E2M1_LEVELS[-1])
    code = _nearest_code(mag, E2M1_LEVELS).astype(np.uint8)
    return code | (np.signbit(v).astype(np.uint8) << 3)


def e4m3_value(code: int) -> float:
    """Value of one E4M3 byte (sign bit honoured; 0x7F/0xFF are NaN)."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> E4M3_MAN_BITS) & ((1 << E4M3_EXP_BITS) - 1)
    m = code & ((1 << E4M3_MAN_BITS) - 1)
    if e == (1 << E4M3_EXP_BITS) - 1 and m == (1 << E4M3_MAN_BITS) - 1:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** (1 - E4M3_BIAS) / (1 << E4M3_MAN_BITS)
    return s * (1.0 + m / (1 << E4M3_MAN_BITS)) * 2.0 ** (e - E4M3_BIAS)


#: decode table for all 256 bytes (float64; NaN at 0x7F and 0xFF)
E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
#: the 127 finite non-negative values, codes 0x00..0x7E, ascending
E4M3_POS = E4M3_TABLE[:0x7F].copy()
E4M3_MAX = E4M3_POS[-1]


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode_satfinite(u: np.ndarray) -> np.ndarray:
    """Round non-negative float32 values to E4M3 bytes: nearest, ties to even,
    values above 448 (including +inf) saturate to 448 (0x7E)."""
    u = np.asarray(u, dtype=np.float32).astype(np.float64)
    if np.any(~(u >= 0)):
        raise ValueError("e4m3_encode_satfinite: inputs must be >= 0 and not NaN")
    mag = np.minimum(u, E4M3_MAX)
    return _nearest_code(mag, E4M3_POS).astype(np.uint8)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[rows, 2n] 4-bit codes -> [rows, n] bytes; element 2i in the low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] & 0xF) | ((codes[..., 1::2] & 0xF) << 4)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out

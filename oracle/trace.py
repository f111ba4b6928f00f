"""TRACE rollout-guided rounding (an optional quantizer mode).

[TRACE] "核心方法": for each training-side activation, take the two E2M1 codes
that neighbour it under the rollout side's scale, {q-, q+}; when the rollout
code q_rollout is known, do not round to nearest but pick
q_TRACE = argmin over q in {q-, q+} of |q - q_rollout|.  Eq. (3): by
construction |q_TRACE - q_rollout| <= |q_RTN - q_rollout| at every element.
"方法步骤详情" step 4 replaces RTN by this choice in the forward fake-quant.

Readings: the scaled value is v = x_train * (1 / d_b) with the rollout block's
d_b (as in the RTN quantizer); q- is the largest signed level <= v and q+ the
smallest signed level >= v, both clamped to [-6, 6] (so q- = q+ when v is a
level or |v| >= 6); a zero result carries the sign of v; a block whose rollout
d_b is 0 (or whose reciprocal overflows) gives 0x0.  Codes are compared by
value, so +0 and -0 are the same level.
"""
from __future__ import annotations

import numpy as np

from .formats import E2M1_LEVELS, e2m1_decode, e2m1_encode, e4m3_decode

BLOCK = 16
#: the 15 distinct signed E2M1 values, ascending (+0 and -0 are one value)
SIGNED_LEVELS = np.unique(np.concatenate([-E2M1_LEVELS, E2M1_LEVELS]))


def _scaled(x_train, rollout_scales, s_t):
    x = np.asarray(x_train, dtype=np.float32)
    rows, cols = x.shape
    s_t = np.float32(s_t)
    d_b = (e4m3_decode(rollout_scales).astype(np.float32) * s_t).astype(np.float32)
    with np.errstate(divide="ignore"):
        r_b = (np.float32(1.0) / d_b).astype(np.float32)
    zero = (d_b == 0) | np.isinf(r_b)
    with np.errstate(invalid="ignore"):
        v = (x.reshape(rows, cols // BLOCK, BLOCK) * r_b[:, :, None]).astype(np.float32)
    v = np.where(zero[:, :, None], np.float32(0.0), v).reshape(rows, cols)
    zero_el = np.repeat(zero, BLOCK, axis=1)
    return v, zero_el


def _value_to_code(q: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Encode an exact E2M1 value; zero takes the sign of v."""
    mag = np.abs(q)
    code = np.searchsorted(E2M1_LEVELS, mag).astype(np.uint8)
    neg = (q < 0) | ((q == 0) & np.signbit(v))
    return code | (neg.astype(np.uint8) << 3)


def neighbours(v: np.ndarray):
    """(q-, q+): largest signed level <= v and smallest signed level >= v, clamped to [-6, 6]."""
    v = np.asarray(v, dtype=np.float64)
    L = SIGNED_LEVELS
    vc = np.clip(v, L[0], L[-1])
    i_hi = np.searchsorted(L, vc, side="left")       # L[i_hi] >= vc
    i_lo = np.searchsorted(L, vc, side="right") - 1  # L[i_lo] <= vc
    return L[i_lo], L[i_hi]


def trace_round(x_train, rollout_codes, rollout_scales, s_t):
    """Returns (codes uint8 [rows, cols], counters dict)."""
    v, zero_el = _scaled(x_train, rollout_scales, s_t)
    q_roll = e2m1_decode(rollout_codes)
    q_lo, q_hi = neighbours(v)
    pick_lo = np.abs(q_lo - q_roll) <= np.abs(q_hi - q_roll)   # never a tie unless q_lo == q_hi
    q_tr = np.where(pick_lo, q_lo, q_hi)
    codes = _value_to_code(q_tr, v)
    codes = np.where(zero_el, np.uint8(0), codes).astype(np.uint8)
    q_rtn = e2m1_decode(np.where(zero_el, np.uint8(0), e2m1_encode(v)))
    return codes, mismatch_counters(q_rtn, e2m1_decode(codes), q_roll)


def mismatch_counters(q_rtn, q_trace, q_roll) -> dict:
    """#RTN != rollout, #TRACE != rollout, and how many RTN mismatches are one
    adjacent level apart (the pages report over 99% for real activations)."""
    mism = q_rtn != q_roll
    i_rtn = np.searchsorted(SIGNED_LEVELS, q_rtn).astype(np.int64)   # -0.0 == 0.0 here
    i_roll = np.searchsorted(SIGNED_LEVELS, q_roll).astype(np.int64)
    adj = mism & (np.abs(i_rtn - i_roll) == 1)
    return dict(rtn_mismatch=int(mism.sum()), trace_mismatch=int((q_trace != q_roll).sum()),
                rtn_off_by_one=int(adj.sum()))


def cross_path_difference(codes_a, codes_b, scales, s_t) -> float:
    """||DQ(q_a) - DQ(q_b)||_F under one set of scales: the cross-path difference
    TRACE minimises ("研究动机", objective (1))."""
    d_b = (e4m3_decode(scales).astype(np.float64) * float(np.float32(s_t)))
    da = e2m1_decode(codes_a).reshape(d_b.shape[0], -1, BLOCK) * d_b[:, :, None]
    db = e2m1_decode(codes_b).reshape(d_b.shape[0], -1, BLOCK) * d_b[:, :, None]
    return float(np.sqrt(np.sum((da - db) ** 2)))


def _mantissa(q: np.ndarray) -> np.ndarray:
    """Mantissa bit of an E2M1 value: the low bit of its magnitude code."""
    return (np.searchsorted(E2M1_LEVELS, np.abs(q)) & 1).astype(np.uint8)


def pack_record(rollout_codes) -> np.ndarray:
    """[TRACE] "核心方法" / "方法步骤详情" step 2: the compact record keeps one
    mantissa bit per value (plus the block scales, kept as they are).
    Returns bytes [rows, cols/8], element 8i+j in bit j of byte i."""
    c = np.asarray(rollout_codes, dtype=np.uint8)
    rows, cols = c.shape
    m = (c & 1).reshape(rows, cols // 8, 8).astype(np.uint16)
    return (m << np.arange(8, dtype=np.uint16)).sum(axis=2).astype(np.uint8)


def unpack_record(bits, cols: int) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint8)[:, : cols // 8]
    return ((b[:, :, None] >> np.arange(8, dtype=np.uint8)) & 1).reshape(b.shape[0], cols)


def trace_round_1bit(x_train, mantissa_bits, rollout_scales, s_t):
    """TRACE with the 1-bit record: of the neighbours {q-, q+} of v take the one
    whose mantissa bit equals the record's (adjacent signed E2M1 levels have
    opposite mantissa bits, so one bit names one of them -- the rollout's code
    whenever it is a neighbour; "核心方法": over 99% of mismatches are one code
    apart).  Same v, clamping, zero sign and zero-block rules as trace_round.

    Returns (codes uint8 [rows, cols], counters dict: changed vs RTN,
    record-bit mismatches)."""
    v, zero_el = _scaled(x_train, rollout_scales, s_t)
    rows, cols = v.shape
    bit = unpack_record(mantissa_bits, cols)
    q_lo, q_hi = neighbours(v)
    pick_lo = (q_lo == q_hi) | (_mantissa(q_lo) == bit)
    q = np.where(pick_lo, q_lo, q_hi)
    codes = np.where(zero_el, np.uint8(0), _value_to_code(q, v)).astype(np.uint8)
    q_rtn = e2m1_decode(np.where(zero_el, np.uint8(0), e2m1_encode(v)))
    q_out = e2m1_decode(codes)
    return codes, dict(changed=int((q_out != q_rtn).sum()),
                       bit_mismatch=int((_mantissa(q_out) != bit).sum()))


def trace_round_mx(x_train, rollout_codes, rollout_e8m0):
    """trace_round under an MXFP4 rollout: v = x_train / 2^e with the rollout
    block's E8M0 scale (32-element blocks, no tensor scale, never a zero block)."""
    x = np.asarray(x_train, dtype=np.float32)
    rows, cols = x.shape
    e = np.asarray(rollout_e8m0, dtype=np.int64) - 127
    v = np.ldexp(x.reshape(rows, cols // 32, 32).astype(np.float64), -e[:, :, None])
    v = v.astype(np.float32).reshape(rows, cols)
    q_roll = e2m1_decode(rollout_codes)
    q_lo, q_hi = neighbours(v)
    pick_lo = np.abs(q_lo - q_roll) <= np.abs(q_hi - q_roll)
    codes = _value_to_code(np.where(pick_lo, q_lo, q_hi), v)
    q_rtn = e2m1_decode(e2m1_encode(v))
    return codes, mismatch_counters(q_rtn, e2m1_decode(codes), q_roll)

"""Pins for the oracle's TRACE mantissa-only mode (CPU only): the record's
size and bit order, the pages' worked example, and the off-by-one property
that lets one bit stand in for the whole rollout code."""
import json
import os

import numpy as np

from nvfp4_w4a4_quantized_quant_gb300 import inputs
from oracle import formats as F
from oracle import nvfp4 as Q
from oracle import trace as T

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_record_is_one_mantissa_bit_per_value_in_element_order():
    codes = np.array([[0x0, 0x1, 0x2, 0x3, 0x9, 0xB, 0xE, 0xF, 0x7, 0x6, 0x5, 0x4, 0x8, 0xA, 0xC, 0xD]],
                     np.uint8)
    bits = T.pack_record(codes)
    # mantissa bits 0,1,0,1,1,1,0,1 | 1,0,1,0,0,0,0,1, element 8i+j in bit j of byte i
    assert bits.shape == (1, 2)
    assert bits[0, 0] == 0b10111010 and bits[0, 1] == 0b10000101
    assert np.array_equal(T.unpack_record(bits, 16)[0], codes[0] & 1)
    # with the 8-bit scale per 16 values the record costs 1.5 bits per value
    g = json.load(open(os.path.join(GOLD, "trace_record_size.json")))
    per_value = (bits.nbytes * 8 + 8 * (16 // 16)) / 16
    assert per_value == g["bits_per_value"]
    assert g["hidden"] * g["layers_kept"] * per_value == g["total_bits"]


def test_adjacent_signed_levels_alternate_mantissa_bits():
    m = T._mantissa(T.SIGNED_LEVELS)
    assert np.all(m[1:] != m[:-1])


def test_one_bit_mode_fixes_the_worked_boundary_example():
    g = json.load(open(os.path.join(GOLD, "trace_worked_example.json")))
    to_bf16 = lambda v: inputs.bf16_bits_to_f32(inputs.f32_to_bf16_bits(np.float32([v])))[0]  # noqa
    xr = np.zeros((1, 16), np.float32)
    xr[0, 0], xr[0, 1] = to_bf16(g["x_rollout"]), 144.0
    xt = xr.copy()
    xt[0, 0] = to_bf16(g["x_train"])
    s_t = Q.tensor_scale(xr)
    rc, rs = Q.quantize(xr, s_t)
    codes, cnt = T.trace_round_1bit(xt, T.pack_record(rc), rs, s_t)
    assert F.e2m1_decode(codes[0, 0]) == g["rounded_levels"][1]
    assert np.array_equal(codes, rc)
    assert cnt["changed"] == 1 and cnt["bit_mismatch"] == 0


def test_one_bit_equals_full_trace_whenever_the_rollout_is_a_neighbour():
    """Brute force over every signed rollout level and a dense grid of scaled
    training values (unit scales): the 1-bit choice always lies in {q-, q+},
    and equals full TRACE when the rollout level is q- or q+, or two levels
    below q- / above q+."""
    L = T.SIGNED_LEVELS
    v = np.linspace(-7.0, 7.0, 561, dtype=np.float32)
    v = np.concatenate([v, L.astype(np.float32)])
    n = v.size
    pad = (-n) % 16
    v = np.concatenate([v, np.zeros(pad, np.float32)])
    xt = v.reshape(-1, 16)
    scales = np.full((xt.shape[0], 1), 0x38, np.uint8)        # E4M3 1.0, tensor scale 1
    q_lo, q_hi = T.neighbours(xt)
    for lev in L:
        rc = np.broadcast_to(T._value_to_code(np.float64(lev), np.float64(lev)), xt.shape).astype(np.uint8)
        full, _ = T.trace_round(xt, rc, scales, 1.0)
        one, _ = T.trace_round_1bit(xt, T.pack_record(rc), scales, 1.0)
        q1 = F.e2m1_decode(one)
        assert np.all((q1 == q_lo) | (q1 == q_hi))
        i_lo, i_hi = np.searchsorted(L, q_lo), np.searchsorted(L, q_hi)
        i_r = np.searchsorted(L, lev)
        # the rollout level is a neighbour, or two levels beyond the nearer one
        # (same mantissa bit as that neighbour), or v sits on a level
        near = ((i_r == i_lo) | (i_r == i_hi) | (i_r == i_lo - 2) | (i_r == i_hi + 2) |
                (i_lo == i_hi))
        fq = F.e2m1_decode(full)
        assert np.array_equal(q1[near], fq[near])
        # elsewhere the two modes can differ (the bit names the farther neighbour)
        if lev == 0.0:
            assert not np.array_equal(q1, fq)


def test_one_bit_mode_on_rollout_like_activations():
    """Student-t activations with a 1% training-side perturbation: the record
    bit is met everywhere except where v sits on a level (or is clamped), and
    the result equals full TRACE at every element whose RTN code is within one
    level of the rollout code."""
    d = inputs.trace_rounding(3, 64, 256)
    xr = inputs.bf16_bits_to_f32(d["x_rollout"])
    xt = inputs.bf16_bits_to_f32(d["x_train"])
    rc, rs, st = Q.quantize_groups(xr)
    one, cnt = T.trace_round_1bit(xt, T.pack_record(rc), rs, st[0])
    full, fcnt = T.trace_round(xt, rc, rs, st[0])
    v, _ = T._scaled(xt, rs, st[0])
    q_rtn = F.e2m1_decode(F.e2m1_encode(v))
    i_rtn = np.searchsorted(T.SIGNED_LEVELS, q_rtn)
    i_roll = np.searchsorted(T.SIGNED_LEVELS, F.e2m1_decode(rc))
    close = np.abs(i_rtn - i_roll) <= 1
    assert np.array_equal(F.e2m1_decode(one)[close], F.e2m1_decode(full)[close])
    assert cnt["changed"] > 0
    q_lo, q_hi = T.neighbours(v)
    assert cnt["bit_mismatch"] <= int((q_lo == q_hi).sum())

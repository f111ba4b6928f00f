"""Pins for the oracle's E2M1 / E4M3 codecs (CPU only)."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_e2m1_codebook_matches_pages():
    g = json.load(open(os.path.join(GOLD, "e2m1_codebook.json")))
    assert F.E2M1_EXP_BITS == g["exponent_bits"] and F.E2M1_MAN_BITS == g["mantissa_bits"]
    levels = F.E2M1_LEVELS
    assert len(levels) == g["levels_per_sign"] == 1 << (F.E2M1_EXP_BITS + F.E2M1_MAN_BITS)
    assert levels[0] == 0.0 and np.all(np.diff(levels) > 0)
    # the worked boundary example needs 2 and 3 to be adjacent levels with the
    # rounding boundary between them at 2.5 (2.51 -> 3, 2.49 -> 2)
    i2 = int(np.nonzero(levels == 2.0)[0][0])
    assert levels[i2 + 1] == 3.0
    assert F.e2m1_decode(F.e2m1_encode(np.float32([2.51, 2.49]))).tolist() == [3.0, 2.0]


def _brute_e2m1(v: float) -> int:
    """argmin over all 8 magnitudes; ties -> even magnitude code; sign from the sign bit."""
    mag = min(abs(v), 6.0)
    best, bestd = None, None
    for c in range(8):
        d = abs(F.e2m1_level(c) - mag)
        if best is None or d < bestd or (d == bestd and c % 2 == 0):
            best, bestd = c, d
    return best | (8 if np.signbit(v) else 0)


def test_e2m1_encode_all_bf16_inputs_brute_force():
    bits = np.arange(1 << 16, dtype=np.uint32)
    v = (bits << 16).view(np.float32)
    v = v[np.isfinite(v)]
    got = F.e2m1_encode(v)
    exp = np.array([_brute_e2m1(float(x)) for x in v], dtype=np.uint8)
    assert np.array_equal(got, exp)


def test_e2m1_ties_and_sign_rules():
    v = np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, -0.1, -0.0, 0.0, -7.0])
    got = F.e2m1_decode(F.e2m1_encode(v))
    assert got.tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, -0.0, -0.0, 0.0, -6.0]
    codes = F.e2m1_encode(v)
    assert codes[8] == 0x8 and codes[9] == 0x8 and codes[10] == 0x0


def test_e4m3_decode_matches_torch_float8():
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.E4M3_TABLE
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert F.E4M3_MAX == 448.0 and F.e4m3_value(0x38) == 1.0 and F.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne():
    # every float32 bit pattern on a fixed stride over [2^-12, 448], plus dense
    # neighbourhoods of all midpoints between consecutive E4M3 values
    lo, hi = np.float32(2.0 ** -12).view(np.uint32), np.float32(448.0).view(np.uint32)
    grid = np.arange(lo, hi + 1, 977, dtype=np.uint32).view(np.float32)
    mids = ((F.E4M3_POS[:-1] + F.E4M3_POS[1:]) / 2).astype(np.float32)
    around = (mids.view(np.uint32)[:, None] + np.arange(-4, 5, dtype=np.int64)[None, :]
              ).astype(np.uint32).view(np.float32).ravel()
    u = np.concatenate([grid, around, np.float32([0.0, 2.0 ** -10, 2.0 ** -11, 448.0])])
    u = u[(u >= 0) & (u <= 448)]
    ours = F.e4m3_encode_satfinite(u)
    ref = torch.from_numpy(u.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturates_above_448():
    u = np.float32([448.0, 449.0, 464.0, 1e6, np.inf])
    assert F.e4m3_encode_satfinite(u).tolist() == [0x7E] * 5
    with pytest.raises(ValueError):
        F.e4m3_encode_satfinite(np.float32([-1.0]))


def test_nibble_packing_roundtrip():
    rng = np.random.default_rng(0)
    c = rng.integers(0, 16, size=(3, 32), dtype=np.uint8)
    p = F.pack_nibbles(c)
    assert p.shape == (3, 16) and p[0, 0] == (c[0, 0] | (c[0, 1] << 4))
    assert np.array_equal(F.unpack_nibbles(p), c)


def test_record_size_arithmetic_implies_16_element_blocks_of_8_bit_scales():
    g = json.load(open(os.path.join(GOLD, "trace_record_size.json")))
    assert g["hidden"] * g["layers_kept"] * g["bits_per_value"] == g["total_bits"]
    assert g["total_bits"] / 8 / 1024 == g["kilobytes_per_token"]
    scale_bits_per_value = g["bits_per_value"] - g["mantissa_bits_per_value"]
    # one 8-bit scale amortised over a 16-element block
    assert scale_bits_per_value == 8 / 16

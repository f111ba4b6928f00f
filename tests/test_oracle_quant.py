"""Pins for the oracle's NVFP4 quantizer, residual, scores, selection and the
second quantization (CPU only)."""
import json
import os

import numpy as np

from nvfp4_w4a4_quantized_quant_gb300 import inputs
from oracle import formats as F
from oracle import nvfp4 as Q

GOLD = os.path.join(os.path.dirname(__file__), "golden")
f32 = np.float32


def _bf16(x):
    return np.float32(inputs.bf16_bits_to_f32(inputs.f32_to_bf16_bits(np.float32([x])))[0])


def test_worked_boundary_example():
    """60.24 (train) and 59.76 (rollout) under one set of scales -> 2.51 / 2.49 ->
    codes 3 / 2 -> dequantized difference 24."""
    g = json.load(open(os.path.join(GOLD, "trace_worked_example.json")))
    xt, xr = _bf16(g["x_train"]), _bf16(g["x_rollout"])
    assert abs((xt - xr) - g["bf16_difference_printed"]) <= 0.03   # bf16: 60.25 - 59.75
    # a block whose largest magnitude is 144 in a tensor with amax 144 gives d_b = 24
    for x in (xt, xr):
        blk = np.zeros((1, 16), np.float32)
        blk[0, 0], blk[0, 1] = x, 144.0
        s_t = Q.tensor_scale(blk)
        codes, sc = Q.quantize(blk, s_t)
        d_b = f32(F.e4m3_value(int(sc[0, 0])) * s_t)
        assert d_b == 24.0
    scaled = [float(f32(xt * f32(1.0 / f32(24.0)))), float(f32(xr * f32(1.0 / f32(24.0))))]
    assert np.allclose(scaled, g["scaled_printed"], atol=0.006)
    lv = []
    for x in (xt, xr):
        blk = np.zeros((1, 16), np.float32)
        blk[0, 0], blk[0, 1] = x, 144.0
        c, sc = Q.quantize(blk, Q.tensor_scale(blk))
        lv.append(float(F.e2m1_decode(c[0, 0])))
        dq = Q.dequantize(c, sc, Q.tensor_scale(blk))
    assert lv == g["rounded_levels"]
    assert (lv[0] - lv[1]) * 24.0 == g["dequantized_difference"]


def test_exact_ties_go_to_even():
    # d_b = 24: 60 -> 2.5 -> 2, 84 -> 3.5 -> 4, 36 -> 1.5 exactly
    blk = np.zeros((1, 16), np.float32)
    blk[0, :4] = [60.0, 84.0, 36.0, 144.0]
    c, sc = Q.quantize(blk, Q.tensor_scale(blk))
    assert F.e2m1_decode(c[0, :4]).tolist() == [2.0, 4.0, 1.5, 6.0]


def test_zero_tensor_and_zero_block():
    x = np.zeros((4, 32), np.float32)
    c, s, st = Q.quantize_groups(x)
    assert st[0] == 1.0 and not c.any() and not s.any()
    x[0, 16:] = 1.0
    c, s, st = Q.quantize_groups(x)
    assert s[0, 0] == 0 and not c[0, :16].any() and s[0, 1] != 0


def test_negative_zero_and_small_negative_keep_sign():
    x = np.zeros((1, 16), np.float32)
    x[0, :3] = [-0.0, -0.01, 6.0]
    c, _, _ = Q.quantize_groups(x)
    assert c[0, 0] == 0x8 and c[0, 1] == 0x8 and c[0, 2] == 0x7


def _exact_tensor(rng, rows, cols):
    """Values level * S (S an E4M3 value) with every block holding level 6, in a
    tensor whose amax is 2688 so that s_t = 1: quantization must be exact."""
    codes = rng.integers(0, 16, size=(rows, cols), dtype=np.uint8)
    codes[:, ::16] = 7                                   # magnitude 6 in every block
    sb = rng.integers(0x20, 0x7F, size=(rows, cols // 16), dtype=np.uint8)
    sb[0, 0] = 0x7E                                      # 448 -> amax = 6 * 448 = 2688
    x = (F.e2m1_decode(codes).reshape(rows, -1, 16) * F.e4m3_decode(sb)[:, :, None])
    x = x.reshape(rows, cols).astype(np.float32)
    return x, codes, sb


def test_exactly_representable_tensor_roundtrips():
    rng = np.random.default_rng(1)
    x, codes, sb = _exact_tensor(rng, 8, 64)
    c, s, st = Q.quantize_groups(x)
    assert st[0] == 1.0
    assert np.array_equal(s, sb)
    # codes agree up to the sign of zero
    assert np.array_equal(F.e2m1_decode(c), F.e2m1_decode(codes))
    assert not Q.residual(x, c, s, st[0]).any()


def test_power_of_two_scaling_leaves_codes_and_block_scales_unchanged():
    rng = np.random.default_rng(2)
    x = inputs.student_t4(rng, (16, 64))
    c1, s1, t1 = Q.quantize_groups(x)
    c2, s2, t2 = Q.quantize_groups(x * f32(8.0))
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2) and t2[0] == t1[0] * 8


def test_codes_are_nearest_levels_and_error_is_bounded():
    rng = np.random.default_rng(3)
    x = inputs.student_t4(rng, (32, 128)) * f32(3.0)
    c, s, st = Q.quantize_groups(x)
    d_b = (F.e4m3_decode(s) * float(st[0])).repeat(16, axis=1)
    lv = F.e2m1_decode(c)
    scaled = x.astype(np.float64) / d_b
    # no other level is closer to the scaled value (beyond float32 rounding)
    dist = np.abs(F.E2M1_LEVELS[None, None, :] - np.abs(scaled)[:, :, None]).min(axis=2)
    assert np.all(np.abs(np.abs(lv) - np.abs(scaled)) <= dist + 1e-5)
    # block amax lands on the top two levels (scale rounding is within 2^-4)
    top = np.abs(lv).reshape(32, -1, 16).max(axis=2)
    assert np.all(np.isin(top, [4.0, 6.0]))


def test_channel_scores_closed_form_and_chunk_order():
    R = np.zeros((70, 32), np.float32)
    R[:, 3] = 1.0
    R[:, 5] = 2.0
    R[::2, 7] = 3.0
    sc = Q.channel_scores(R)[0]
    assert sc[3] == 70.0 and sc[5] == 280.0 and sc[7] == 35 * 9.0 and sc[0] == 0.0
    rng = np.random.default_rng(4)
    R = rng.standard_normal((200, 48)).astype(np.float32)
    ref = (R.astype(np.float64) ** 2).sum(axis=0)
    assert np.allclose(Q.channel_scores(R)[0], ref, rtol=1e-5)
    # groups: each group summed on its own rows only
    sc2 = Q.channel_scores(R, [0, 64, 200])
    assert np.allclose(sc2[0], (R[:64].astype(np.float64) ** 2).sum(0), rtol=1e-5)
    assert np.allclose(sc2[1], (R[64:].astype(np.float64) ** 2).sum(0), rtol=1e-5)


def test_select_matches_stable_sort_and_ties_take_lower_index():
    rng = np.random.default_rng(5)
    s = rng.integers(0, 20, size=300).astype(np.float32)    # many ties
    for k in (1, 16, 64, 300):
        ref = np.sort(np.argsort(-s, kind="stable")[:k])
        assert np.array_equal(Q.select_channels(s, k), ref)
    assert Q.select_channels(np.zeros(32, np.float32), 16).tolist() == list(range(16))


def test_second_quantization_never_increases_error_on_selected_channels():
    """Compensation invariant: |R - DQ(Q(R_sel))| <= |R| on every selected element,
    so ||X - X_hat|| does not grow there ([QUADS] 2.2 B, "Goal")."""
    rng = np.random.default_rng(6)
    d = inputs.single_linear(0)
    x = inputs.bf16_bits_to_f32(d["x"])
    r = Q.quantize_full(x, 16)
    sel = r["sel"][0]
    Rs = r["R"][:, sel]
    dqR = Q.dequantize(r["r_codes"], r["r_scales"], r["r_s_t"][0])
    d_r = (F.e4m3_decode(r["r_scales"]) * float(r["r_s_t"][0])).repeat(16, axis=1)
    slack = 2.0 ** -22 * d_r
    assert np.all(np.abs(Rs - dqR) <= np.abs(Rs) + slack)
    assert np.linalg.norm(Rs - dqR) < 0.5 * np.linalg.norm(Rs)


def test_weight_column_requant_keeps_a_block_taken_from_one_source_block():
    rng = np.random.default_rng(7)
    w = (rng.standard_normal((8, 64)) * 0.02).astype(np.float32)
    c, s, st = Q.quantize_groups(w)
    # select all 16 channels of source block 2 plus those of block 0: the new
    # blocks coincide with old blocks, so codes and scales come back unchanged
    # whenever the source block's top level is 6 (scale = max/6 exactly)
    sel = np.concatenate([np.arange(0, 16), np.arange(32, 48)])
    wc, ws = Q.requantize_weight_columns(c, s, sel)
    units_old = Q.weight_units(c, s)[:, sel]
    units_new = Q.weight_units(wc, ws)
    top6 = np.abs(F.e2m1_decode(c[:, sel])).reshape(8, 2, 16).max(axis=2) == 6.0
    for r in range(8):
        for b in range(2):
            if top6[r, b]:
                assert np.array_equal(units_new[r, b * 16:(b + 1) * 16],
                                      units_old[r, b * 16:(b + 1) * 16])
    assert top6.any()


def test_quantize_full_on_single_linear_shapes():
    d = inputs.single_linear(0)
    x = inputs.bf16_bits_to_f32(d["x"])
    r = Q.quantize_full(x, d["k"])
    assert r["codes"].shape == (64, 256) and r["scales"].shape == (64, 16)
    assert r["sel"].shape == (1, 16) and np.all(np.diff(r["sel"][0]) > 0)
    assert r["r_codes"].shape == (64, 16) and r["r_scales"].shape == (64, 1)
    # selected channels are exactly the 16 largest residual energies
    sc = r["scores"][0]
    assert sc[r["sel"][0]].min() >= np.delete(sc, r["sel"][0]).max()

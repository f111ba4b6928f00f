"""Pins for the oracle's compensated GEMM, TRACE rounding and MoE routing/combine (CPU only)."""
import json
import os

import numpy as np
import torch

from nvfp4_w4a4_quantized_quant_gb300 import inputs
from oracle import formats as F
from oracle import gemm as G
from oracle import moe as M
from oracle import nvfp4 as Q
from oracle import trace as T

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------- GEMM
def _dq_python(codes, scales, s_t):
    """Element-by-element dequantization with Python floats."""
    rows, cols = codes.shape
    out = np.zeros((rows, cols))
    for r in range(rows):
        for c in range(cols):
            out[r, c] = F.e2m1_decode(codes[r, c]) * F.e4m3_value(int(scales[r, c // 16])) * float(s_t)
    return out


def test_gemm_matches_triple_loop_on_tiny_shapes():
    rng = np.random.default_rng(0)
    x = inputs.student_t4(rng, (5, 64))
    w = (rng.standard_normal((7, 64)) * 0.02).astype(np.float32)
    xq = Q.quantize_full(x, 16)
    wc, ws, wst = Q.quantize_groups(w)
    wsc, wss = Q.requantize_weight_columns(wc, ws, xq["sel"][0])
    Y, B = G.gemm_comp(xq["codes"], xq["scales"], xq["s_t"][0], wc, ws, wst[0],
                       xq["r_codes"], xq["r_scales"], xq["r_s_t"][0], wsc, wss)
    ref = G.naive_gemm(_dq_python(xq["codes"], xq["scales"], xq["s_t"][0]),
                       _dq_python(wc, ws, wst[0]))
    ref += G.naive_gemm(_dq_python(xq["r_codes"], xq["r_scales"], xq["r_s_t"][0]),
                        _dq_python(wsc, wss, wst[0]))
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)
    assert np.all(B >= np.abs(Y) - 1e-12)


def test_gemm_exact_integer_case():
    # unit block scales (E4M3 1.0 = 0x38), tensor scales 1: Y is a sum of level products
    rng = np.random.default_rng(1)
    a = rng.integers(0, 16, size=(3, 32), dtype=np.uint8)
    b = rng.integers(0, 16, size=(4, 32), dtype=np.uint8)
    one = np.full((3, 2), 0x38, np.uint8)
    Y, _ = G.gemm_comp(a, one, 1.0, b, np.full((4, 2), 0x38, np.uint8), 1.0)
    from fractions import Fraction
    for m in range(3):
        for n in range(4):
            s = sum(Fraction(F.e2m1_decode(a[m, k]).item()) * Fraction(F.e2m1_decode(b[n, k]).item())
                    for k in range(32))
            assert Y[m, n] == float(s)


def test_compensation_is_plain_w4a4_when_residual_is_zero():
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 16, size=(8, 64), dtype=np.uint8)
    codes[:, ::16] = 7
    sb = rng.integers(0x20, 0x7F, size=(8, 4), dtype=np.uint8)
    sb[0, 0] = 0x7E
    x = (F.e2m1_decode(codes).reshape(8, -1, 16) * F.e4m3_decode(sb)[:, :, None]).reshape(8, 64)
    xq = Q.quantize_full(x.astype(np.float32), 16)
    assert not xq["r_codes"].any()
    w = (rng.standard_normal((6, 64)) * 0.02).astype(np.float32)
    wc, ws, wst = Q.quantize_groups(w)
    wsc, wss = Q.requantize_weight_columns(wc, ws, xq["sel"][0])
    Yc, _ = G.gemm_comp(xq["codes"], xq["scales"], xq["s_t"][0], wc, ws, wst[0],
                        xq["r_codes"], xq["r_scales"], xq["r_s_t"][0], wsc, wss)
    Yp, _ = G.gemm_comp(xq["codes"], xq["scales"], xq["s_t"][0], wc, ws, wst[0])
    assert np.array_equal(Yc, Yp)


def test_compensation_moves_output_toward_the_bf16_activation_reference():
    """[QUADS] 2.2 B "Goal": the correction reduces the distance between the rollout
    output and the BF16 reference (here: the same quantized weights, BF16 activations)."""
    d = inputs.single_linear(0)
    x = inputs.bf16_bits_to_f32(d["x"])
    w = inputs.bf16_bits_to_f32(d["w"])
    xq = Q.quantize_full(x, d["k"])
    wc, ws, wst = Q.quantize_groups(w)
    wsc, wss = Q.requantize_weight_columns(wc, ws, xq["sel"][0])
    Yc, _ = G.gemm_comp(xq["codes"], xq["scales"], xq["s_t"][0], wc, ws, wst[0],
                        xq["r_codes"], xq["r_scales"], xq["r_s_t"][0], wsc, wss)
    Yp, _ = G.gemm_comp(xq["codes"], xq["scales"], xq["s_t"][0], wc, ws, wst[0])
    Yref = x.astype(np.float64) @ Q.dequantize(wc, ws, wst[0]).astype(np.float64).T
    assert np.linalg.norm(Yc - Yref) < 0.9 * np.linalg.norm(Yp - Yref)


# ---------------------------------------------------------------------- TRACE
def test_trace_fixes_the_worked_boundary_example():
    """TRACE copies the rollout's rounding answer: with the rollout at 59.76 (code 2)
    the training value 60.24 (RTN code 3) is rounded to 2 and the difference of 24 vanishes."""
    g = json.load(open(os.path.join(GOLD, "trace_worked_example.json")))
    to_bf16 = lambda v: inputs.bf16_bits_to_f32(inputs.f32_to_bf16_bits(np.float32([v])))[0]  # noqa
    xr = np.zeros((1, 16), np.float32)
    xr[0, 0], xr[0, 1] = to_bf16(g["x_rollout"]), 144.0
    xt = xr.copy()
    xt[0, 0] = to_bf16(g["x_train"])
    s_t = Q.tensor_scale(xr)
    rc, rs = Q.quantize(xr, s_t)
    codes, cnt = T.trace_round(xt, rc, rs, s_t)
    assert F.e2m1_decode(codes[0, 0]) == g["rounded_levels"][1]
    assert cnt["rtn_mismatch"] == 1 and cnt["trace_mismatch"] == 0 and cnt["rtn_off_by_one"] == 1
    assert T.cross_path_difference(codes, rc, rs, s_t) == 0.0


def _trace_case(seed=0, rows=64, cols=256):
    d = inputs.trace_rounding(seed, rows, cols)
    xr = inputs.bf16_bits_to_f32(d["x_rollout"])
    xt = inputs.bf16_bits_to_f32(d["x_train"])
    rc, rs, st = Q.quantize_groups(xr)
    return xr, xt, rc, rs, st[0]


def test_trace_inequality_eq3_at_every_element():
    xr, xt, rc, rs, st = _trace_case()
    codes, cnt = T.trace_round(xt, rc, rs, st)
    v, zero = T._scaled(xt, rs, st)
    q_rtn = F.e2m1_decode(np.where(zero, 0, F.e2m1_encode(v)))
    q_roll = F.e2m1_decode(rc)
    q_tr = F.e2m1_decode(codes)
    assert np.all(np.abs(q_tr - q_roll) <= np.abs(q_rtn - q_roll))
    assert cnt["trace_mismatch"] <= cnt["rtn_mismatch"]
    assert cnt["rtn_mismatch"] > 0
    # identical paths: TRACE equals RTN equals the rollout codes
    same, c2 = T.trace_round(xr, rc, rs, st)
    assert np.array_equal(F.e2m1_decode(same), q_roll) and c2["rtn_mismatch"] == 0


def test_trace_brute_force_over_values_and_rollout_codes():
    levels = sorted(set(list(F.E2M1_LEVELS) + list(-F.E2M1_LEVELS)))
    vs = np.round(np.arange(-7.0, 7.0, 0.0625), 6).astype(np.float32)
    for rcode in range(16):
        qr = F.e2m1_decode(rcode)
        lo = np.array([max([l for l in levels if l <= max(v, -6)], default=-6) for v in vs])
        hi = np.array([min([l for l in levels if l >= min(v, 6)], default=6) for v in vs])
        exp = np.where(np.abs(lo - qr) <= np.abs(hi - qr), lo, hi)
        # feed v directly: unit scale (E4M3 1.0) and tensor scale 1.0
        x = vs.reshape(-1, 16)
        sc = np.full((x.shape[0], 1), 0x38, np.uint8)
        codes, _ = T.trace_round(x, np.full(x.shape, rcode, np.uint8), sc, 1.0)
        assert np.array_equal(F.e2m1_decode(codes).ravel(), exp)
        # zero results keep the sign of v
        z = (exp == 0)
        assert np.array_equal((codes.ravel()[z] >> 3).astype(bool), np.signbit(vs[z]))


def test_cross_path_difference_closed_form():
    rs = np.full((1, 1), 0x38, np.uint8)     # block scale 1.0
    a = np.zeros((1, 16), np.uint8)
    b = a.copy()
    b[0, 3] = 0x5                            # level 3 against level 0
    b[0, 4] = 0xC                            # level -2 against 0
    assert T.cross_path_difference(a, b, rs, 0.5) == np.sqrt((3 * 0.5) ** 2 + (2 * 0.5) ** 2)


# ------------------------------------------------------------------------ MoE
def test_route_matches_stable_argsort_and_gates_renormalise():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((40, 16)).astype(np.float32)
    logits[0, :] = 0.5                                   # all tied
    idx, gates = M.route(logits, 4)
    for t in range(40):
        ref = np.sort(np.argsort(-logits[t], kind="stable")[:4])
        assert np.array_equal(idx[t], ref)
    assert idx[0].tolist() == [0, 1, 2, 3]
    assert np.allclose(gates.sum(1), 1.0, atol=1e-6)
    ref_g = torch.softmax(torch.from_numpy(logits).double(), -1).numpy()
    ref_g = np.take_along_axis(ref_g, idx, 1)
    assert np.allclose(gates, ref_g / ref_g.sum(1, keepdims=True), rtol=1e-6)


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(100000) * 10.0 ** rng.integers(-8, 8, 100000)).astype(np.float32)
    ours = M.bf16_round(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(ours, ref)


def test_single_expert_top1_layer_reduces_to_the_dense_path():
    rng = np.random.default_rng(5)
    T_, H, Fd = 32, 64, 32
    x = inputs.student_t4(rng, (T_, H))
    w1 = (rng.standard_normal((1, 2 * Fd, H)) * 0.02).astype(np.float32)
    w2 = (rng.standard_normal((1, H, Fd)) * 0.02).astype(np.float32)
    w1q, w2q = M.quantize_weights(w1), M.quantize_weights(w2)
    res = M.moe_layer(x, np.zeros((T_, 1), np.float32), w1q, w2q, 16, 16, topk=1)
    assert np.all(res["gates"] == 1.0)
    xq = Q.quantize_full(x, 16)
    wsc, wss = Q.requantize_weight_columns(w1q[0][0], w1q[1][0], xq["sel"][0])
    y1, _ = G.gemm_comp(xq["codes"], xq["scales"], xq["s_t"][0], w1q[0][0], w1q[1][0], w1q[2][0],
                        xq["r_codes"], xq["r_scales"], xq["r_s_t"][0], wsc, wss)
    assert np.array_equal(res["y1"][0], y1)
    h = M.bf16_round(M.silu_mul(y1[:, :Fd], y1[:, Fd:]))
    assert np.array_equal(res["h"][0], h)
    assert np.array_equal(res["out"], M.bf16_round(M.bf16_round(res["y2"][0])))


def test_combine_closed_form():
    idx = np.array([[0, 2]], np.int32)
    gates = np.array([[0.25, 0.75]], np.float32)
    y = np.array([[[4.0, 8.0], [8.0, -4.0]]])
    assert M.combine(idx, gates, y).tolist() == [[7.0, -1.0]]


def test_dispatch_covers_every_slot_once():
    rng = np.random.default_rng(6)
    idx, _ = M.route(rng.standard_normal((50, 12)).astype(np.float32), 3)
    toks = M.dispatch(idx, 12)
    assert sum(len(t) for t in toks) == 150
    for e, t in enumerate(toks):
        assert np.all(np.diff(t) > 0) and all(e in idx[i] for i in t)


def test_silu_mul_matches_torch_silu_and_closed_forms():
    # an independent library: torch's SiLU in float64, on a dense grid out to +-80
    g = np.concatenate([np.linspace(-80.0, 80.0, 4001), [-1e-300, 0.0, 1e-300, 1e-3, -1e-3]])
    u = np.linspace(-3.0, 5.0, g.size)
    ref = torch.nn.functional.silu(torch.from_numpy(g)).numpy() * u
    assert np.allclose(M.silu_mul(g, u), ref, rtol=1e-14, atol=1e-300)
    one = np.ones(1)
    assert M.silu_mul(np.zeros(1), one)[0] == 0.0                       # silu(0) = 0
    assert M.silu_mul(np.array([40.0]), one)[0] / 40.0 == 1.0           # silu(g)/g -> 1
    neg = M.silu_mul(np.array([-40.0]), one)[0]                         # silu(g) -> 0 from below
    assert -1e-15 < neg < 0.0
    assert abs(neg - (-40.0 * np.exp(-40.0))) <= 1e-12 * abs(neg)
    # sigma(-g) = 1 - sigma(g)  =>  silu(-g) = silu(g) - g
    gg = np.linspace(-12.0, 12.0, 97)
    assert np.allclose(M.silu_mul(-gg, np.ones_like(gg)), M.silu_mul(gg, np.ones_like(gg)) - gg,
                       rtol=0, atol=1e-13)
    # the second operand multiplies: silu(g) * u, not silu(u) * g
    assert np.isclose(M.silu_mul(np.array([2.0]), np.array([-3.0]))[0],
                      -3.0 * 2.0 / (1.0 + np.exp(-2.0)), rtol=1e-15)


def test_w1_rows_are_gate_then_up():
    # W1 of one expert with F = 16: rows [0, 16) (gate) pick -4 * x0, rows
    # [16, 32) (up) pick +4 * x0.  With x0 = 2 the gate is -8 and the up value
    # 8, so h = silu(-8) * 8 ~ -0.0215; the swapped reading silu(8) * (-8)
    # would give ~ -7.997.  +-4 is the matrix's absolute maximum, so it is
    # represented exactly up to the float32 rounding of the scales.
    T_, H, Fd = 8, 32, 16
    x = np.zeros((T_, H), np.float32)
    x[:, 0] = 2.0
    x[:, 1] = 1.0                     # a second non-zero channel keeps the blocks non-trivial
    w1 = np.zeros((1, 2 * Fd, H), np.float32)
    w1[0, :Fd, 0] = -4.0
    w1[0, Fd:, 0] = 4.0
    w2 = np.zeros((1, H, Fd), np.float32)
    w2[0, :, 0] = 1.0
    w1q, w2q = M.quantize_weights(w1), M.quantize_weights(w2)
    res = M.moe_layer(x, np.zeros((T_, 1), np.float32), w1q, w2q, 16, 16, topk=1)
    y1 = res["y1"][0]
    assert np.allclose(y1[:, :Fd], -8.0, rtol=1e-5) and np.allclose(y1[:, Fd:], 8.0, rtol=1e-5)
    want = -8.0 / (1.0 + np.exp(8.0)) * 8.0
    assert np.allclose(res["h"][0], want, rtol=2e-2)


def test_chunk_partials_add_up_to_channel_scores():
    # groups starting at multiples of the 32-row chunk: adding a group's chunk
    # partials in ascending chunk order from 0 in float32 is the score, bit for bit
    rng = np.random.default_rng(11)
    rows, cols = 221, 48
    R = (rng.standard_normal((rows, cols)) * 10.0 ** rng.integers(-3, 3, (rows, cols))).astype(np.float32)
    offs = np.array([0, 64, 96, 192, rows], np.int32)
    part = Q.chunk_partials(R)
    assert part.shape == ((rows + 31) // 32, cols)
    scores = Q.channel_scores(R, offs)
    for g in range(len(offs) - 1):
        a, b = int(offs[g]), int(offs[g + 1])
        acc = np.zeros(cols, np.float32)
        for c in range(a // 32, (b + 31) // 32):
            acc = (acc + part[c]).astype(np.float32)
        assert np.array_equal(acc.view(np.uint32), scores[g].view(np.uint32))
    # and each partial is its own rows' sum of squares (float64 agreement)
    ref = np.add.reduceat((R.astype(np.float64) ** 2), np.arange(0, rows, 32), axis=0)
    assert np.allclose(part, ref, rtol=1e-5)

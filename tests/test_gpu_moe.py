"""GPU parity of the MoE expert layer (routing plan, gather, grouped GEMM1 with
SwiGLU, per-expert quantization and selection of h, grouped GEMM2, combine)
against the oracle.  Integer stages are bit-exact; GEMM stages use the stated
tolerance.  GEMM2 is checked with teacher forcing: the oracle quantizes the
GPU's own h, because a float32-vs-float64 difference in GEMM1 can move an h
value across a rounding boundary."""
import numpy as np
import pytest
import torch

from helpers import bf16_tensor, check_combine, codes_np, f32, unswizzle
from nvfp4_w4a4_quantized_quant_gb300 import inputs
from oracle import gemm as G
from oracle import moe as M
from oracle import nvfp4 as Q

pytestmark = pytest.mark.gpu


def _layer(lib, d, k1, k2, compensate=True):
    from nvfp4_w4a4_quantized_quant_gb300.layer import MoEExpertLayer
    E, twoF, H = d["w1"].shape
    w1 = bf16_tensor(d["w1"].reshape(E * twoF, H)).reshape(E, twoF, H)
    w2 = bf16_tensor(d["w2"].reshape(E * H, twoF // 2)).reshape(E, H, twoF // 2)
    layer = MoEExpertLayer(w1, w2, d["topk"], k1, k2, d["x"].shape[0], compensate=compensate)
    res = layer.forward(bf16_tensor(d["x"]), torch.from_numpy(d["logits"]).cuda())
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    return layer, res


def _h_tol(y1, b1, F):
    g, u = y1[:, :F], y1[:, F:]
    eg, eu = 1e-3 * b1[:, :F], 1e-3 * b1[:, F:]
    s = np.abs(M.silu_mul(g, np.ones_like(g)))
    return 1.1 * eg * (np.abs(u) + eu) + (s + 1.1 * eg) * eu + 2.0 ** -8 * np.abs(M.silu_mul(g, u)) + 1e-6


def _check_layer(lib, d, k1, k2):
    layer, res = _layer(lib, d, k1, k2)
    E, twoF, H = d["w1"].shape
    F, T, topk = twoF // 2, d["x"].shape[0], d["topk"]
    plan = res["plan"]
    xf = f32(d["x"])
    w1q, w2q = M.quantize_weights(f32(d["w1"])), M.quantize_weights(f32(d["w2"]))

    # --- weights (offline pre-quantization; W1 rows interleaved for SwiGLU tiles)
    ri = lib.swiglu_row_index(E, F, H, "cpu").numpy()
    g1c = codes_np(layer.w1q.codes, H)
    assert np.array_equal(g1c, w1q[0].reshape(E * twoF, H)[ri])
    assert np.array_equal(unswizzle(layer.w1q.scales, E * twoF, H), w1q[1].reshape(E * twoF, -1)[ri])
    assert np.array_equal(layer.w1q.tensor_scale.cpu().numpy(), w1q[2])
    assert np.array_equal(codes_np(layer.w2q.codes, F), w2q[0].reshape(E * H, F))
    assert np.array_equal(layer.w2q.tensor_scale.cpu().numpy(), w2q[2])

    # --- routing plan
    oidx, ogates = M.route(d["logits"], topk)
    assert np.array_equal(plan["idx"].cpu().numpy(), oidx)
    assert np.allclose(plan["gates"].cpu().numpy(), ogates, rtol=2e-6, atol=1e-7)
    toks = M.dispatch(oidx, E)
    cnt = plan["counts"].cpu().numpy()
    off = plan["offsets"].cpu().numpy()
    rt = plan["row_token"].cpu().numpy()
    trow = plan["token_row"].cpu().numpy()
    assert np.array_equal(cnt, [len(t) for t in toks])
    assert off[0] == 0 and np.all(np.diff(off) == (cnt + 127) // 128 * 128)
    for e in range(E):
        assert np.array_equal(rt[off[e]: off[e] + cnt[e]], toks[e])
        assert np.all(rt[off[e] + cnt[e]: off[e + 1]] == -1)
    for t in range(T):
        for j in range(topk):
            assert rt[trow[t, j]] == t and off[oidx[t, j]] <= trow[t, j] < off[oidx[t, j] + 1]

    # --- activation side of GEMM1 + gather
    ref = M.moe_layer(xf, d["logits"], w1q, w2q, k1, k2, topk)
    xq = ref["xq"]
    assert np.array_equal(res["sel1"].cpu().numpy(), xq["sel"])
    a1c = codes_np(res["a1"].codes, H)
    a1s = unswizzle(res["a1"].scales, layer.cap, H)
    live = rt[: off[E]] >= 0
    rows_live = np.nonzero(live)[0]
    assert np.array_equal(a1c[rows_live], xq["codes"][rt[rows_live]])
    assert np.array_equal(a1s[rows_live], xq["scales"][rt[rows_live]])
    pad = np.nonzero(~live)[0]
    assert not a1c[pad].any() and not a1s[pad].any()
    kp1 = lib.kpad(k1)
    r1c = codes_np(res["r1"].codes, kp1)
    assert np.array_equal(r1c[rows_live, :k1], xq["r_codes"][rt[rows_live]])

    # --- GEMM1 + SwiGLU
    h = res["h"].float().cpu().numpy().astype(np.float64)
    worst = 0.0
    for e in range(E):
        n = cnt[e]
        if n == 0:
            continue
        hg = h[off[e]: off[e] + n]
        tol = _h_tol(ref["y1"][e], ref["b1"][e], F)
        err = np.abs(hg - ref["h"][e])
        assert np.all(err <= tol), (e, err.max())
        worst = max(worst, float((err / tol).max()))
        assert not h[off[e] + n: off[e + 1]].any()

    # --- GEMM2 with teacher forcing on the GPU's h
    hov = {e: h[off[e]: off[e] + cnt[e]].astype(np.float32) for e in range(E)}
    ref2 = M.moe_layer(xf, d["logits"], w1q, w2q, k1, k2, topk, h_override=hov)
    hqc = codes_np(res["hq"].codes, F)
    hqs = unswizzle(res["hq"].scales, layer.cap, F)
    hts = res["hq"].tensor_scale.cpu().numpy()
    sel2 = res["sel2"].cpu().numpy()
    kp2 = lib.kpad(k2)
    r2c = codes_np(res["r2"].codes, kp2)
    r2ts = res["r2"].tensor_scale.cpu().numpy()
    y = res["y"].float().cpu().numpy().astype(np.float64)
    for e in range(E):
        n = cnt[e]
        hq = ref2["hq"][e]
        assert hts[e] == hq["s_t"][0]
        assert np.array_equal(sel2[e], hq["sel"][0])
        if n == 0:
            continue
        rows = slice(off[e], off[e] + n)
        assert np.array_equal(hqc[rows], hq["codes"])
        assert np.array_equal(hqs[rows], hq["scales"])
        assert r2ts[e] == hq["r_s_t"][0]
        assert np.array_equal(r2c[rows, :k2], hq["r_codes"])
        Y2, B2 = ref2["y2"][e], ref2["b2"][e]
        assert np.all(np.abs(y[rows] - Y2) <= 1e-3 * B2 + 2.0 ** -8 * np.abs(Y2) + 1e-30)

    # --- combine (the oracle's, on the GPU's gates and y)
    out = res["out"].float().cpu().numpy()
    check_combine(out, oidx, plan["gates"].cpu().numpy(), y[trow])
    return worst


def test_moe_layer_small(lib):
    d = inputs.moe_layer(0, tokens=256, hidden=256, experts=8, topk=2, ffn=128, k=16)
    _check_layer(lib, d, 16, 16)


def test_moe_layer_decode_shaped_with_empty_experts(lib):
    # 40 tokens over 16 experts, top-2: a few rows per expert, some experts empty
    d = inputs.moe_layer(1, tokens=40, hidden=256, experts=16, topk=2, ffn=128, k=32)
    d["logits"][:, 15] = -10.0                           # expert 15 never chosen
    _check_layer(lib, d, 32, 16)


def test_moe_layer_ragged_tokens_three_tiles(lib):
    d = inputs.moe_layer(2, tokens=300, hidden=512, experts=4, topk=2, ffn=256, k=64)
    _check_layer(lib, d, 64, 64)


def _check_plain_layer(lib, d, experts=None):
    """The layer without compensation (plain W4A4 both GEMMs): routing, A rows,
    h within the GEMM1 tolerance of the oracle's plain product, h's per-expert
    codes bit for bit (teacher-forced on the GPU's h), y within tolerance of the
    plain GEMM2 on those codes, and the combine."""
    layer, res = _layer(lib, d, 16, 16, compensate=False)
    E, twoF, H = d["w1"].shape
    F, topk = twoF // 2, d["topk"]
    plan = res["plan"]
    xf = f32(d["x"])
    w1q, w2q = M.quantize_weights(f32(d["w1"])), M.quantize_weights(f32(d["w2"]))
    oidx, _ = M.route(d["logits"], topk)
    assert np.array_equal(plan["idx"].cpu().numpy(), oidx)
    toks = M.dispatch(oidx, E)
    cnt = plan["counts"].cpu().numpy()
    off = plan["offsets"].cpu().numpy()
    trow = plan["token_row"].cpu().numpy()
    xc, xs, xst = Q.quantize_groups(xf)
    h = res["h"].float().cpu().numpy().astype(np.float64)
    y = res["y"].float().cpu().numpy().astype(np.float64)
    hqc = codes_np(res["hq"].codes, F)
    hqs = unswizzle(res["hq"].scales, layer.cap, F)
    hts = res["hq"].tensor_scale.cpu().numpy()
    for e in (range(E) if experts is None else experts):
        n = cnt[e]
        if n == 0:
            continue
        rows = slice(off[e], off[e] + n)
        t = toks[e]
        Y1, B1 = G.gemm_comp(xc[t], xs[t], xst[0], w1q[0][e], w1q[1][e], w1q[2][e])
        href = M.bf16_round(M.silu_mul(Y1[:, :F], Y1[:, F:]))
        assert np.all(np.abs(h[rows] - href) <= _h_tol(Y1, B1, F))
        hc, hs, hst = Q.quantize_groups(h[rows].astype(np.float32))
        assert hts[e] == hst[0]
        assert np.array_equal(hqc[rows], hc) and np.array_equal(hqs[rows], hs)
        Y2, B2 = G.gemm_comp(hc, hs, hst[0], w2q[0][e], w2q[1][e], w2q[2][e])
        assert np.all(np.abs(y[rows] - Y2) <= 1e-3 * B2 + 2.0 ** -8 * np.abs(Y2) + 1e-30)
    if experts is None:
        check_combine(res["out"].float().cpu().numpy(), oidx, plan["gates"].cpu().numpy(),
                      res["y"].float().cpu().numpy()[trow])


def test_moe_layer_plain_w4a4(lib):
    d = inputs.moe_layer(2, tokens=300, hidden=512, experts=4, topk=2, ffn=256, k=64)
    _check_plain_layer(lib, d)


def test_moe_layer_fused_activation_side_gives_the_same_outputs(lib):
    """GEMM1's activation side as one cooperative launch gives the layer the
    same outputs, bit for bit, as the quantizer and selection calls."""
    from nvfp4_w4a4_quantized_quant_gb300.layer import MoEExpertLayer
    d = inputs.moe_layer(2, tokens=300, hidden=512, experts=4, topk=2, ffn=256, k=64)
    E, twoF, H = d["w1"].shape
    w1 = bf16_tensor(d["w1"].reshape(E * twoF, H)).reshape(E, twoF, H)
    w2 = bf16_tensor(d["w2"].reshape(E * H, twoF // 2)).reshape(E, H, twoF // 2)
    x, lg = bf16_tensor(d["x"]), torch.from_numpy(d["logits"]).cuda()
    res = []
    for fused in (False, True):
        layer = MoEExpertLayer(w1, w2, d["topk"], 64, 64, d["x"].shape[0], fused_activation_side=fused)
        r = layer.forward(x, lg)
        torch.cuda.synchronize()
        assert lib.device_status() == 0
        res.append({k: r[k].clone() for k in ("out", "h", "y")} | {"sel1": r["sel1"].clone()})
    for k in res[0]:
        assert torch.equal(res[0][k], res[1][k]), k


@pytest.mark.parametrize("tokens,experts", [(300, 4), (40, 16)])
def test_moe_layer_fused_expert_side_gives_the_same_outputs(lib, tokens, experts):
    """h's per-expert quantization and selection as one launch with a block
    per expert gives the layer the same outputs, bit for bit, as the quantizer
    and selection calls (three tiles per expert, and a few rows per expert)."""
    from nvfp4_w4a4_quantized_quant_gb300.layer import MoEExpertLayer
    d = inputs.moe_layer(3, tokens=tokens, hidden=512, experts=experts, topk=2, ffn=256, k=64)
    E, twoF, H = d["w1"].shape
    w1 = bf16_tensor(d["w1"].reshape(E * twoF, H)).reshape(E, twoF, H)
    w2 = bf16_tensor(d["w2"].reshape(E * H, twoF // 2)).reshape(E, H, twoF // 2)
    x, lg = bf16_tensor(d["x"]), torch.from_numpy(d["logits"]).cuda()
    res = []
    for fused in (False, True):
        layer = MoEExpertLayer(w1, w2, d["topk"], 64, 64, tokens, fused_expert_side=fused)
        r = layer.forward(x, lg)
        torch.cuda.synchronize()
        assert lib.device_status() == 0
        used = int(r["plan"]["offsets"][-1])
        res.append({"out": r["out"].clone(), "y": r["y"][:used].clone(), "sel2": r["sel2"].clone(),
                    "hc": r["hq"].codes[:used].clone(),
                    "hs": r["hq"].scales[: used * (twoF // 32)].clone(),
                    "hts": r["hq"].tensor_scale.clone(), "r2c": r["r2"].codes.clone(),
                    "r2s": r["r2"].scales.clone(), "r2ts": r["r2"].tensor_scale.clone()})
    for k in res[0]:
        assert torch.equal(res[0][k], res[1][k]), k

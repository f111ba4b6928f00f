"""GPU parity of the MoE expert layer at the workload sizes the benchmark runs:
the 8192-token prefill layer (hidden 2048, 128 experts, top-8, FFN 768, k=64,
same launch configuration as the timed step) and the 512-token decode layer.

The oracle cannot evaluate 128 experts' float64 GEMMs in seconds, so it checks
what it can compute exactly everywhere -- the routing plan, the quantization
and selection of X, the gathered operand rows, the combine over every token
(on the GPU's y) -- and samples experts for the GEMM stages: their weights,
h (GEMM1 + SwiGLU), the per-expert quantization and selection of h, and y
(GEMM2, teacher-forced on the GPU's h as in test_gpu_moe)."""
import numpy as np
import pytest
import torch

from helpers import check_combine, codes_np, f32, unswizzle
from nvfp4_w4a4_quantized_quant_gb300 import inputs
from oracle import moe as M
from test_gpu_moe import _h_tol, _layer

pytestmark = pytest.mark.gpu


def _weights_subset(w: np.ndarray, experts):
    """Oracle NVFP4 weights with only the sampled experts filled in."""
    E, N, K = w.shape
    codes = np.zeros((E, N, K), np.uint8)
    scales = np.zeros((E, N, K // 16), np.uint8)
    st = np.zeros(E, np.float32)
    for e in experts:
        c, s, t = M.quantize_weights(f32(w[e:e + 1]))
        codes[e], scales[e], st[e] = c[0], s[0], t[0]
    return codes, scales, st


def _sampled_check(lib, d, k1, k2, experts):
    layer, res = _layer(lib, d, k1, k2)
    E, twoF, H = d["w1"].shape
    F, T, topk = twoF // 2, d["x"].shape[0], d["topk"]
    plan = res["plan"]
    xf = f32(d["x"])
    w1q, w2q = _weights_subset(d["w1"], experts), _weights_subset(d["w2"], experts)

    # --- weights of the sampled experts (W1 rows interleaved for SwiGLU tiles)
    ri = lib.swiglu_row_index(E, F, H, "cpu").numpy().reshape(E, twoF) - np.arange(E)[:, None] * twoF
    g1c = codes_np(layer.w1q.codes, H).reshape(E, twoF, H)
    g2c = codes_np(layer.w2q.codes, F).reshape(E, H, F)
    w1ts, w2ts = layer.w1q.tensor_scale.cpu().numpy(), layer.w2q.tensor_scale.cpu().numpy()
    for e in experts:
        assert np.array_equal(g1c[e], w1q[0][e][ri[e]])
        assert np.array_equal(g2c[e], w2q[0][e])
        assert w1ts[e] == w1q[2][e] and w2ts[e] == w2q[2][e]

    # --- routing plan, every token
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
    assert np.all(rt[trow] == np.arange(T)[:, None])

    # --- X: quantization, selection and the gathered operands, every row
    ref = M.moe_layer(xf, d["logits"], w1q, w2q, k1, k2, topk, experts_subset=experts)
    xq = ref["xq"]
    assert np.array_equal(res["xq"].tensor_scale.cpu().numpy(), xq["s_t"])
    assert np.array_equal(res["sel1"].cpu().numpy(), xq["sel"])
    live = np.nonzero(rt[: off[E]] >= 0)[0]
    a1c = codes_np(res["a1"].codes, H)
    assert np.array_equal(a1c[live], xq["codes"][rt[live]])
    del a1c
    a1s = unswizzle(res["a1"].scales, layer.cap, H)
    assert np.array_equal(a1s[live], xq["scales"][rt[live]])
    r1c = codes_np(res["r1"].codes, lib.kpad(k1))
    assert np.array_equal(r1c[live, :k1], xq["r_codes"][rt[live]])

    # --- GEMM1 + SwiGLU on the sampled experts
    h = res["h"].float().cpu().numpy()
    for e in experts:
        n = cnt[e]
        hg = h[off[e]: off[e] + n].astype(np.float64)
        err = np.abs(hg - ref["h"][e])
        tol = _h_tol(ref["y1"][e], ref["b1"][e], F)
        assert np.all(err <= tol), (e, float((err / tol).max()))
        assert not h[off[e] + n: off[e + 1]].any()

    # --- h quantization / selection and GEMM2, teacher-forced on the GPU's h
    hov = {e: h[off[e]: off[e] + cnt[e]].astype(np.float32) for e in experts}
    ref2 = M.moe_layer(xf, d["logits"], w1q, w2q, k1, k2, topk, experts_subset=experts, h_override=hov)
    hqc = codes_np(res["hq"].codes, F)
    hqs = unswizzle(res["hq"].scales, layer.cap, F)
    hts = res["hq"].tensor_scale.cpu().numpy()
    sel2 = res["sel2"].cpu().numpy()
    r2c = codes_np(res["r2"].codes, lib.kpad(k2))
    r2ts = res["r2"].tensor_scale.cpu().numpy()
    y = res["y"].float().cpu().numpy()
    for e in experts:
        n, hq = cnt[e], ref2["hq"][e]
        rows = slice(off[e], off[e] + n)
        assert hts[e] == hq["s_t"][0] and r2ts[e] == hq["r_s_t"][0]
        assert np.array_equal(sel2[e], hq["sel"][0])
        assert np.array_equal(hqc[rows], hq["codes"])
        assert np.array_equal(hqs[rows], hq["scales"])
        assert np.array_equal(r2c[rows, :k2], hq["r_codes"])
        Y2, B2 = ref2["y2"][e], ref2["b2"][e]
        assert np.all(np.abs(y[rows].astype(np.float64) - Y2) <= 1e-3 * B2 + 2.0 ** -8 * np.abs(Y2) + 1e-30)

    # --- combine over every token (the oracle's, on the GPU's gates and y)
    out = res["out"].float().cpu().numpy()
    gates = plan["gates"].cpu().numpy()
    for t0 in range(0, T, 512):
        ts = slice(t0, min(T, t0 + 512))
        check_combine(out[ts], oidx[ts], gates[ts], y[trow[ts]])


def test_moe_prefill_8192_tokens_sampled_experts(lib):
    d = inputs.moe_layer(0)                    # the benchmark workload's shapes and recipe
    _sampled_check(lib, d, 64, 64, experts=[0, 77, 127])


def test_moe_decode_512_tokens_sampled_experts(lib):
    d = inputs.moe_decode(0)
    _sampled_check(lib, d, 64, 64, experts=[5, 64, 100, 126])

"""MoE expert layer around the compensated W4A4 GEMMs.

[TRACE] "MoE 专家路由敏感性": each layer's router gives every token a small set
of experts by gate score.  [QUADS] section 4 / 2.2 B: the W4A4 GEMMs with
residual compensation are the MoE expert linear layers of the rollout engine.

Readings where the pages are silent:
  * routing: the top-8 logits (equal logits -> lower expert id); gate weights =
    softmax over all experts restricted to the chosen 8 and renormalised to sum
    to 1 (float64, stored as float32); each token's 8 slots are kept in
    ascending expert order;
  * dispatch order: rows grouped by expert (ascending), tokens ascending inside
    an expert;
  * expert FFN: W1 rows [0, F) are the gate projection, rows [F, 2F) the up
    projection; h = silu(g) * u with silu(g) = g / (1 + exp(-g)), computed in
    float64 and stored as bf16; W2 maps F back to the hidden size;
  * GEMM1's activation operand is the token matrix X, quantized once with one
    tensor scale and one channel selection shared by all experts; GEMM2's
    operand h is quantized per expert (own tensor scale, own selection);
  * expert outputs y are stored as bf16 and combined as
    out[t] = sum_j gate[t, j] * y[row(t, j)] in float64, ascending expert order,
    then rounded to bf16.
"""
from __future__ import annotations

import numpy as np

from . import nvfp4
from .gemm import gemm_comp


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even); returns float64.
    Normal-range values only (the layer's activations never reach bf16 subnormals)."""
    x = np.asarray(x, dtype=np.float64)
    bits = x.view(np.uint64)
    drop = np.uint64(45)                       # 52 - 7 mantissa bits dropped
    lsb = (bits >> drop) & np.uint64(1)
    rounded = (bits + (np.uint64(1) << (drop - np.uint64(1))) - np.uint64(1) + lsb) >> drop << drop
    out = rounded.view(np.float64)
    return np.where(x == 0, x, out)


def route(logits: np.ndarray, topk: int = 8):
    """Returns (expert ids int32 [T, topk] ascending, gates float32 [T, topk])."""
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    idx = np.zeros((T, topk), np.int32)
    gates = np.zeros((T, topk), np.float32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:topk]
        chosen = sorted(order)
        l64 = logits[t].astype(np.float64)
        p = np.exp(l64 - l64.max())
        p = p / p.sum()
        g = p[chosen] / p[chosen].sum()
        idx[t] = chosen
        gates[t] = g.astype(np.float32)
    return idx, gates


def dispatch(idx: np.ndarray, experts: int):
    """Token list of every expert, in ascending token order: list of int arrays."""
    return [np.nonzero((idx == e).any(axis=1))[0].astype(np.int64) for e in range(experts)]


def silu_mul(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    g = np.asarray(g, np.float64)
    return g / (1.0 + np.exp(-g)) * np.asarray(u, np.float64)


def combine(idx, gates, y_of_slot) -> np.ndarray:
    """out[t] = bf16( sum_j gates[t, j] * y_of_slot[t][j] ), j ascending (expert order)."""
    T, topk = idx.shape
    H = y_of_slot.shape[-1]
    out = np.zeros((T, H), np.float64)
    for t in range(T):
        acc = np.zeros(H, np.float64)
        for j in range(topk):
            acc = acc + float(gates[t, j]) * y_of_slot[t, j].astype(np.float64)
        out[t] = acc
    return bf16_round(out)


def quantize_weights(w: np.ndarray):
    """Per-expert NVFP4 weights: w float32 [E, N, K] -> codes [E, N, K], scales
    [E, N, K/16], tensor scales [E] (one per expert matrix)."""
    E, N, K = w.shape
    codes = np.zeros((E, N, K), np.uint8)
    scales = np.zeros((E, N, K // 16), np.uint8)
    st = np.zeros(E, np.float32)
    for e in range(E):
        c, s, t = nvfp4.quantize_groups(w[e])
        codes[e], scales[e], st[e] = c, s, t[0]
    return codes, scales, st


def expert_gemm1(xq: dict, tokens, e, w1q, k_unused=None):
    """y1 = Q(X)[tokens] Q(W1_e)^T + Q(R_sel)[tokens] Q(W1_e[:, sel])^T  (float64, [n, 2F])."""
    wc, ws, wst = w1q
    sel = xq["sel"][0]
    wsc, wss = nvfp4.requantize_weight_columns(wc[e], ws[e], sel)
    return gemm_comp(xq["codes"][tokens], xq["scales"][tokens], xq["s_t"][0],
                     wc[e], ws[e], wst[e],
                     xq["r_codes"][tokens], xq["r_scales"][tokens], xq["r_s_t"][0], wsc, wss)


def expert_gemm2(hq: dict, w2q, e):
    wc, ws, wst = w2q
    sel = hq["sel"][0]
    wsc, wss = nvfp4.requantize_weight_columns(wc[e], ws[e], sel)
    return gemm_comp(hq["codes"], hq["scales"], hq["s_t"][0], wc[e], ws[e], wst[e],
                     hq["r_codes"], hq["r_scales"], hq["r_s_t"][0], wsc, wss)


def moe_layer(x: np.ndarray, logits: np.ndarray, w1q, w2q, k1: int, k2: int, topk: int = 8,
              experts_subset=None, h_override=None):
    """The whole expert layer in float64 on quantized operands.

    x: float32 [T, H] (bf16 values); w1q/w2q: outputs of ``quantize_weights``.
    ``h_override[e]`` (optional) replaces the oracle's own h of expert e before
    its quantization -- used to compare GEMM2 on the GPU's h (teacher forcing),
    since a float32-vs-float64 difference in GEMM1 may flip an h code.
    Returns dict with routing, per-expert intermediates and (when all experts
    are evaluated) the combined output."""
    E = w1q[0].shape[0]
    F = w1q[0].shape[1] // 2
    idx, gates = route(logits, topk)
    toks = dispatch(idx, E)
    xq = nvfp4.quantize_full(x, k1)
    res = dict(idx=idx, gates=gates, tokens=toks, xq=xq, y1={}, b1={}, h={}, hq={}, y2={}, b2={})
    experts = range(E) if experts_subset is None else experts_subset
    for e in experts:
        t = toks[e]
        y1, b1 = expert_gemm1(xq, t, e, w1q)
        h = bf16_round(silu_mul(y1[:, :F], y1[:, F:]))
        res["y1"][e], res["b1"][e], res["h"][e] = y1, b1, h
        hin = h if h_override is None else h_override[e]
        hq = nvfp4.quantize_full(np.asarray(hin, np.float32), k2)
        y2, b2 = expert_gemm2(hq, w2q, e)
        res["hq"][e], res["y2"][e], res["b2"][e] = hq, y2, b2
    if experts_subset is None:
        T = x.shape[0]
        y_slot = np.zeros((T, topk, w2q[0].shape[1]), np.float64)
        for e in range(E):
            for r, t in enumerate(toks[e]):
                j = int(np.nonzero(idx[t] == e)[0][0])
                y_slot[t, j] = bf16_round(res["y2"][e][r])
        res["out"] = combine(idx, gates, y_slot)
    return res

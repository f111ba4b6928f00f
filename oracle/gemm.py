"""Compensated W4A4 product in float64 on dequantized operands.

[QUADS] 2.2 B "Mechanism": the residual correction of the selected channels is
added back to the output of the quantized product; [QUADS] section 1: the bulk
of the work stays a native W4A4 (4-bit weights, 4-bit activations) GEMM.

    Y = s_X s_W * sum_K a b  +  s_R s_W * sum_k a' b'

a, b, a', b' are the operands in block-scale units (E2M1 level times the E4M3
block-scale value); every such product is exact in float64 and the sums are a
float64 library matmul.  The bound B = the same expression on |a|, |b|, |a'|,
|b'| is returned for the per-element tolerance check.
"""
from __future__ import annotations

import numpy as np

from .formats import e2m1_decode, e4m3_decode

BLOCK = 16


def operand_units(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """[rows, cols] codes and [rows, cols/16] scale bytes -> float64 level * scale."""
    codes = np.asarray(codes, dtype=np.uint8)
    rows, cols = codes.shape
    lv = e2m1_decode(codes).reshape(rows, cols // BLOCK, BLOCK)
    return (lv * e4m3_decode(scales)[:, :, None]).reshape(rows, cols)


def gemm_comp(a_codes, a_scales, a_st, w_codes, w_scales, w_st,
              r_codes=None, r_scales=None, r_st=None, ws_codes=None, ws_scales=None):
    """Returns (Y float64 [M, N], bound float64 [M, N]).  Pass no r_*/ws_* for plain W4A4."""
    A = operand_units(a_codes, a_scales)
    W = operand_units(w_codes, w_scales)
    alpha1 = float(np.float32(a_st)) * float(np.float32(w_st))
    Y = alpha1 * (A @ W.T)
    B = alpha1 * (np.abs(A) @ np.abs(W).T)
    if r_codes is not None:
        Rq = operand_units(r_codes, r_scales)
        Ws = operand_units(ws_codes, ws_scales)
        alpha2 = float(np.float32(r_st)) * float(np.float32(w_st))
        Y = Y + alpha2 * (Rq @ Ws.T)
        B = B + alpha2 * (np.abs(Rq) @ np.abs(Ws).T)
    return Y, B


def naive_gemm(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Triple loop sum_k a[m,k] b[n,k] in float64 -- for tiny shapes only."""
    M, K = a.shape
    N = b.shape[0]
    out = np.zeros((M, N), np.float64)
    for m in range(M):
        for n in range(N):
            s = 0.0
            for kk in range(K):
                s += float(a[m, kk]) * float(b[n, kk])
            out[m, n] = s
    return out

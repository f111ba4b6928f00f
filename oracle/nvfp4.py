"""NVFP4 quantization, residual, channel scoring, top-k selection and the second
quantization of the residual slice -- written as plainly as possible.

[TRACE] "NVFP4 与 E2M1 码本": a tensor is scaled by a global (per-tensor) scale
and a per-block scale, then every value is rounded to the nearest E2M1 code.
[QUADS] 2.1: the activation quantization error is Delta X_q = X - DQ(Q(X)).
[QUADS] 2.2 B "Mechanism": the channels with the largest FP4 error ("high
residual" channels) get a second-pass quantization and the correction is added
back; "Implementation": a binary channel mask chooses the top channels by
residual magnitude.  [QUADS-news] "重点思路": the high-residual channels are
chosen online, per batch.

Readings where the pages are silent (each also listed in the design notes):
  * block = 16 consecutive elements along a row; block scale = E4M3 byte;
    tensor scale s_t = amax / (6 * 448) in float32, s_t = 1 when that is 0;
  * u_b = m_b / (6 * s_t); s_b = E4M3(u_b); d_b = E4M3value(s_b) * s_t;
    codes = E2M1(x * (1 / d_b)) -- a correctly rounded reciprocal, then a
    multiply; a block whose d_b is 0 or whose reciprocal overflows to +inf
    (tensor amax below about 2^-107) gets all codes 0x0;
  * every step is one IEEE float32 operation rounded to nearest even, no fused
    multiply-add;
  * residual magnitude of channel c = sum over the group's rows of R^2, summed
    in float32 in a fixed order: rows in chunks of 32 consecutive rows counted
    from the group's first row, each chunk summed row by row, then the chunk
    sums added in ascending chunk order;
  * top-k: largest score first, equal scores -> lower channel index; the
    selected indices are returned in ascending order;
  * the residual slice R[:, sel] is quantized as a tensor of its own (own
    tensor scale), blocks of 16 along the selected channels;
  * Q(W_sel): the weights exist only in NVFP4 on the rollout side, so W_sel is
    the dequantized weight columns DQ(Q(W))[:, sel] in units of W's tensor
    scale, requantized in new 16-blocks along the selected channels with the
    tensor scale kept at W's (so the unit tensor scale 1.0 in the formulas).
"""
from __future__ import annotations

import numpy as np

from .formats import e2m1_decode, e2m1_encode, e4m3_decode, e4m3_encode_satfinite

BLOCK = 16
E2M1_MAX = np.float32(6.0)
E4M3_MAX = np.float32(448.0)
SCORE_CHUNK_ROWS = 32

f32 = np.float32


def tensor_scale(x: np.ndarray) -> np.float32:
    """s_t = fl(amax / 2688); 1.0 when that is zero (all-zero or underflowing tensor)."""
    x = np.asarray(x, dtype=np.float32)
    amax = f32(np.max(np.abs(x))) if x.size else f32(0.0)
    s = f32(amax / f32(E2M1_MAX * E4M3_MAX))
    return s if s != 0 else f32(1.0)


def quantize(x: np.ndarray, s_t) -> tuple[np.ndarray, np.ndarray]:
    """RTN NVFP4 quantization of a [rows, cols] float32 array under tensor scale s_t.

    Returns (codes uint8 [rows, cols] -- one 4-bit code per element,
             scale bytes uint8 [rows, cols / 16]).
    """
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    assert cols % BLOCK == 0
    s_t = f32(s_t)
    xb = x.reshape(rows, cols // BLOCK, BLOCK)
    m_b = np.max(np.abs(xb), axis=2)                              # block amax (exact)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        u_b = (m_b / f32(E2M1_MAX * s_t)).astype(np.float32)      # fl(m_b / fl(6 s_t))
    s_b = e4m3_encode_satfinite(u_b)
    d_b = (e4m3_decode(s_b).astype(np.float32) * s_t).astype(np.float32)
    with np.errstate(divide="ignore"):
        r_b = (f32(1.0) / d_b).astype(np.float32)
    zero = (d_b == 0) | np.isinf(r_b)     # scale underflow: the block quantizes to 0x0
    with np.errstate(invalid="ignore"):
        v = (xb * r_b[:, :, None]).astype(np.float32)
    codes = e2m1_encode(np.where(zero[:, :, None], f32(0.0), v))
    codes = np.where(zero[:, :, None], np.uint8(0), codes)
    return codes.reshape(rows, cols).astype(np.uint8), s_b.astype(np.uint8)


def dequantize(codes: np.ndarray, scales: np.ndarray, s_t) -> np.ndarray:
    """dq = fl(level * d_b), d_b = fl(E4M3value(s_b) * s_t); float32."""
    codes = np.asarray(codes, dtype=np.uint8)
    rows, cols = codes.shape
    d_b = (e4m3_decode(scales).astype(np.float32) * f32(s_t)).astype(np.float32)
    lv = e2m1_decode(codes).astype(np.float32).reshape(rows, cols // BLOCK, BLOCK)
    return (lv * d_b[:, :, None]).astype(np.float32).reshape(rows, cols)


def residual(x: np.ndarray, codes: np.ndarray, scales: np.ndarray, s_t) -> np.ndarray:
    """R = fl(x - dq): the per-element FP4 error Delta X_q ([QUADS] 2.1)."""
    return (np.asarray(x, dtype=np.float32) - dequantize(codes, scales, s_t)).astype(np.float32)


def group_bounds(rows: int, group_offsets) -> list[tuple[int, int]]:
    if group_offsets is None:
        return [(0, rows)]
    g = [int(v) for v in group_offsets]
    return [(g[i], g[i + 1]) for i in range(len(g) - 1)]


def quantize_groups(x: np.ndarray, group_offsets=None, tensor_scales=None):
    """Quantize row groups, each with its own tensor scale.

    Returns (codes [rows, cols], scale bytes [rows, cols/16], s_t float32 [G])."""
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    bounds = group_bounds(rows, group_offsets)
    codes = np.zeros((rows, cols), np.uint8)
    scales = np.zeros((rows, cols // BLOCK), np.uint8)
    st = np.zeros(len(bounds), np.float32)
    for g, (a, b) in enumerate(bounds):
        st[g] = tensor_scale(x[a:b]) if tensor_scales is None else f32(tensor_scales[g])
        if b > a:
            codes[a:b], scales[a:b] = quantize(x[a:b], st[g])
    return codes, scales, st


def channel_scores(R: np.ndarray, group_offsets=None, chunk: int = SCORE_CHUNK_ROWS) -> np.ndarray:
    """Residual magnitude per channel and group: sum of R^2 over the group's rows,
    in the fixed float32 order stated in the module docstring.  Returns [G, cols]."""
    R = np.asarray(R, dtype=np.float32)
    rows, cols = R.shape
    bounds = group_bounds(rows, group_offsets)
    out = np.zeros((len(bounds), cols), np.float32)
    for g, (a, b) in enumerate(bounds):
        score = np.zeros(cols, np.float32)
        for c0 in range(a, b, chunk):
            acc = np.zeros(cols, np.float32)
            for r in range(c0, min(c0 + chunk, b)):
                sq = (R[r] * R[r]).astype(np.float32)
                acc = (acc + sq).astype(np.float32)
            score = (score + acc).astype(np.float32)
        out[g] = score
    return out


def chunk_partials(R: np.ndarray, end: int | None = None, chunk: int = SCORE_CHUNK_ROWS) -> np.ndarray:
    """The per-chunk sums that ``channel_scores`` adds up: row c of the result is
    the row-by-row float32 sum of R^2 over rows [32c, 32c+32) (rows < end).  Only
    meaningful when every group starts at a multiple of the chunk size."""
    R = np.asarray(R, dtype=np.float32)
    end = R.shape[0] if end is None else end
    n = (end + chunk - 1) // chunk
    out = np.zeros((n, R.shape[1]), np.float32)
    for c in range(n):
        acc = np.zeros(R.shape[1], np.float32)
        for r in range(c * chunk, min(c * chunk + chunk, end)):
            acc = (acc + (R[r] * R[r]).astype(np.float32)).astype(np.float32)
        out[c] = acc
    return out


def select_channels(scores: np.ndarray, k: int) -> np.ndarray:
    """Top-k channels by score (ties -> lower index), returned in ascending order."""
    scores = np.asarray(scores, dtype=np.float32)
    order = sorted(range(len(scores)), key=lambda c: (-float(scores[c]), c))
    return np.array(sorted(order[:k]), dtype=np.int32)


def quantize_residual_slice(R: np.ndarray, sel: np.ndarray, group_offsets=None):
    """Second-pass quantization of R[:, sel] ([QUADS] 2.2 B "Mechanism").

    ``sel`` is [G, k]: group g uses its own selected channels and its own tensor
    scale.  Returns (codes [rows, k], scale bytes [rows, k/16], s_tR [G])."""
    R = np.asarray(R, dtype=np.float32)
    rows = R.shape[0]
    sel = np.atleast_2d(np.asarray(sel, dtype=np.int64))
    k = sel.shape[1]
    assert k % BLOCK == 0
    bounds = group_bounds(rows, group_offsets)
    codes = np.zeros((rows, k), np.uint8)
    scales = np.zeros((rows, k // BLOCK), np.uint8)
    st = np.zeros(len(bounds), np.float32)
    for g, (a, b) in enumerate(bounds):
        rs = R[a:b][:, sel[g]]
        st[g] = tensor_scale(rs)
        if b > a:
            codes[a:b], scales[a:b] = quantize(rs, st[g])
    return codes, scales, st


def weight_units(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dequantized weights in units of the tensor scale: level * E4M3value(s_b), float32 (exact)."""
    codes = np.asarray(codes, dtype=np.uint8)
    rows, cols = codes.shape
    lv = e2m1_decode(codes).reshape(rows, cols // BLOCK, BLOCK)
    return (lv * e4m3_decode(scales)[:, :, None]).astype(np.float32).reshape(rows, cols)


def requantize_weight_columns(w_codes: np.ndarray, w_scales: np.ndarray, sel: np.ndarray):
    """Q(W_sel): gather the selected input channels of the NVFP4 weight and quantize
    them again in new 16-blocks along the selection, in units of W's tensor scale.
    Returns (codes [N, k], scale bytes [N, k/16])."""
    wt = weight_units(w_codes, w_scales)[:, np.asarray(sel, dtype=np.int64)]
    return quantize(wt, f32(1.0))


def quantize_full(x: np.ndarray, k: int, group_offsets=None, tensor_scales=None):
    """The whole activation side of one compensated linear, step by step:
    quantize -> residual -> channel scores -> top-k -> second quantization."""
    x = np.asarray(x, dtype=np.float32)
    codes, scales, st = quantize_groups(x, group_offsets, tensor_scales)
    bounds = group_bounds(x.shape[0], group_offsets)
    R = np.zeros_like(x)
    for g, (a, b) in enumerate(bounds):
        if b > a:
            R[a:b] = residual(x[a:b], codes[a:b], scales[a:b], st[g])
    scores = channel_scores(R, group_offsets)
    sel = np.stack([select_channels(scores[g], k) for g in range(len(bounds))])
    rcodes, rscales, rst = quantize_residual_slice(R, sel, group_offsets)
    return dict(codes=codes, scales=scales, s_t=st, R=R, scores=scores, sel=sel,
                r_codes=rcodes, r_scales=rscales, r_s_t=rst)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern (uint16), rounded to nearest, ties to even."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)).astype(np.uint16)


def qdq(x: np.ndarray, group_offsets=None, tensor_scales=None):
    """Trainer-side W4A16 fake quantization ([QUADS] 2.2 A, asymmetric QAT; 2.1
    "Weights": the trainer applies the rollout's quantize-dequantize path).
    Per row group: the NVFP4 codes and scales of `quantize`, their dequantized
    values fl(level * d_b) (`dequantize`), rounded to bf16.

    Returns (bf16 bits uint16 [rows, cols], codes, scale bytes, s_t [G])."""
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    codes, scales, st = quantize_groups(x, group_offsets, tensor_scales)
    dq = np.zeros((rows, cols), np.float32)
    for g, (a, b) in enumerate(group_bounds(rows, group_offsets)):
        if b > a:
            dq[a:b] = dequantize(codes[a:b], scales[a:b], st[g])
    return bf16_bits(dq), codes, scales, st

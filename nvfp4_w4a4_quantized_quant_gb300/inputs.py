"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module draws random numbers and rounds them to bf16 storage; it holds none
of the quantization method's arithmetic.  Every generator takes an explicit
seed and uses numpy's PCG64 bit generator, so the same seed gives the same
arrays on any host.

Workload shapes follow the pages' MoE setting (hidden 2048, 128 routed experts,
top-8, expert FFN 768) and the heavy-tailed activations that make FP4
activation error dominant (QUADS technical summary, section 2.1 "Error Analysis
and Diagnosis": activations are recomputed online and carry the largest
quantization error).  Arrays of bf16 values are returned as their uint16 bit
patterns so that nothing depends on a framework's bf16 type.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "make_rng", "f32_to_bf16_bits", "bf16_bits_to_f32", "student_t4",
    "single_linear", "dense_projection", "moe_layer", "moe_decode",
    "trace_rounding", "CONFIG_NAMES",
]

CONFIG_NAMES = ("single_linear", "dense_projection", "moe_layer", "moe_decode",
                "trace_rounding")


def make_rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns uint16 bits.

    Used only to store generated inputs in bf16; inputs are finite.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def student_t4(rng: np.random.Generator, shape) -> np.ndarray:
    """Student-t with 4 degrees of freedom: N(0,1) / sqrt(chi2_4 / 4), float32."""
    z = rng.standard_normal(shape, dtype=np.float32)
    chi2 = rng.chisquare(4.0, size=shape).astype(np.float32)
    return (z / np.sqrt(chi2 / np.float32(4.0))).astype(np.float32)


def _outlier_channels(rng, x: np.ndarray, n: int, factor: float) -> np.ndarray:
    ch = np.sort(rng.choice(x.shape[1], size=n, replace=False))
    x = x.copy()
    x[:, ch] *= np.float32(factor)
    return x, ch


def single_linear(seed: int = 0):
    """64x256 activations ~N(0,1) with 4 outlier channels x20; W 256x256 ~N(0,0.02); k=16."""
    rng = make_rng(seed)
    x = rng.standard_normal((64, 256), dtype=np.float32)
    x, ch = _outlier_channels(rng, x, 4, 20.0)
    w = (rng.standard_normal((256, 256), dtype=np.float32) * np.float32(0.02))
    return dict(name="single_linear", x=f32_to_bf16_bits(x), w=f32_to_bf16_bits(w),
                k=16, outlier_channels=ch, out_dtype="f32")


def dense_projection(seed: int = 0, rows: int = 4096, hidden: int = 2048, out: int = 6144,
                     k: int = 128):
    """Student-t(4) activations with 1% outlier channels x20; W ~N(0,0.02); k selected channels."""
    rng = make_rng(seed)
    x = student_t4(rng, (rows, hidden))
    x, ch = _outlier_channels(rng, x, max(1, hidden // 100), 20.0)
    w = rng.standard_normal((out, hidden), dtype=np.float32) * np.float32(0.02)
    return dict(name="dense_projection", x=f32_to_bf16_bits(x), w=f32_to_bf16_bits(w),
                k=k, outlier_channels=ch, out_dtype="bf16")


def moe_layer(seed: int = 0, tokens: int = 8192, hidden: int = 2048, experts: int = 128,
              topk: int = 8, ffn: int = 768, k: int = 64, with_weights: bool = True):
    """MoE expert layer input: Student-t(4) activations, N(0,1) router logits,
    W1 [E, 2*ffn, hidden] (rows [0,ffn) gate, [ffn,2ffn) up) and W2 [E, hidden, ffn], ~N(0,0.02)."""
    rng = make_rng(seed)
    x = student_t4(rng, (tokens, hidden))
    logits = rng.standard_normal((tokens, experts), dtype=np.float32)
    d = dict(name="moe_layer", x=f32_to_bf16_bits(x), logits=logits, experts=experts,
             topk=topk, ffn=ffn, hidden=hidden, k=k)
    if with_weights:
        d["w1"] = f32_to_bf16_bits(
            rng.standard_normal((experts, 2 * ffn, hidden), dtype=np.float32) * np.float32(0.02))
        d["w2"] = f32_to_bf16_bits(
            rng.standard_normal((experts, hidden, ffn), dtype=np.float32) * np.float32(0.02))
    return d


def moe_decode(seed: int = 0, **kw):
    """Decode-shaped MoE: 512 tokens (about 32 rows per expert at top-8 of 128)."""
    kw.setdefault("tokens", 512)
    d = moe_layer(seed, **kw)
    d["name"] = "moe_decode"
    return d


def trace_rounding(seed: int = 0, rows: int = 16384, cols: int = 2048):
    """Rollout activations Student-t(4); training-side copy X_train = X_rollout + N(0, (0.01|x|)^2)."""
    rng = make_rng(seed)
    xr = f32_to_bf16_bits(student_t4(rng, (rows, cols)))
    xr_f = bf16_bits_to_f32(xr)
    eps = rng.standard_normal((rows, cols), dtype=np.float32) * (np.float32(0.01) * np.abs(xr_f))
    xt = f32_to_bf16_bits(xr_f + eps)
    return dict(name="trace_rounding", x_rollout=xr, x_train=xt)

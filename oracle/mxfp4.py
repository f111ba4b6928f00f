"""MXFP4: the microscaling FP4 format ([TRACE] "技术新颖性" and "实验结果": the
method is also validated with MXFP4 W4A4 and W4A8 rollouts).

The pages give no definition; the reading here is the OCP Microscaling
format: blocks of 32 consecutive elements along a row share one scale 2^e
stored as an E8M0 byte (e + 127); elements are E2M1 codes.  Conversion of a
block with absolute maximum m > 0:
    e = floor(log2(m)) - 2        (2 = exponent of the largest E2M1 level, 6 = 1.5 * 2^2)
    e clamped to [-127, 127]
    code_i = E2M1 round-to-nearest-even of x_i / 2^e, saturating at +-6
An all-zero block gets e = -127 (byte 0) and zero codes.  Dividing by a power
of two is exact, so there is no tensor scale and no rounding before the
element encode.  Dequantized value: level * 2^e.

Test infrastructure only: the library never imports this module.
"""
from __future__ import annotations

import numpy as np

from .formats import e2m1_decode, e2m1_encode

BLOCK = 32


def scale_exponents(x: np.ndarray) -> np.ndarray:
    """e per 32-block of a [rows, cols] float32 array (int32 [rows, cols/32])."""
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    assert cols % BLOCK == 0
    m = np.max(np.abs(x.reshape(rows, cols // BLOCK, BLOCK)), axis=2).astype(np.float64)
    e = np.full(m.shape, -127, np.int64)
    nz = m > 0
    # floor(log2(m)) exactly: frexp gives m = f * 2^E with f in [0.5, 1)
    _, E = np.frexp(m[nz])
    e[nz] = np.clip(E.astype(np.int64) - 1 - 2, -127, 127)
    return e.astype(np.int32)


def quantize(x: np.ndarray):
    """-> (codes uint8 [rows, cols], E8M0 scale bytes uint8 [rows, cols/32])."""
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    e = scale_exponents(x)
    v = np.ldexp(x.reshape(rows, cols // BLOCK, BLOCK).astype(np.float64),
                 -e[:, :, None].astype(np.int64))
    codes = e2m1_encode(v.astype(np.float32)).reshape(rows, cols).astype(np.uint8)
    return codes, (e + 127).astype(np.uint8)


def dequantize(codes: np.ndarray, scale_bytes: np.ndarray) -> np.ndarray:
    """level * 2^e as float64 (exact)."""
    codes = np.asarray(codes, dtype=np.uint8)
    rows, cols = codes.shape
    e = np.asarray(scale_bytes, dtype=np.int64) - 127
    lv = e2m1_decode(codes).reshape(rows, cols // BLOCK, BLOCK).astype(np.float64)
    return np.ldexp(lv, e[:, :, None]).reshape(rows, cols)


def gemm(a_codes, a_scales, w_codes, w_scales):
    """Y = DQ(A) DQ(W)^T in float64 (every product exact), and B = |DQ(A)| |DQ(W)|^T
    for the tolerance."""
    a = dequantize(a_codes, a_scales)
    w = dequantize(w_codes, w_scales)
    return a @ w.T, np.abs(a) @ np.abs(w).T

"""Pins for the oracle's MXFP4 (OCP microscaling) quantizer and GEMM (CPU only)."""
import numpy as np

from nvfp4_w4a4_quantized_quant_gb300 import inputs
from oracle import formats as F
from oracle import mxfp4 as MX

f32 = np.float32


def test_power_of_two_block_scale_in_closed_form():
    """A block whose maximum is 6 has e = floor(log2 6) - 2 = 0 (byte 127): codes
    are plain E2M1 rounding (ties to even, saturation); a block scaled by 2^-5
    keeps the codes and lowers the byte by 5."""
    x = np.zeros((2, 32), f32)
    x[0, :8] = [6, 0.25, 0.75, 2.5, 5.0, -3.5, 1.75, -0.2]
    x[1] = x[0] * f32(2.0 ** -5)
    codes, sb = MX.quantize(x)
    assert sb[0, 0] == 127 and sb[1, 0] == 122
    want = f32([6, 0, 1, 2, 4, -4, 2, -0.0])
    assert np.array_equal(F.e2m1_decode(codes[0, :8]), want)
    assert np.array_equal(codes[0], codes[1])


def test_exponent_is_floor_log2_of_the_block_max_minus_two():
    for m, e in [(1.0, -2), (7.99, 0), (8.0, 1), (0.75, -3), (2.0 ** -130, -127), (3.0e38, 125)]:
        x = np.zeros((1, 32), f32)
        x[0, 3] = f32(m)
        assert MX.scale_exponents(x)[0, 0] == e, (m, e)
    assert MX.scale_exponents(np.zeros((1, 32), f32))[0, 0] == -127


def test_block_max_saturates_only_above_six_units():
    """The block max lands in [4, 8) units: 6.5..8 saturate to 6, 5 rounds to 4
    (tie to even), 5.5 to 6."""
    x = np.zeros((4, 32), f32)
    x[:, 0] = [7.5, 5.0, 5.5, 4.0]
    codes, sb = MX.quantize(x)
    assert np.all(sb[:, 0] == 127)
    assert list(F.e2m1_decode(codes[:, 0])) == [6.0, 4.0, 6.0, 4.0]


def test_quantization_error_bound_and_gemm_exactness():
    rng = np.random.default_rng(4)
    x = inputs.student_t4(rng, (16, 128))
    codes, sb = MX.quantize(x)
    dq = MX.dequantize(codes, sb)
    e = sb.astype(np.int64) - 127
    step = np.ldexp(1.0, e + 1).repeat(32, axis=1)          # largest gap (4 -> 6) is 2 * 2^e
    clip = np.abs(x) > np.ldexp(6.0, e).repeat(32, axis=1)
    assert np.all((np.abs(x - dq) <= step / 2 + 1e-30) | clip)
    w = rng.standard_normal((8, 128)).astype(f32)
    wc, ws = MX.quantize(w)
    Y, B = MX.gemm(codes, sb, wc, ws)
    assert np.allclose(Y, dq @ MX.dequantize(wc, ws).T, rtol=0, atol=0)
    assert np.all(np.abs(Y) <= B)


def test_trace_under_mx_scales_fixes_the_boundary_case():
    """The worked boundary example with power-of-two scales: rollout 2.49 units
    (code 2), training 2.51 units (RTN code 3) -> TRACE gives 2."""
    from oracle import trace as T
    xr = np.zeros((1, 32), f32)
    xr[0, 0], xr[0, 1] = f32(2.49 * 8), f32(6 * 8)          # block max 48 -> e = 3
    xt = xr.copy()
    xt[0, 0] = f32(2.51 * 8)
    rc, sb = MX.quantize(xr)
    assert sb[0, 0] == 130
    codes, cnt = T.trace_round_mx(xt, rc, sb)
    assert F.e2m1_decode(codes[0, 0]) == 2.0
    assert cnt["rtn_mismatch"] == 1 and cnt["trace_mismatch"] == 0

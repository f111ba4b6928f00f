"""Pins for the oracle's trainer-side W4A16 fake quantization (CPU only):
grid rounding in closed form, bf16 rounding against PyTorch's conversion,
power-of-two equivariance and per-group independence."""
import numpy as np
import torch

from nvfp4_w4a4_quantized_quant_gb300 import inputs
from oracle import nvfp4 as Q

f32 = np.float32


def _vals(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def test_unit_scale_block_rounds_to_the_e2m1_grid():
    """Tensor scale 1 and a block whose largest magnitude is 6: the block scale
    is exactly 1, so fake quantization is rounding to the grid {0, .5, 1, 1.5,
    2, 3, 4, 6} (ties to the even code, saturating, sign kept)."""
    x = f32([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -5, 0.3, 2.9, 4.9, 5.1, 0, 1.0])
    want = f32([6, 0, 1, 1, 2, 2, 4, 4, -0.0, -4, 0.5, 3, 4, 6, 0, 1])
    y, codes, scales, st = Q.qdq(x[None, :], tensor_scales=[1.0])
    assert st[0] == 1.0 and scales[0, 0] == 0x38          # E4M3 1.0
    got = _vals(y[0])
    assert np.array_equal(got, want) and np.array_equal(np.signbit(got), np.signbit(want))


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(4096).astype(f32) * f32(100),
                        (rng.standard_normal(256) * 1e-39).astype(f32),    # subnormals
                        f32([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 0.0, -0.0, 3.0e38])])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(Q.bf16_bits(x), ref)
    assert Q.bf16_bits(f32([1 + 2 ** -8]))[0] == 0x3F80          # tie -> even (down)
    assert Q.bf16_bits(f32([1 + 3 * 2 ** -8]))[0] == 0x3F82      # tie -> even (up)


def test_power_of_two_scaling_commutes_with_fake_quantization():
    rng = np.random.default_rng(6)
    x = inputs.student_t4(rng, (24, 64)) * f32(0.05)
    y1 = _vals(Q.qdq(x)[0])
    y2 = _vals(Q.qdq(x * f32(8.0))[0])
    assert np.array_equal(y1 * f32(8.0), y2)


def test_result_is_the_dequantized_rtn_value_and_within_half_a_level_step():
    rng = np.random.default_rng(7)
    x = inputs.student_t4(rng, (32, 128))
    y, codes, scales, st = Q.qdq(x)
    dq = Q.dequantize(codes, scales, st[0])
    assert np.array_equal(_vals(y), _vals(Q.bf16_bits(dq)))
    # |x - dq| is at most half the level gap at |dq| (gap 2 d_b near 6, d_b/2 near 0)
    d_b = (Q.e4m3_decode(scales).astype(np.float64) * float(st[0])).repeat(16, axis=1)
    assert np.all(np.abs(x - dq) <= d_b * 1.0 + 1e-12)


def test_groups_are_fake_quantized_independently():
    rng = np.random.default_rng(8)
    x = inputs.student_t4(rng, (96, 64))
    x[32:64] *= f32(50.0)
    offs = [0, 32, 64, 96]
    y, _, _, st = Q.qdq(x, group_offsets=offs)
    for g in range(3):
        yg, _, _, sg = Q.qdq(x[offs[g]: offs[g + 1]])
        assert sg[0] == st[g] and np.array_equal(yg, y[offs[g]: offs[g + 1]])

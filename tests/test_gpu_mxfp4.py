"""GPU parity of the MXFP4 variant (32-element blocks, E8M0 scales): quantizer
codes and scale bytes bit for bit (both layouts), its bf16 QDQ output, the
block-scaled MXFP4 GEMM against the oracle's float64 product (max |dY| <=
1e-3 * sum|a||b|), and TRACE rounding under MXFP4 rollout scales."""
import numpy as np
import pytest
import torch

from helpers import bf16_tensor, codes_np, f32, unswizzle
from nvfp4_w4a4_quantized_quant_gb300 import inputs
from oracle import mxfp4 as MX
from oracle import nvfp4 as Q
from oracle import trace as T

pytestmark = pytest.mark.gpu


def _x(name):
    rng = inputs.make_rng(31)
    if name == "t4":
        return inputs.f32_to_bf16_bits(inputs.student_t4(rng, (256, 512)))
    if name == "ragged":
        return inputs.f32_to_bf16_bits(inputs.student_t4(rng, (389, 384)) * np.float32(3))
    if name == "edge":            # zero blocks, ties, saturation, tiny and huge blocks
        x = np.zeros((40, 128), np.float32)
        x[0, :8] = [6, 0.25, 0.75, 2.5, 5.0, -3.5, 1.75, -0.2]
        x[1, :4] = [7.5, 5.0, 5.5, 4.0]
        x[2] = 1e-30 * inputs.student_t4(rng, (128,))
        x[3] = 1e30 * inputs.student_t4(rng, (128,))
        x[4, 32:64] = -0.0
        x[8:] = inputs.student_t4(rng, (32, 128))
        return inputs.f32_to_bf16_bits(x)
    raise KeyError(name)


def _sf(q, rows, cols):
    if q.layout == 1:
        return unswizzle(q.scales, rows, cols // 2)      # one scale column per 32 elements
    return q.scales.cpu().numpy().reshape(rows, cols // 32)


@pytest.mark.parametrize("name", ["t4", "ragged", "edge"])
@pytest.mark.parametrize("layout", [0, 1])
def test_mx_quantize_and_qdq_bit_exact(lib, name, layout):
    bits = _x(name)
    rows, cols = bits.shape
    q, y = lib.mx_quantize(bf16_tensor(bits), scale_layout=layout, want_qdq=True)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    oc, osb = MX.quantize(f32(bits))
    assert np.array_equal(codes_np(q.codes, cols), oc)
    assert np.array_equal(_sf(q, rows, cols), osb)
    oy = Q.bf16_bits(MX.dequantize(oc, osb).astype(np.float32))
    assert np.array_equal(y.view(torch.int16).cpu().numpy().view(np.uint16), oy)


@pytest.mark.parametrize("M,N,K", [(64, 256, 256), (200, 384, 640), (129, 128, 1024)])
def test_mx_gemm_f32(lib, M, N, K):
    rng = inputs.make_rng(M * 7 + N + K)
    xb = inputs.f32_to_bf16_bits(inputs.student_t4(rng, (M, K)))
    wb = inputs.f32_to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    a, _ = lib.mx_quantize(bf16_tensor(xb), scale_layout=1)
    w, _ = lib.mx_quantize(bf16_tensor(wb), scale_layout=1)
    y = lib.mx_gemm(a, w, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    ac, asb = MX.quantize(f32(xb))
    wc, wsb = MX.quantize(f32(wb))
    Y, B = MX.gemm(ac, asb, wc, wsb)
    yv = y.cpu().numpy().astype(np.float64)
    err = np.abs(yv - Y)
    assert np.all(err <= 1e-3 * B + 1e-30), float((err / (B + 1e-30)).max())
    assert np.linalg.norm(yv - Y) / max(np.linalg.norm(Y), 1e-30) <= 1e-5


def test_mx_gemm_dense_projection_sampled_rows(lib):
    """4096x2048 activations, 6144x2048 weights, bf16 output, 64 sampled rows."""
    d = inputs.dense_projection(0)
    a, _ = lib.mx_quantize(bf16_tensor(d["x"]), scale_layout=1)
    w, _ = lib.mx_quantize(bf16_tensor(d["w"]), scale_layout=1)
    y = lib.mx_gemm(a, w)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(1).choice(4096, 64, replace=False))
    ac, asb = MX.quantize(f32(d["x"])[rows])
    wc, wsb = MX.quantize(f32(d["w"]))
    Y, B = MX.gemm(ac, asb, wc, wsb)
    yv = y[torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(yv - Y) <= 1e-3 * B + 2.0 ** -8 * np.abs(Y) + 1e-30)


@pytest.mark.parametrize("rows,cols", [(64, 256), (16384, 2048)])
def test_trace_round_mx_bit_exact(lib, rows, cols):
    d = inputs.trace_rounding(2, rows, cols)
    rq, _ = lib.mx_quantize(bf16_tensor(d["x_rollout"]))
    codes, cnt = lib.trace_round_mx(bf16_tensor(d["x_train"]), rq)
    torch.cuda.synchronize()
    rc, rsb = MX.quantize(f32(d["x_rollout"]))
    oc, ocnt = T.trace_round_mx(f32(d["x_train"]), rc, rsb)
    assert np.array_equal(codes_np(codes, cols), oc)
    assert cnt.cpu().numpy().tolist() == [ocnt["rtn_mismatch"], ocnt["trace_mismatch"],
                                          ocnt["rtn_off_by_one"]]

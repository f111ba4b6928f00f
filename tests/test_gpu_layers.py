"""The composed layers the benchmark times: the compensated dense projection
against the oracle (sampled rows of the benchmark's 4096x2048 x 6144x2048,
k = 128 workload), and both layers replayed from a captured CUDA graph (their
side streams joined by events become graph edges) against eager calls, bit
for bit."""
import numpy as np
import pytest
import torch

from helpers import bf16_tensor, f32
from nvfp4_w4a4_quantized_quant_gb300 import inputs
from oracle import gemm as G
from oracle import nvfp4 as Q

pytestmark = pytest.mark.gpu


def _graph_of(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_compensated_linear_dense_projection(lib):
    from nvfp4_w4a4_quantized_quant_gb300.layer import CompensatedLinear
    d = inputs.dense_projection(0)
    x, w = bf16_tensor(d["x"]), bf16_tensor(d["w"])
    lin = CompensatedLinear(w, d["k"], x.shape[0])
    y = lin.forward(x).clone()
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    rows = np.sort(np.random.default_rng(3).choice(x.shape[0], 48, replace=False))
    ref = Q.quantize_full(f32(d["x"]), d["k"])
    wc, ws, wst = Q.quantize_groups(f32(d["w"]))
    wsc, wss = Q.requantize_weight_columns(wc, ws, ref["sel"][0])
    Y, B = G.gemm_comp(ref["codes"][rows], ref["scales"][rows], ref["s_t"][0], wc, ws, wst[0],
                       ref["r_codes"][rows], ref["r_scales"][rows], ref["r_s_t"][0], wsc, wss)
    yv = y[torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(yv - Y) <= 1e-3 * B + 2.0 ** -8 * np.abs(Y) + 1e-30)
    # the same call replayed from a captured graph
    g = _graph_of(lambda: lin.forward(x))
    lin.bufs["y"].zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(lin.bufs["y"], y)


def test_moe_layer_graph_replay_matches_eager(lib):
    from nvfp4_w4a4_quantized_quant_gb300.layer import MoEExpertLayer
    d = inputs.moe_layer(5, tokens=512, hidden=256, experts=16, topk=4, ffn=128, k=32)
    E, twoF, H = d["w1"].shape
    w1 = bf16_tensor(d["w1"].reshape(E * twoF, H)).reshape(E, twoF, H)
    w2 = bf16_tensor(d["w2"].reshape(E * H, twoF // 2)).reshape(E, H, twoF // 2)
    layer = MoEExpertLayer(w1, w2, d["topk"], 32, 32, 512)
    x, logits = bf16_tensor(d["x"]), torch.from_numpy(d["logits"]).cuda()
    out = layer.forward(x, logits)["out"].clone()
    h = layer.b["h"].clone()
    torch.cuda.synchronize()
    g = _graph_of(lambda: layer.forward(x, logits))
    for _ in range(2):
        layer.b["out"].zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(layer.b["out"], out)
    offs = layer.b["route"]["offsets"].cpu().numpy()
    assert torch.equal(layer.b["h"][: offs[-1]], h[: offs[-1]])
    assert lib.device_status() == 0

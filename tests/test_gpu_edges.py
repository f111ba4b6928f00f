"""Edge cases on the GPU: empty inputs are no-ops for every row-wise entry
point (PyTorch passes NULL data pointers for empty tensors), the selection of
every channel (k = K), and degenerate MoE routing (one expert taking every
token; a batch of a single token)."""
import numpy as np
import pytest
import torch

from nvfp4_w4a4_quantized_quant_gb300 import inputs
from test_gpu_gemm import _check, _oracle, _run
from test_gpu_moe import _check_layer

pytestmark = pytest.mark.gpu


def test_empty_inputs_are_noops(lib):
    dev = "cuda"
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=dev)
    for layout in (1, 0):                                   # LINEAR last: TRACE reads it
        q, part = lib.quantize_nvfp4(x, scores=True, scale_layout=layout)
    assert q.rows == 0 and part.shape[0] == 0
    sel, _, r = lib.select_residual_channels(x, q, part, 32)
    y, _ = lib.qdq_nvfp4(x, want_codes=True)
    assert y.shape == (0, 256)
    xw = torch.randn((128, 256), device=dev).to(torch.bfloat16)
    wq, _ = lib.quantize_nvfp4(xw, scale_layout=1)
    lib.weight_columns(wq)
    qa, _ = lib.quantize_nvfp4(x, scale_layout=1)
    assert lib.w4a4_gemm_comp(qa, wq, out_dtype=torch.float32).shape == (0, 128)
    mq, yq = lib.mx_quantize(x, want_qdq=True)
    mqa, _ = lib.mx_quantize(x, scale_layout=1)
    mw, _ = lib.mx_quantize(xw, scale_layout=1)
    assert lib.mx_gemm(mqa, mw).shape == (0, 128)
    codes, cnt = lib.trace_round(x, q)
    bits = lib.trace_pack_record(q)
    codes1, cnt1 = lib.trace_round_1bit(x, bits, q)
    codesm, cntm = lib.trace_round_mx(x, mq)
    logits = torch.empty((0, 16), dtype=torch.float32, device=dev)
    plan = lib.moe_route(logits, 2)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    assert cnt.sum().item() == 0 and cnt1.sum().item() == 0 and cntm.sum().item() == 0
    # no rows at all: every offset is 0 (rows past offsets[E] are outside the plan)
    assert plan["counts"].sum().item() == 0 and plan["offsets"].abs().sum().item() == 0


def test_every_channel_selected(lib):
    """k = K: the correction covers every channel (kpad = K)."""
    rng = inputs.make_rng(41)
    xb = inputs.f32_to_bf16_bits(inputs.student_t4(rng, (96, 256)))
    wb = inputs.f32_to_bf16_bits(rng.standard_normal((128, 256), dtype=np.float32) * np.float32(0.02))
    y, sel, _ = _run(lib, xb, wb, 256, torch.float32)
    torch.cuda.synchronize()
    Y, B, ref, _ = _oracle(xb, wb, 256)
    assert np.array_equal(sel.cpu().numpy()[0], np.arange(256))
    _check(y, Y, B, False)


def test_moe_layer_one_expert_takes_every_token(lib):
    d = inputs.moe_layer(3, tokens=96, hidden=256, experts=4, topk=1, ffn=128, k=16)
    d["logits"][:, 2] = 50.0                             # expert 2 wins for every token
    _check_layer(lib, d, 16, 16)


def test_moe_layer_single_token(lib):
    d = inputs.moe_layer(4, tokens=1, hidden=256, experts=8, topk=2, ffn=128, k=16)
    _check_layer(lib, d, 16, 16)


@pytest.mark.parametrize("experts,topk", [(33, 4), (64, 8), (100, 8), (200, 8), (256, 6)])
def test_routing_across_expert_counts(lib, experts, topk):
    """moe_route with 33-256 experts (one, two, four and eight 32-expert words
    per lane) against the oracle: expert ids (exact ties to the lower id),
    gates within float32 rounding, counts, padded offsets and the row maps."""
    from oracle import moe as M
    rng = inputs.make_rng(experts)
    T = 700
    logits = rng.standard_normal((T, experts)).astype(np.float32)
    logits[::7, 5] = logits[::7, 6]                 # exact ties
    logits[::11, experts - 1] = np.float32(9.0)     # the last expert always taken there
    plan = lib.moe_route(torch.from_numpy(logits).cuda(), topk)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    idx, gates = M.route(logits, topk)
    assert np.array_equal(plan["idx"].cpu().numpy(), idx)
    assert np.allclose(plan["gates"].cpu().numpy(), gates, rtol=2e-6, atol=1e-7)
    toks = M.dispatch(idx, experts)
    cnt, off = plan["counts"].cpu().numpy(), plan["offsets"].cpu().numpy()
    rt, trow = plan["row_token"].cpu().numpy(), plan["token_row"].cpu().numpy()
    assert np.array_equal(cnt, [len(t) for t in toks])
    assert off[0] == 0 and np.all(np.diff(off) == (cnt + 127) // 128 * 128)
    for e in range(experts):
        assert np.array_equal(rt[off[e]: off[e] + cnt[e]], toks[e])
        assert np.all(rt[off[e] + cnt[e]: off[e + 1]] == -1)
    assert np.all(rt[trow] == np.arange(T)[:, None])

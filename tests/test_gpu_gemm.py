"""GPU parity of the compensated W4A4 GEMM (tcgen05 block-scaled MMA) against
the oracle's float64 product: max |dY| <= 1e-3 * sum|a||b| per element and a
relative Frobenius error <= 1e-5 (float32 output); bf16 output additionally
allows its own rounding (2^-8 relative).  Q(W_sel), built inside the call, is
read back from the workspace and must match bit for bit."""
import numpy as np
import pytest
import torch

from helpers import bf16_tensor, codes_np, f32, unswizzle
from nvfp4_w4a4_quantized_quant_gb300 import inputs
from oracle import gemm as G
from oracle import nvfp4 as Q

pytestmark = pytest.mark.gpu


def _run(lib, xb, wb, k, out_dtype, comp=True):
    x, w = bf16_tensor(xb), bf16_tensor(wb)
    xq, part = lib.quantize_nvfp4(x, scores=True, scale_layout=1)
    wq, _ = lib.quantize_nvfp4(w, scale_layout=1)
    lib.weight_columns(wq)
    if not comp:
        return lib.w4a4_gemm_comp(xq, wq, out_dtype=out_dtype), None, None
    sel, _, r = lib.select_residual_channels(x, xq, part, k, r_scale_layout=1)
    N, K = wb.shape
    ws = torch.zeros(lib.workspace_size(lib.OP_GEMM, 0, K, N, k, 1), dtype=torch.uint8, device="cuda")
    y = lib.w4a4_gemm_comp(xq, wq, r, sel, k, out_dtype=out_dtype, workspace=ws)
    return y, sel, ws


def _oracle(xb, wb, k, rows=None, comp=True):
    xf, wf = f32(xb), f32(wb)
    ref = Q.quantize_full(xf, k)
    wc, ws, wst = Q.quantize_groups(wf)
    rows = slice(None) if rows is None else rows
    if not comp:
        return G.gemm_comp(ref["codes"][rows], ref["scales"][rows], ref["s_t"][0], wc, ws, wst[0]) + (ref, None)
    wsc, wss = Q.requantize_weight_columns(wc, ws, ref["sel"][0])
    Y, B = G.gemm_comp(ref["codes"][rows], ref["scales"][rows], ref["s_t"][0], wc, ws, wst[0],
                       ref["r_codes"][rows], ref["r_scales"][rows], ref["r_s_t"][0], wsc, wss)
    return Y, B, ref, (wsc, wss)


def _check(y, Y, B, bf16_out):
    yv = y.float().cpu().numpy().astype(np.float64)
    err = np.abs(yv - Y)
    tol = 1e-3 * B + (2.0 ** -8 * np.abs(Y) if bf16_out else 0.0) + 1e-30
    assert np.all(err <= tol), f"max err {err.max()} at {np.unravel_index(np.argmax(err - tol), err.shape)}"
    if not bf16_out:
        rel = np.linalg.norm(yv - Y) / max(np.linalg.norm(Y), 1e-30)
        assert rel <= 1e-5, rel
    return float(err.max())


def _check_wsel(lib, ws, N, k, oracle_wsel):
    kp = lib.kpad(k)
    raw = ws.cpu().numpy()
    codes = raw[: N * kp // 2].reshape(N, kp // 2)
    off = (N * kp // 2 + 1023) // 1024 * 1024
    sf = torch.from_numpy(raw[off: off + N * kp // 16].copy())
    from oracle.formats import unpack_nibbles
    c = unpack_nibbles(codes)
    s = unswizzle(sf, N, kp)
    wsc, wss = oracle_wsel
    assert np.array_equal(c[:, :k], wsc) and not c[:, k:].any()
    assert np.array_equal(s[:, : k // 16], wss) and not s[:, k // 16:].any()


def test_single_linear_f32(lib):
    d = inputs.single_linear(0)
    y, sel, ws = _run(lib, d["x"], d["w"], d["k"], torch.float32)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    Y, B, ref, wsel = _oracle(d["x"], d["w"], d["k"])
    assert np.array_equal(sel.cpu().numpy(), ref["sel"])
    _check(y, Y, B, False)
    _check_wsel(lib, ws, 256, d["k"], wsel)


def test_single_linear_plain_w4a4(lib):
    d = inputs.single_linear(0)
    y, _, _ = _run(lib, d["x"], d["w"], d["k"], torch.float32, comp=False)
    Y, B, _, _ = _oracle(d["x"], d["w"], d["k"], comp=False)
    _check(y, Y, B, False)


@pytest.mark.parametrize("M,N,K,k", [(200, 256, 320, 48), (1, 128, 64, 16), (129, 384, 1024, 256),
                                     (300, 128, 512, 272)])
def test_ragged_shapes_f32(lib, M, N, K, k):
    rng = inputs.make_rng(M + N + K)
    xb = inputs.f32_to_bf16_bits(inputs.student_t4(rng, (M, K)))
    wb = inputs.f32_to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    y, sel, ws = _run(lib, xb, wb, k, torch.float32)
    torch.cuda.synchronize()
    Y, B, ref, wsel = _oracle(xb, wb, k)
    assert np.array_equal(sel.cpu().numpy(), ref["sel"])
    _check(y, Y, B, False)
    _check_wsel(lib, ws, N, k, wsel)


def test_dense_projection_full_size_sampled_rows(lib):
    """4096x2048 activations, 6144x2048 weights, k=128, bf16 output -- the
    benchmark's dense configuration; 96 sampled rows checked against float64."""
    d = inputs.dense_projection(0)
    y, sel, ws = _run(lib, d["x"], d["w"], d["k"], torch.bfloat16)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(4096, 96, replace=False))
    rows[-1] = 4095
    Y, B, ref, wsel = _oracle(d["x"], d["w"], d["k"], rows)
    assert np.array_equal(sel.cpu().numpy(), ref["sel"])
    _check(y[torch.from_numpy(rows).cuda()], Y, B, True)
    _check_wsel(lib, ws, 6144, d["k"], wsel)


def test_repeat_calls_are_deterministic(lib):
    d = inputs.single_linear(0)
    y1, _, _ = _run(lib, d["x"], d["w"], d["k"], torch.float32)
    y2, _, _ = _run(lib, d["x"], d["w"], d["k"], torch.float32)
    assert torch.equal(y1, y2)


def test_prebuilt_w_sel_matches_oracle_and_the_built_in_path(lib):
    """select_weight_channels gives the oracle's Q(W_sel) bit for bit, and a GEMM
    fed that operand returns exactly the output of one that builds it itself."""
    d = inputs.single_linear(0)
    y_in, sel, _ = _run(lib, d["x"], d["w"], d["k"], torch.float32)
    wq, _ = lib.quantize_nvfp4(bf16_tensor(d["w"]), scale_layout=1)
    lib.weight_columns(wq)
    k, N = d["k"], d["w"].shape[0]
    wsel = lib.select_weight_channels(wq, sel, k)
    x = bf16_tensor(d["x"])
    xq, part = lib.quantize_nvfp4(x, scores=True, scale_layout=1)
    sel2, _, r = lib.select_residual_channels(x, xq, part, k, r_scale_layout=1)
    y_pre = lib.w4a4_gemm_comp(xq, wq, r, sel2, k, out_dtype=torch.float32, w_sel=wsel)
    torch.cuda.synchronize()
    assert torch.equal(sel, sel2) and torch.equal(y_in, y_pre)
    _, _, ref, (wsc, wss) = _oracle(d["x"], d["w"], k)
    c = codes_np(wsel.codes, wsel.cols)
    s = unswizzle(wsel.scales, N, wsel.cols)
    assert np.array_equal(c[:, :k], wsc) and not c[:, k:].any()
    assert np.array_equal(s[:, : k // 16], wss) and not s[:, k // 16:].any()


@pytest.mark.parametrize("G,N,K,k", [(3, 256, 512, 48), (2, 640, 320, 320)])
def test_select_weight_channels_per_group(lib, G, N, K, k):
    """Grouped weights with one selection per group (the MoE GEMM2 case), against
    the oracle group by group; k == K takes every column."""
    rng = inputs.make_rng(G * N + K + k)
    wb = inputs.f32_to_bf16_bits(rng.standard_normal((G * N, K), dtype=np.float32) * np.float32(0.02))
    sel = np.stack([np.sort(rng.choice(K, k, replace=False)) for _ in range(G)]).astype(np.int32)
    wq, _ = lib.quantize_nvfp4(bf16_tensor(wb), scale_layout=1, group_offsets=None)
    lib.weight_columns(wq, num_groups=G)
    out = lib.select_weight_channels(wq, torch.from_numpy(sel).cuda(), k, num_groups=G,
                                     sel_per_group=True)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    c = codes_np(out.codes, out.cols)
    s = unswizzle(out.scales, G * N, out.cols)
    wf = f32(wb)
    wc, ws, _ = Q.quantize_groups(wf)
    for g in range(G):
        rows = slice(g * N, (g + 1) * N)
        wsc, wss = Q.requantize_weight_columns(wc[rows], ws[rows], sel[g])
        assert np.array_equal(c[rows, :k], wsc) and not c[rows, k:].any()
        assert np.array_equal(s[rows, : k // 16], wss) and not s[rows, k // 16:].any()


@pytest.mark.parametrize("M,N,K,k", [(384, 256, 768, 64), (64, 128, 64, 64)])
def test_correction_shares_the_last_stage(lib, M, N, K, k):
    """K = 768 (three 256-element sub-tiles): the k-channel correction rides in
    the second slot of the last stage; K = 64: main and correction sub-tiles
    share the only stage.  M = 384 leaves the second CTA pair half-empty."""
    rng = inputs.make_rng(M * 7 + K)
    xb = inputs.f32_to_bf16_bits(inputs.student_t4(rng, (M, K)))
    wb = inputs.f32_to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    y, sel, ws = _run(lib, xb, wb, k, torch.float32)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    Y, B, ref, wsel = _oracle(xb, wb, k)
    assert np.array_equal(sel.cpu().numpy(), ref["sel"])
    _check(y, Y, B, False)


def test_gemm_wait_timeout_is_reported_and_the_device_stays_usable(lib):
    """The test hook makes the next GEMM's MMA issuer issue nothing under a 1 ms
    wait limit: its producers' and epilogue's bounded waits run out, the kernel
    reports QUADS_ERR_DEVICE_TIMEOUT and returns.  The next call is normal and
    matches the oracle."""
    # K = 4096: eight ring stages per tile, more than the ring holds, so the
    # producers also block on a free stage with their copies landed
    rng = inputs.make_rng(5)
    x = bf16_tensor(inputs.f32_to_bf16_bits(inputs.student_t4(rng, (256, 4096))))
    w = bf16_tensor(inputs.f32_to_bf16_bits(rng.standard_normal((256, 4096), dtype=np.float32)))
    xq, _ = lib.quantize_nvfp4(x, scale_layout=1)
    wq, _ = lib.quantize_nvfp4(w, scale_layout=1)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    lib.test_gemm_wait_timeout(True)
    lib.w4a4_gemm_comp(xq, wq, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert lib.device_status() == 5          # QUADS_ERR_DEVICE_TIMEOUT, read and cleared
    assert lib.device_status() == 0
    d = inputs.single_linear(0)
    y, _, _ = _run(lib, d["x"], d["w"], d["k"], torch.float32, comp=False)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    Y, B, _, _ = _oracle(d["x"], d["w"], d["k"], comp=False)
    _check(y, Y, B, False)


@pytest.mark.parametrize("policy", [1, 2])
@pytest.mark.parametrize("M,N,K,k,comp", [(200, 256, 320, 48, True), (384, 512, 768, 64, True),
                                          (129, 768, 1024, 256, True), (300, 256, 512, 16, False),
                                          (64, 256, 64, 64, True)])
def test_tile_policies_match_the_oracle(lib, policy, M, N, K, k, comp):
    """Both tile widths on shapes whose N allows 256-wide tiles: 128x128 for
    everything (policy 1), 128x256 with the correction folded into the single
    accumulator by scaling its partial sum in tensor memory (policy 2)."""
    rng = inputs.make_rng(M * 3 + N + K + policy)
    xb = inputs.f32_to_bf16_bits(inputs.student_t4(rng, (M, K)))
    wb = inputs.f32_to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    prev = lib.set_gemm_tile_policy(policy)
    try:
        y, sel, _ = _run(lib, xb, wb, k, torch.float32, comp=comp)
        torch.cuda.synchronize()
        assert lib.device_status() == 0
    finally:
        lib.set_gemm_tile_policy(prev)
    if comp:
        Y, B, ref, _ = _oracle(xb, wb, k)
        assert np.array_equal(sel.cpu().numpy(), ref["sel"])
    else:
        Y, B, _, _ = _oracle(xb, wb, k, comp=False)
    _check(y, Y, B, False)


def test_tile_policy_rejects_unknown_values(lib):
    prev = lib.set_gemm_tile_policy(0)
    try:
        with pytest.raises(ValueError):
            lib.set_gemm_tile_policy(7)
    finally:
        lib.set_gemm_tile_policy(prev)

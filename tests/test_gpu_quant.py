"""GPU parity of the activation-side kernels against the oracle: quantizer
(codes, scale bytes in both layouts, tensor scales, residual-energy partials),
channel selection and the second quantization, and TRACE rounding.  Integer
outputs must match bit for bit."""
import numpy as np
import pytest
import torch

from helpers import bf16_tensor, codes_np, f32, linear_scales
from nvfp4_w4a4_quantized_quant_gb300 import inputs
from oracle import formats as F
from oracle import nvfp4 as Q
from oracle import trace as T

pytestmark = pytest.mark.gpu


def _case(name):
    rng = inputs.make_rng(11)
    if name == "single_linear":
        return inputs.single_linear(0)["x"]
    if name == "dense_projection":
        return inputs.dense_projection(0)["x"]
    if name == "ragged":          # 3 tiles of rows + a ragged tail, 2 slabs + partial
        return inputs.f32_to_bf16_bits(inputs.student_t4(rng, (389, 320)) * np.float32(4))
    if name == "edge":            # zeros, ties, -0, saturation, huge/tiny blocks
        x = np.zeros((70, 128), np.float32)
        x[0, :4] = [60.0, 84.0, 36.0, 144.0]            # exact ties with d = 24
        x[1, :16] = -0.0
        x[2, :3] = [-0.01, 1e-3, 6.0]
        x[3] = 3.0e4 * inputs.student_t4(rng, (128,))
        x[4] = 1e-6 * inputs.student_t4(rng, (128,))
        x[5, ::16] = 448.0 * 6
        x[6:] = inputs.student_t4(rng, (64, 128))
        return inputs.f32_to_bf16_bits(x)
    if name == "zeros":
        return np.zeros((33, 64), np.uint16)
    raise KeyError(name)


CASES = ["single_linear", "ragged", "edge", "zeros", "dense_projection"]


@pytest.mark.parametrize("name", CASES)
@pytest.mark.parametrize("layout", [0, 1])
def test_quantize_bit_exact(lib, name, layout):
    bits = _case(name)
    rows, cols = bits.shape
    if layout == 1 and cols % 64:
        pytest.skip("tensor-core layout needs cols % 64 == 0")
    x = bf16_tensor(bits)
    q, part = lib.quantize_nvfp4(x, scale_layout=layout, scores=True)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    xf = f32(bits)
    oc, osc, ost = Q.quantize_groups(xf)
    assert q.tensor_scale.cpu().numpy()[0] == ost[0]
    assert np.array_equal(codes_np(q.codes, cols), oc)
    assert np.array_equal(linear_scales(q), osc)
    R = Q.residual(xf, oc, osc, ost[0])
    assert np.array_equal(part.cpu().numpy(), Q.chunk_partials(R))


def test_quantize_groups_and_row_index(lib):
    rng = inputs.make_rng(3)
    x = inputs.student_t4(rng, (256, 192))
    x[64:160] *= np.float32(50.0)
    bits = inputs.f32_to_bf16_bits(x)
    perm = rng.permutation(256).astype(np.int32)
    offs = np.array([0, 64, 160, 224, 256], np.int32)
    xt = bf16_tensor(bits)
    q, part = lib.quantize_nvfp4(xt, group_offsets=torch.from_numpy(offs).cuda(), num_groups=4,
                                 row_index=torch.from_numpy(perm).cuda(), scores=True)
    torch.cuda.synchronize()
    xp = f32(bits)[perm]
    oc, osc, ost = Q.quantize_groups(xp, offs)
    assert np.array_equal(q.tensor_scale.cpu().numpy(), ost)
    assert np.array_equal(codes_np(q.codes, 192), oc)
    assert np.array_equal(linear_scales(q), osc)
    R = np.concatenate([Q.residual(xp[a:b], oc[a:b], osc[a:b], ost[g])
                        for g, (a, b) in enumerate(zip(offs[:-1], offs[1:]))])
    assert np.array_equal(part.cpu().numpy(), Q.chunk_partials(R))


@pytest.mark.parametrize("layout", [0, 1])
def test_quantize_scores_per_expert_groups_sampled_chunks(lib, layout):
    # 128 groups of 12-25 chunks of 32 rows x 768 columns: enough (chunk,
    # 16-column block) pairs for the thread-per-pair score kernel (the shape
    # of the per-expert h quantization); every tensor scale checked, codes,
    # scales and partials on 48 sampled chunks
    rng = inputs.make_rng(21)
    sizes = 32 * rng.integers(12, 26, 128)
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows, cols = int(offs[-1]), 768
    x = inputs.student_t4(rng, (rows, cols))
    x *= np.repeat(np.float32(2.0) ** rng.integers(-3, 4, 128).astype(np.float32), sizes)[:, None]
    bits = inputs.f32_to_bf16_bits(x)
    q, part = lib.quantize_nvfp4(bf16_tensor(bits), group_offsets=torch.from_numpy(offs).cuda(),
                                 num_groups=128, scale_layout=layout, scores=True)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    xf = f32(bits)
    ts = q.tensor_scale.cpu().numpy()
    for g in range(128):
        assert ts[g] == Q.tensor_scale(xf[offs[g]:offs[g + 1]])
    codes = codes_np(q.codes, cols)
    scales = linear_scales(q)
    pc = part.cpu().numpy()
    for ch in rng.choice(rows // 32, 48, replace=False):
        a, b = 32 * ch, 32 * ch + 32
        g = int(np.searchsorted(offs, a, side="right") - 1)
        oc, osc = Q.quantize(xf[a:b], ts[g])
        assert np.array_equal(codes[a:b], oc)
        assert np.array_equal(scales[a:b], osc)
        R = Q.residual(xf[a:b], oc, osc, ts[g])
        assert np.array_equal(pc[ch:ch + 1], Q.chunk_partials(R))


def _padded_groups(rng, counts, tile, cols):
    """Row groups of `counts` real rows, each padded up to a multiple of
    `tile` rows (at least one tile), the padding filled with nonzero values;
    returns (x with garbage padding, x with zero padding, offsets)."""
    sizes = np.maximum((counts + tile - 1) // tile, 1) * tile
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    x = inputs.student_t4(rng, (int(offs[-1]), cols))
    xz = x.copy()
    for g, c in enumerate(counts):
        xz[offs[g] + c:offs[g + 1]] = 0.0
    return x, xz, offs


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("scores", [False, True])
@pytest.mark.parametrize("many", [False, True])
def test_quantize_group_counts_take_padding_rows_as_zero(lib, layout, scores, many):
    """With group_counts, rows past each group's count are zero rows whatever
    they hold: the amax pass, codes, scales and score partials equal the
    oracle's on x with those rows zeroed (and the call without counts on that
    zeroed x), on the 32x256-task quantizer; `many`: 300 groups of 32-row
    tiles (more groups than the kernel caches in shared memory), counts
    outside [0, size] included."""
    rng = inputs.make_rng(12)
    if many:
        sizes = 32 * rng.integers(1, 3, 300)
        counts = rng.integers(-3, 80, 300).astype(np.int32)   # below 0 and past the size too
        offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
        x = inputs.student_t4(rng, (int(offs[-1]), 256))
        xz = x.copy()
        for g in range(300):
            xz[offs[g] + min(max(int(counts[g]), 0), int(sizes[g])):offs[g + 1]] = 0.0
    else:
        counts = np.array([5, 0, 128, 33, 64, 100, 250], np.int32)
        x, xz, offs = _padded_groups(rng, counts, 128, 256)
    G = len(counts)
    bits, bz = inputs.f32_to_bf16_bits(x), inputs.f32_to_bf16_bits(xz)
    ot, ct = torch.from_numpy(offs).cuda(), torch.from_numpy(counts).cuda()
    q, part = lib.quantize_nvfp4(bf16_tensor(bits), group_offsets=ot, num_groups=G, group_counts=ct,
                                 scores=scores, scale_layout=layout)
    qz, partz = lib.quantize_nvfp4(bf16_tensor(bz), group_offsets=ot, num_groups=G, scores=scores,
                                   scale_layout=layout)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    assert torch.equal(q.codes, qz.codes) and torch.equal(q.scales, qz.scales)
    assert torch.equal(q.tensor_scale, qz.tensor_scale)
    xf = f32(bz)
    oc, osc, ost = Q.quantize_groups(xf, offs)
    assert np.array_equal(q.tensor_scale.cpu().numpy(), ost)
    assert np.array_equal(codes_np(q.codes, 256), oc)
    assert np.array_equal(linear_scales(q), osc)
    if scores:
        assert torch.equal(part, partz)
        R = np.concatenate([Q.residual(xf[a:b], oc[a:b], osc[a:b], ost[g])
                            for g, (a, b) in enumerate(zip(offs[:-1], offs[1:]))])
        assert np.array_equal(part.cpu().numpy(), Q.chunk_partials(R))


def test_quantize_group_counts_thread_per_chunk_kernel(lib):
    """The same rule on the thread-per-(chunk, block) score kernel (the shape
    of the per-expert h quantization: 128 groups of up to 512 rows x 768),
    with the groups' amax given as in the layer: bit-equal to the call without
    counts on the zeroed input, the oracle checked on sampled chunks, padding
    chunks included."""
    rng = inputs.make_rng(13)
    counts = rng.integers(300, 513, 128).astype(np.int32)   # enough pairs for that kernel
    counts[:4] = [0, 1, 512, 31]
    x, xz, offs = _padded_groups(rng, counts, 128, 768)
    bits, bz = inputs.f32_to_bf16_bits(x), inputs.f32_to_bf16_bits(xz)
    xf = f32(bz)
    amax = np.array([np.abs(xf[a:b]).max() if b > a else 0.0
                     for a, b in zip(offs[:-1], offs[1:])], np.float32)
    ot, ct = torch.from_numpy(offs).cuda(), torch.from_numpy(counts).cuda()
    at = torch.from_numpy(amax).cuda()
    q, part = lib.quantize_nvfp4(bf16_tensor(bits), group_offsets=ot, num_groups=128, group_counts=ct,
                                 tensor_amax_in=at, scores=True, scale_layout=1)
    qz, partz = lib.quantize_nvfp4(bf16_tensor(bz), group_offsets=ot, num_groups=128,
                                   tensor_amax_in=at, scores=True, scale_layout=1)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    assert torch.equal(q.codes, qz.codes) and torch.equal(q.scales, qz.scales)
    assert torch.equal(part, partz)
    ts = q.tensor_scale.cpu().numpy()
    codes, scales, pc = codes_np(q.codes, 768), linear_scales(q), part.cpu().numpy()
    pad_chunks = [c for g in range(128) for c in range((offs[g] + counts[g] + 31) // 32, offs[g + 1] // 32)]
    sample = list(rng.choice(int(offs[-1]) // 32, 24, replace=False)) + pad_chunks[:8]
    for ch in sample:
        a, b = 32 * ch, 32 * ch + 32
        g = int(np.searchsorted(offs, a, side="right") - 1)
        oc, osc = Q.quantize(xf[a:b], ts[g])
        assert np.array_equal(codes[a:b], oc) and np.array_equal(scales[a:b], osc)
        assert np.array_equal(pc[ch:ch + 1], Q.chunk_partials(Q.residual(xf[a:b], oc, osc, ts[g])))


def test_quantize_given_tensor_scale(lib):
    bits = _case("ragged")
    x = bf16_tensor(bits)
    ts = torch.tensor([0.0123], dtype=torch.float32, device="cuda")
    q, _ = lib.quantize_nvfp4(x, tensor_scale_in=ts)
    oc, osc = Q.quantize(f32(bits), np.float32(0.0123))
    assert np.array_equal(codes_np(q.codes, bits.shape[1]), oc)
    assert np.array_equal(linear_scales(q), osc)


@pytest.mark.parametrize("name,k,layout", [("single_linear", 16, 0), ("ragged", 48, 1),
                                           ("dense_projection", 128, 1), ("edge", 32, 0),
                                           ("zeros", 16, 0)])
def test_select_and_second_quantization_bit_exact(lib, name, k, layout):
    bits = _case(name)
    rows, cols = bits.shape
    if layout == 1 and cols % 64:
        layout = 0
    x = bf16_tensor(bits)
    q, part = lib.quantize_nvfp4(x, scores=True, scale_layout=layout)
    sel, scores, r = lib.select_residual_channels(x, q, part, k, r_scale_layout=layout,
                                                  want_scores=True)
    torch.cuda.synchronize()
    ref = Q.quantize_full(f32(bits), k)
    assert np.array_equal(scores.cpu().numpy(), ref["scores"])
    assert np.array_equal(sel.cpu().numpy(), ref["sel"])
    assert r.tensor_scale.cpu().numpy()[0] == ref["r_s_t"][0]
    kp = lib.kpad(k)
    rc = codes_np(r.codes, kp)
    assert np.array_equal(rc[:, :k], ref["r_codes"]) and not rc[:, k:].any()
    rs = linear_scales(r, rows, kp)
    assert np.array_equal(rs[:, : k // 16], ref["r_scales"]) and not rs[:, k // 16:].any()


def test_select_per_group(lib):
    rng = inputs.make_rng(5)
    x = inputs.student_t4(rng, (320, 256))
    x[:, 7] *= 30
    x[128:, 200] *= 30
    bits = inputs.f32_to_bf16_bits(x)
    offs = np.array([0, 128, 256, 320], np.int32)
    ot = torch.from_numpy(offs).cuda()
    xt = bf16_tensor(bits)
    q, part = lib.quantize_nvfp4(xt, group_offsets=ot, num_groups=3, scores=True, scale_layout=1)
    sel, _, r = lib.select_residual_channels(xt, q, part, 32, group_offsets=ot, num_groups=3,
                                             r_scale_layout=1)
    torch.cuda.synchronize()
    ref = Q.quantize_full(f32(bits), 32, offs)
    assert np.array_equal(sel.cpu().numpy(), ref["sel"])
    assert np.array_equal(r.tensor_scale.cpu().numpy(), ref["r_s_t"])
    assert np.array_equal(codes_np(r.codes, 64)[:, :32], ref["r_codes"])
    assert np.array_equal(linear_scales(r, 320, 64)[:, :2], ref["r_scales"])


@pytest.mark.parametrize("rows,cols", [(64, 256), (1000, 512), (16384, 2048)])
def test_trace_round_bit_exact(lib, rows, cols):
    d = inputs.trace_rounding(0, rows, cols)
    xr, xt = bf16_tensor(d["x_rollout"]), bf16_tensor(d["x_train"])
    rq, _ = lib.quantize_nvfp4(xr)
    codes, cnt = lib.trace_round(xt, rq)
    torch.cuda.synchronize()
    xrf, xtf = f32(d["x_rollout"]), f32(d["x_train"])
    rc, rs, st = Q.quantize_groups(xrf)
    oc, ocnt = T.trace_round(xtf, rc, rs, st[0])
    assert np.array_equal(codes_np(codes, cols), oc)
    c = cnt.cpu().numpy().tolist()
    assert c == [ocnt["rtn_mismatch"], ocnt["trace_mismatch"], ocnt["rtn_off_by_one"]]
    assert c[1] <= c[0]


def test_trace_worked_example_on_gpu(lib):
    xr = np.zeros((1, 16), np.float32)
    xr[0, 0], xr[0, 1] = 59.75, 144.0
    xt = xr.copy()
    xt[0, 0] = 60.25
    rq, _ = lib.quantize_nvfp4(bf16_tensor(inputs.f32_to_bf16_bits(xr)))
    codes, cnt = lib.trace_round(bf16_tensor(inputs.f32_to_bf16_bits(xt)), rq)
    assert F.e2m1_decode(codes_np(codes, 16)[0, 0]) == 2.0
    assert cnt.cpu().tolist() == [1, 0, 1]


def test_conversions_exhaustive_against_oracle(lib):
    """Every bf16 bit pattern through the quantizer with unit scales: each block
    holds 6*448 so s_t = 1, and the block scale is 448 -> d = 448."""
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = f32(allb)
    keep = np.isfinite(v) & (np.abs(v) <= 2688)
    vals = allb[keep]
    n = (len(vals) + 14) // 15 * 15
    vals = np.concatenate([vals, np.zeros(n - len(vals), np.uint16)]).reshape(-1, 15)
    big = inputs.f32_to_bf16_bits(np.full((vals.shape[0], 1), 2688.0, np.float32))
    bits = np.concatenate([big, vals], axis=1)
    q, _ = lib.quantize_nvfp4(bf16_tensor(bits))
    oc, osc, _ = Q.quantize_groups(f32(bits))
    assert np.array_equal(codes_np(q.codes, 16), oc)
    assert np.array_equal(linear_scales(q), osc)


def test_block_scale_encoding_exhaustive(lib):
    """Every bf16 magnitude as a block maximum under tensor scale 1: scale byte = E4M3(m / 6)."""
    allb = np.arange(1 << 15, dtype=np.uint32).astype(np.uint16)      # sign bit clear
    v = f32(allb)
    vals = allb[np.isfinite(v)]
    bits = np.zeros((len(vals), 16), np.uint16)
    bits[:, 0] = vals
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    q, _ = lib.quantize_nvfp4(bf16_tensor(bits), tensor_scale_in=one)
    oc, osc = Q.quantize(f32(bits), np.float32(1.0))
    assert np.array_equal(linear_scales(q), osc)
    assert np.array_equal(codes_np(q.codes, 16), oc)


@pytest.mark.parametrize("name", ["single_linear", "ragged", "edge", "zeros"])
def test_w4a16_qdq_bit_exact(lib, name):
    """Trainer-side fake quantization: bf16 output, codes and scales bit for bit."""
    bits = _case(name)
    rows, cols = bits.shape
    x = bf16_tensor(bits)
    y, q = lib.qdq_nvfp4(x, want_codes=True)
    y_only, _ = lib.qdq_nvfp4(x)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    oy, oc, osc, ost = Q.qdq(f32(bits))
    got = y.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oy)
    assert torch.equal(y, y_only)
    assert q.tensor_scale.cpu().numpy()[0] == ost[0]
    assert np.array_equal(codes_np(q.codes, cols), oc)
    assert np.array_equal(linear_scales(q), osc)


def test_w4a16_qdq_per_expert_groups_and_given_scale(lib):
    """Expert-stacked weights (one tensor scale per expert) and a given scale."""
    rng = inputs.make_rng(21)
    w = rng.standard_normal((3 * 128, 192), dtype=np.float32) * np.float32(0.02)
    w[128:256] *= np.float32(7.0)
    bits = inputs.f32_to_bf16_bits(w)
    offs = np.array([0, 128, 256, 384], np.int32)
    x = bf16_tensor(bits)
    y, q = lib.qdq_nvfp4(x, group_offsets=torch.from_numpy(offs).cuda(), num_groups=3,
                         want_codes=True, scale_layout=1)
    ts = torch.tensor([2.0 ** -9], dtype=torch.float32, device="cuda")
    y2, _ = lib.qdq_nvfp4(x, tensor_scale_in=ts)
    torch.cuda.synchronize()
    oy, oc, osc, ost = Q.qdq(f32(bits), group_offsets=offs)
    assert np.array_equal(y.view(torch.int16).cpu().numpy().view(np.uint16), oy)
    assert np.array_equal(q.tensor_scale.cpu().numpy(), ost)
    assert np.array_equal(linear_scales(q), osc)
    oy2 = Q.qdq(f32(bits), tensor_scales=[2.0 ** -9])[0]
    assert np.array_equal(y2.view(torch.int16).cpu().numpy().view(np.uint16), oy2)


@pytest.mark.parametrize("rows,cols", [(64, 256), (389, 320), (16384, 2048)])
def test_trace_record_and_1bit_round_bit_exact(lib, rows, cols):
    """Mantissa-only record and the rounding it guides, against the oracle; the
    16384x2048 case is the benchmark's TRACE workload."""
    d = inputs.trace_rounding(1, rows, cols)
    xr, xt = bf16_tensor(d["x_rollout"]), bf16_tensor(d["x_train"])
    rq, _ = lib.quantize_nvfp4(xr)
    bits = lib.trace_pack_record(rq)
    codes, cnt = lib.trace_round_1bit(xt, bits, rq)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    xrf, xtf = f32(d["x_rollout"]), f32(d["x_train"])
    rc, rs, st = Q.quantize_groups(xrf)
    obits = T.pack_record(rc)
    assert np.array_equal(bits.cpu().numpy(), obits)
    oc, ocnt = T.trace_round_1bit(xtf, obits, rs, st[0])
    assert np.array_equal(codes_np(codes, cols), oc)
    assert cnt.cpu().numpy().tolist() == [ocnt["changed"], ocnt["bit_mismatch"]]


def test_trace_1bit_worked_example_on_gpu(lib):
    xr = np.zeros((1, 16), np.float32)
    xr[0, 0], xr[0, 1] = 59.75, 144.0
    xt = xr.copy()
    xt[0, 0] = 60.25
    rq, _ = lib.quantize_nvfp4(bf16_tensor(inputs.f32_to_bf16_bits(xr)))
    bits = lib.trace_pack_record(rq)
    codes, cnt = lib.trace_round_1bit(bf16_tensor(inputs.f32_to_bf16_bits(xt)), bits, rq)
    assert F.e2m1_decode(codes_np(codes, 16)[0, 0]) == 2.0
    assert cnt.cpu().tolist() == [1, 0]


@pytest.mark.parametrize("layout", [0, 1])
def test_select_many_groups_one_block_per_group(lib, layout):
    """40 row groups (the per-expert shape: one selection and one R_sel tensor
    scale per group), with empty groups, uneven sizes and capacity rows past the
    last offset, which must come out as zero codes and scales."""
    rng = inputs.make_rng(9)
    sizes = rng.choice([0, 32, 64, 96, 160, 256], size=40)
    sizes[[3, 17]] = 0
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    end, cap = int(offs[-1]), int(offs[-1]) + 200
    x = inputs.student_t4(rng, (cap, 256))
    x[:, 11] *= 25
    bits = inputs.f32_to_bf16_bits(x)
    ot = torch.from_numpy(offs).cuda()
    xt = bf16_tensor(bits)
    q, part = lib.quantize_nvfp4(xt, group_offsets=ot, num_groups=40, scores=True, scale_layout=layout)
    sel, _, r = lib.select_residual_channels(xt, q, part, 32, group_offsets=ot, num_groups=40,
                                             r_scale_layout=layout)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    ref = Q.quantize_full(f32(bits[:end]), 32, offs)
    assert np.array_equal(sel.cpu().numpy(), ref["sel"])
    assert np.array_equal(r.tensor_scale.cpu().numpy(), ref["r_s_t"])
    rc = codes_np(r.codes, 64)
    rsc = linear_scales(r, cap, 64)
    assert np.array_equal(rc[:end, :32], ref["r_codes"]) and not rc[:end, 32:].any()
    assert np.array_equal(rsc[:end, :2], ref["r_scales"]) and not rsc[:end, 2:].any()
    assert not rc[end:].any() and not rsc[end:].any()


@pytest.mark.parametrize("rows,cols,k,groups", [
    (64, 512, 64, 1),       # one group, scores formed by the top-k block
    (64, 512, 400, 1),      # more channels than non-zero scores: zero-score ties
    (2112, 512, 64, 1),     # long group: scores from the score chain first
    (64, 4096, 64, 1),      # more than 2048 channels: 8 channels per thread
    (96, 512, 32, 3),       # row groups
])
def test_select_ties_take_lowest_index(lib, rows, cols, k, groups):
    """Repeated 16-channel blocks give channels with equal scores and zero
    blocks give zero scores, so the k-th largest score is tied: the selection
    takes every larger score and then the lowest channel indices among the
    equal ones, as the oracle does."""
    rng = inputs.make_rng(77)
    distinct = inputs.student_t4(rng, (rows, 64))
    x = np.zeros((rows, cols), np.float32)
    live = (cols // 16) * 3 // 4
    for b in range(live):
        x[:, 16 * b:16 * b + 16] = distinct[:, 16 * (b % 4):16 * (b % 4) + 16]
    bits = inputs.f32_to_bf16_bits(x)
    xt = bf16_tensor(bits)
    if groups > 1:
        offs = np.arange(groups + 1, dtype=np.int32) * (rows // groups)
        ot = torch.from_numpy(offs).cuda()
        q, part = lib.quantize_nvfp4(xt, group_offsets=ot, num_groups=groups, scores=True)
        sel, _, _ = lib.select_residual_channels(xt, q, part, k, group_offsets=ot, num_groups=groups)
        ref = Q.quantize_full(f32(bits), k, offs)
    else:
        q, part = lib.quantize_nvfp4(xt, scores=True)
        sel, _, _ = lib.select_residual_channels(xt, q, part, k)
        ref = Q.quantize_full(f32(bits), k)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    sc = ref["scores"].reshape(groups, cols)
    got = sel.cpu().numpy().reshape(groups, k)
    for g in range(groups):
        kth = np.sort(sc[g])[::-1][k - 1]
        assert (sc[g] == kth).sum() > 1   # the case really has a tie at the threshold
    assert np.array_equal(got, ref["sel"].reshape(groups, k))


def test_w4a16_qdq_full_expert_stack_sampled_experts(lib):
    """The benchmark's QDQ configuration: the 128 experts' gate/up weights
    (196608 x 2048, one tensor scale per expert); three experts checked bit for
    bit (their groups are quantized independently of the others)."""
    E, R, H = 128, 1536, 2048
    g = torch.Generator(device="cuda")
    g.manual_seed(2)
    w = (torch.randn((E * R, H), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    offs = torch.arange(0, E * R + 1, R, dtype=torch.int32, device="cuda")
    y, q = lib.qdq_nvfp4(w, group_offsets=offs, num_groups=E, want_codes=True)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    ts = q.tensor_scale.cpu().numpy()
    for e in (0, 63, 127):
        rows = slice(e * R, (e + 1) * R)
        bits = w[rows].view(torch.int16).cpu().numpy().view(np.uint16)
        oy, oc, osc, ost = Q.qdq(f32(bits))
        assert ts[e] == ost[0]
        assert np.array_equal(y[rows].view(torch.int16).cpu().numpy().view(np.uint16), oy)
        assert np.array_equal(codes_np(q.codes[rows], H), oc)


@pytest.mark.parametrize("rows,cols,k,layout", [(8192, 2048, 64, 0), (4096, 2048, 128, 1),
                                                (512, 2048, 64, 1), (300, 256, 16, 0),
                                                (77, 512, 64, 1)])
def test_fused_quantize_select_matches_the_two_calls(lib, rows, cols, k, layout):
    """The cooperative quantize + select kernel gives exactly the outputs of
    quantize_nvfp4 (scores on) followed by select_residual_channels (grids of
    every SM's blocks down to one block per 32x256 task: 128, 10 and 6)."""
    rng = inputs.make_rng(rows + cols + k)
    xf = inputs.student_t4(rng, (rows, cols))
    xf[:, rng.choice(cols, max(1, cols // 100), replace=False)] *= np.float32(20.0)
    x = bf16_tensor(inputs.f32_to_bf16_bits(xf))
    q, part = lib.quantize_nvfp4(x, scores=True, scale_layout=layout)
    sel, sc, r = lib.select_residual_channels(x, q, part, k, r_scale_layout=layout, want_scores=True)
    fq, fsel, fsc, fr = lib.quantize_select_nvfp4(x, k, scale_layout=layout, r_scale_layout=layout,
                                                  want_scores=True)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    assert torch.equal(fq.codes, q.codes) and torch.equal(fq.scales, q.scales)
    assert torch.equal(fq.tensor_scale, q.tensor_scale)
    assert torch.equal(fsc, sc) and torch.equal(fsel, sel)
    assert torch.equal(fr.codes, r.codes) and torch.equal(fr.scales, r.scales)
    assert torch.equal(fr.tensor_scale, r.tensor_scale)
    if rows <= 300:
        ref = Q.quantize_full(f32(inputs.f32_to_bf16_bits(xf)), k)
        assert np.array_equal(fsel.cpu().numpy(), ref["sel"])
        assert np.array_equal(codes_np(fr.codes, lib.kpad(k))[:, :k], ref["r_codes"])


def test_quantize_scores_large_input_sampled_chunks(lib):
    """65536 x 2048 with score partials: enough (chunk, 16-column block) pairs
    that the thread-per-pair kernel keeps four rows of loads in flight; the
    tensor scale against its definition on the input's max |x|, and codes,
    scales and partials against the oracle on 24 sampled chunks (the last
    one included)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(31)
    rows, cols = 65536, 2048
    x = (torch.randn((rows, cols), generator=g, device="cuda") *
         torch.exp2(torch.randint(-3, 4, (rows, 1), generator=g, device="cuda").float())).to(torch.bfloat16)
    q, part = lib.quantize_nvfp4(x, scores=True)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    amax = np.float32(x.abs().max().float().item())
    ts = q.tensor_scale.cpu().numpy()[0]
    assert ts == Q.tensor_scale(np.array([amax], np.float32))   # the oracle on the maximum alone
    rng = inputs.make_rng(31)
    for ch in list(rng.choice(rows // 32 - 1, 23, replace=False)) + [rows // 32 - 1]:
        a, b = 32 * int(ch), 32 * int(ch) + 32
        xf = x[a:b].float().cpu().numpy()
        oc, osc = Q.quantize(xf, ts)
        assert np.array_equal(codes_np(q.codes[a:b], cols), oc)
        assert np.array_equal(q.scales.cpu().numpy().reshape(rows, cols // 16)[a:b], osc)
        R = Q.residual(xf, oc, osc, ts)
        assert np.array_equal(part[int(ch):int(ch) + 1].cpu().numpy(), Q.chunk_partials(R))

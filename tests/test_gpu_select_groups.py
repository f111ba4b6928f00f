"""GPU parity of quads_quantize_select_groups_nvfp4 (one block per row group:
the group's quantization, channel scores, top-k and the second quantization
of R_sel in one launch): bit for bit against the oracle on the groups' real
rows, and against the quantizer + selection calls it stands for, on padded
groups whose padding rows hold garbage (the counts make them zero rows)."""
import numpy as np
import pytest
import torch

from helpers import bf16_tensor, codes_np, f32, linear_scales
from nvfp4_w4a4_quantized_quant_gb300 import inputs
from oracle import nvfp4 as Q

pytestmark = pytest.mark.gpu


def _padded(rng, counts, tile, cols, extra_rows=0, sizes=None):
    """Groups of `counts` real rows, each padded to a multiple of `tile` rows
    (at least one tile; or of the given sizes), padding and `extra_rows` rows
    past the last group filled with nonzero values.  -> (bits with garbage,
    bits with the padding zeroed, offsets)."""
    if sizes is None:
        sizes = np.maximum((np.maximum(counts, 0) + tile - 1) // tile, 1) * tile
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    x = inputs.student_t4(rng, (int(offs[-1]) + extra_rows, cols))
    x[:, 3] *= 25.0                 # a channel that every group selects
    xz = x.copy()
    for g, c in enumerate(counts):
        xz[offs[g] + min(max(int(c), 0), int(sizes[g])):offs[g + 1]] = 0.0
    return inputs.f32_to_bf16_bits(x), inputs.f32_to_bf16_bits(xz), offs


def _run(lib, bits, offs, counts, k, layout, rlayout, mode, amax=None, scale=None):
    G = len(counts)
    ot, ct = torch.from_numpy(offs).cuda(), torch.from_numpy(counts).cuda()
    kw = {}
    if mode == "amax":
        kw["tensor_amax_in"] = torch.from_numpy(amax).cuda()
    elif mode == "scale":
        kw["tensor_scale_in"] = torch.from_numpy(scale).cuda()
    return lib.quantize_select_groups_nvfp4(bf16_tensor(bits), k, ot, G, group_counts=ct,
                                            scale_layout=layout, r_scale_layout=rlayout,
                                            want_scores=True, **kw)


@pytest.mark.parametrize("layout,rlayout", [(0, 0), (1, 1), (0, 1)])
@pytest.mark.parametrize("mode", ["none", "amax", "scale"])
def test_select_groups_bit_exact_against_the_oracle(lib, layout, rlayout, mode):
    """Seven groups (empty, ragged, full, a count past the group's size) of a
    256-column input, k = 32: codes, scale bytes, tensor scales, scores,
    selections and R_sel against the oracle on the input with each group's
    padding zeroed; the tensor scale from the block's own amax, from a given
    amax, or given."""
    rng = inputs.make_rng(21)
    counts = np.array([5, 0, 128, 33, 64, 100, 300], np.int32)
    sizes = np.array([128, 128, 128, 64, 64, 128, 256])
    bits, bz, offs = _padded(rng, counts, 128, 256, sizes=sizes)
    xz = f32(bz)
    G, k, rows = len(counts), 32, int(offs[-1])
    amax = np.array([np.abs(xz[a:b]).max() if b > a else 0.0
                     for a, b in zip(offs[:-1], offs[1:])], np.float32)
    scale = (amax / np.float32(2688.0) * np.float32(1.25)).astype(np.float32)
    scale[1] = np.float32(1.0)
    q, sel, scores, r = _run(lib, bits, offs, counts, k, layout, rlayout, mode, amax, scale)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    ref = Q.quantize_full(xz, k, offs, tensor_scales=scale if mode == "scale" else None)
    assert np.array_equal(q.tensor_scale.cpu().numpy(), ref["s_t"])
    assert np.array_equal(codes_np(q.codes, 256)[:rows], ref["codes"])
    assert np.array_equal(linear_scales(q, rows, 256), ref["scales"])
    assert np.array_equal(scores.cpu().numpy(), ref["scores"])
    assert np.array_equal(sel.cpu().numpy(), ref["sel"])
    assert np.array_equal(r.tensor_scale.cpu().numpy(), ref["r_s_t"])
    kp = lib.kpad(k)
    rc = codes_np(r.codes, kp)
    assert np.array_equal(rc[:, :k], ref["r_codes"]) and not rc[:, k:].any()
    rs = linear_scales(r, rows, kp)
    assert np.array_equal(rs[:, : k // 16], ref["r_scales"]) and not rs[:, k // 16:].any()


def _two_calls(lib, bz, offs, counts, k, layout, rlayout, rows, **kw):
    """The quantizer (with counts) and the per-group selection on the input
    with the padding zeroed."""
    G = len(counts)
    ot, ct = torch.from_numpy(offs).cuda(), torch.from_numpy(counts).cuda()
    x = bf16_tensor(bz)
    q, part = lib.quantize_nvfp4(x, group_offsets=ot, num_groups=G, group_counts=ct,
                                 scores=True, scale_layout=layout, rows=rows, **kw)
    sel, scores, r = lib.select_residual_channels(x, q, part, k, group_offsets=ot, num_groups=G,
                                                  r_scale_layout=rlayout, want_scores=True)
    return q, sel, scores, r


def _assert_same(lib, a, b, rows_used, cols, k):
    qa, sela, sca, ra = a
    qb, selb, scb, rb = b
    assert torch.equal(qa.codes[:rows_used], qb.codes[:rows_used])
    assert np.array_equal(linear_scales(qa, rows_used, cols), linear_scales(qb, rows_used, cols))
    assert torch.equal(qa.tensor_scale, qb.tensor_scale)
    assert torch.equal(sca, scb) and torch.equal(sela, selb)
    assert torch.equal(ra.codes, rb.codes) and torch.equal(ra.scales, rb.scales)
    assert torch.equal(ra.tensor_scale, rb.tensor_scale)


@pytest.mark.parametrize("shape", ["moe_8192", "decode_512"])
def test_select_groups_matches_the_two_calls_on_expert_shapes(lib, shape):
    """h of the MoE layer: 128 experts, 768 channels, k = 64, tensor-core
    scale layouts, each expert's amax given (as GEMM1's epilogue leaves it),
    the input holding 200 rows past the last group (their R_sel rows are
    zeroed).  8192 tokens: about 512 rows per expert; decode: about 32.  Every
    output equals the quantizer + selection calls' bit for bit."""
    rng = inputs.make_rng(22)
    if shape == "moe_8192":
        counts = rng.integers(440, 600, 128).astype(np.int32)
    else:
        counts = rng.integers(18, 46, 128).astype(np.int32)
    counts[:3] = [0, 1, 128]
    bits, bz, offs = _padded(rng, counts, 128, 768, extra_rows=200)
    rows, used, k = bits.shape[0], int(offs[-1]), 64
    xz = f32(bz)
    amax = np.array([np.abs(xz[a:b]).max() if b > a else 0.0
                     for a, b in zip(offs[:-1], offs[1:])], np.float32)
    at = torch.from_numpy(amax).cuda()
    ot, ct = torch.from_numpy(offs).cuda(), torch.from_numpy(counts).cuda()
    fused = lib.quantize_select_groups_nvfp4(bf16_tensor(bits), k, ot, 128, group_counts=ct,
                                             tensor_amax_in=at, scale_layout=1, r_scale_layout=1,
                                             want_scores=True)
    two = _two_calls(lib, bz, offs, counts, k, 1, 1, rows, tensor_amax_in=at)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    _assert_same(lib, fused, two, used, 768, k)
    kp = lib.kpad(k)
    assert not codes_np(fused[3].codes, kp)[used:].any()
    # the oracle on sampled experts (their rows alone, tensor scale from the amax)
    ts = fused[0].tensor_scale.cpu().numpy()
    codes, scales = codes_np(fused[0].codes, 768), linear_scales(fused[0], used, 768)
    sel, sc = fused[1].cpu().numpy(), fused[2].cpu().numpy()
    rc, rsc = codes_np(fused[3].codes, kp), linear_scales(fused[3], rows, kp)
    rts = fused[3].tensor_scale.cpu().numpy()
    for g in (0, 1, 2, 57, 127):
        a, b = int(offs[g]), int(offs[g + 1])
        assert ts[g] == Q.tensor_scale(xz[a:b])
        ref = Q.quantize_full(xz[a:b], k, tensor_scales=ts[g:g + 1])
        assert np.array_equal(codes[a:b], ref["codes"]) and np.array_equal(scales[a:b], ref["scales"])
        assert np.array_equal(sc[g], ref["scores"][0]) and np.array_equal(sel[g], ref["sel"][0])
        assert rts[g] == ref["r_s_t"][0]
        assert np.array_equal(rc[a:b, :k], ref["r_codes"]) and np.array_equal(rsc[a:b, :k // 16], ref["r_scales"])


@pytest.mark.parametrize("cols,k,tile", [(1024, 128, 32), (64, 64, 32), (512, 16, 64)])
def test_select_groups_many_groups_and_extreme_widths(lib, cols, k, tile):
    """300 groups of one or two tiles (more groups than the grid's first
    wave), counts below 0 and past the group size, the widest input the
    block holds (1024 channels, one per thread), k = cols (every channel
    selected), and the smallest k; linear scale layouts."""
    rng = inputs.make_rng(23)
    G = 300
    sizes = tile * rng.integers(1, 3, G)
    counts = rng.integers(-3, int(sizes.max()) + 8, G).astype(np.int32)
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    x = inputs.student_t4(rng, (int(offs[-1]), cols))
    xz = x.copy()
    for g in range(G):
        xz[offs[g] + min(max(int(counts[g]), 0), int(sizes[g])):offs[g + 1]] = 0.0
    bits, bz = inputs.f32_to_bf16_bits(x), inputs.f32_to_bf16_bits(xz)
    ot, ct = torch.from_numpy(offs).cuda(), torch.from_numpy(counts).cuda()
    fused = lib.quantize_select_groups_nvfp4(bf16_tensor(bits), k, ot, G, group_counts=ct,
                                             want_scores=True)
    # the two calls, with the groups' tensor scales from the fused call's
    # in-block amax passed to the quantizer (it has no per-group amax pass of
    # its own for a given scale) -- and checked against the oracle's
    two = _two_calls(lib, bz, offs, counts, k, 0, 0, int(offs[-1]),
                     tensor_scale_in=fused[0].tensor_scale)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    _assert_same(lib, fused, two, int(offs[-1]), cols, k)
    xf = f32(bz)
    ts = fused[0].tensor_scale.cpu().numpy()
    for g in (0, 1, 150, 299):
        assert ts[g] == Q.tensor_scale(xf[offs[g]:offs[g + 1]])


def test_select_groups_flags_groups_off_the_chunk_grid(lib):
    """A group that does not start at a multiple of 32 rows latches the device
    check (its chunks would not be the score definition's)."""
    bits = inputs.f32_to_bf16_bits(inputs.student_t4(inputs.make_rng(24), (96, 64)))
    offs = torch.tensor([0, 40, 96], dtype=torch.int32, device="cuda")
    lib.quantize_select_groups_nvfp4(bf16_tensor(bits), 16, offs, 2)
    torch.cuda.synchronize()
    assert lib.device_status() == 6      # QUADS_ERR_DEVICE_CHECK (and cleared by the read)
    assert lib.device_status() == 0


@pytest.mark.parametrize("groups", [128, 8])
def test_select_group_counts_take_padding_rows_as_zero(lib, groups):
    """The selection call given the quantizer's group counts reads no padding
    row: on garbage padding it gives what it gives without counts on the
    zeroed padding (128 groups: the per-group R_sel block; 8: the sliced
    residual kernel), and the oracle's R_sel on sampled groups."""
    rng = inputs.make_rng(25)
    counts = rng.integers(0, 200, groups).astype(np.int32)
    counts[:2] = [0, 128]
    bits, bz, offs = _padded(rng, counts, 128, 256)
    G, k = groups, 32
    ot, ct = torch.from_numpy(offs).cuda(), torch.from_numpy(counts).cuda()
    q, part = lib.quantize_nvfp4(bf16_tensor(bits), group_offsets=ot, num_groups=G, group_counts=ct,
                                 scores=True, scale_layout=1)
    a = lib.select_residual_channels(bf16_tensor(bits), q, part, k, group_offsets=ot, num_groups=G,
                                     group_counts=ct, r_scale_layout=1, want_scores=True)
    b = lib.select_residual_channels(bf16_tensor(bz), q, part, k, group_offsets=ot, num_groups=G,
                                     r_scale_layout=1, want_scores=True)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(a[2].codes, b[2].codes) and torch.equal(a[2].scales, b[2].scales)
    assert torch.equal(a[2].tensor_scale, b[2].tensor_scale)
    xz, rows, kp = f32(bz), int(offs[-1]), lib.kpad(k)
    rc, rsc = codes_np(a[2].codes, kp), linear_scales(a[2], rows, kp)
    rts, sel = a[2].tensor_scale.cpu().numpy(), a[0].cpu().numpy()
    for g in (0, 1, groups - 1):
        lo, hi = int(offs[g]), int(offs[g + 1])
        ref = Q.quantize_full(xz[lo:hi], k)
        assert np.array_equal(sel[g], ref["sel"][0]) and rts[g] == ref["r_s_t"][0]
        assert np.array_equal(rc[lo:hi, :k], ref["r_codes"]) and np.array_equal(rsc[lo:hi, :k // 16], ref["r_scales"])


def test_select_groups_on_chip_limits(lib):
    """Groups on both sides of the kernel's two on-chip limits at 768 channels,
    k = 64: the real rows kept in shared memory (about 77 rows) and R kept in
    the squares' buffer ((real rows) * k <= 32 * cols, 384 rows); every output
    equals the two calls'."""
    rng = inputs.make_rng(26)
    counts = np.array(list(range(70, 91)) + list(range(378, 391)), np.int32)
    bits, bz, offs = _padded(rng, counts, 128, 768)
    G, k, rows = len(counts), 64, int(offs[-1])
    ot, ct = torch.from_numpy(offs).cuda(), torch.from_numpy(counts).cuda()
    fused = lib.quantize_select_groups_nvfp4(bf16_tensor(bits), k, ot, G, group_counts=ct,
                                             scale_layout=1, r_scale_layout=1, want_scores=True)
    two = _two_calls(lib, bz, offs, counts, k, 1, 1, rows,
                     tensor_scale_in=fused[0].tensor_scale)
    torch.cuda.synchronize()
    assert lib.device_status() == 0
    _assert_same(lib, fused, two, rows, 768, k)

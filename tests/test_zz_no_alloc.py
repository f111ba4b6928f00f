"""The allocation-free selection entry point gives the same results as the
workspace one.

quads_select_residual_channels_noalloc exists for callers that cannot allocate
device memory (and so cannot pass a workspace): it keeps its scratch in an
array compiled into the library.  This file is collected last so that a run
stopping at the first failure has already run every other test; it must pass
both alone in a fresh process and after the other tests, which is why it
compares against the workspace entry point rather than relying on state left
by earlier tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import bf16_tensor
from nvfp4_w4a4_quantized_quant_gb300 import inputs

pytestmark = pytest.mark.gpu


def _inputs(seed, rows, cols, groups):
    rng = inputs.make_rng(seed)
    x = inputs.student_t4(rng, (rows, cols))
    x[:, rng.choice(cols, 3, replace=False)] *= np.float32(20.0)
    offs = np.linspace(0, rows, groups + 1).astype(np.int32) // 32 * 32
    offs[-1] = rows
    return bf16_tensor(inputs.f32_to_bf16_bits(x)), torch.from_numpy(offs).cuda()


def _both(lib, x, offs, groups, k, layout):
    q, part = lib.quantize_nvfp4(x, group_offsets=offs, num_groups=groups, scores=True,
                                 scale_layout=layout)
    ref = lib.select_residual_channels(x, q, part, k, group_offsets=offs, num_groups=groups,
                                       r_scale_layout=layout, want_scores=True)
    got = lib.select_residual_channels_noalloc(x, q, part, k, group_offsets=offs,
                                               num_groups=groups, r_scale_layout=layout,
                                               want_scores=True)
    torch.cuda.synchronize()
    return ref, got


def test_noalloc_matches_workspace_entry_point_on_two_calls(lib):
    # two calls in a row with different shapes and inputs: the shared scratch
    # array keeps the first call's contents when the second one runs
    for seed, rows, cols, groups, k, layout in [(1, 4096, 2048, 1, 128, 1), (2, 640, 768, 5, 64, 0)]:
        x, offs = _inputs(seed, rows, cols, groups)
        (sel_r, sc_r, r_r), (sel_g, sc_g, r_g) = _both(lib, x, offs, groups, k, layout)
        assert torch.equal(sel_g, sel_r)
        assert torch.equal(sc_g, sc_r)
        assert torch.equal(r_g.codes, r_r.codes)
        assert torch.equal(r_g.scales, r_r.scales)
        assert torch.equal(r_g.tensor_scale, r_r.tensor_scale)
    assert lib.device_status() == 0


def test_noalloc_rejects_shapes_beyond_the_builtin_scratch(lib):
    raw = lib.load()
    limit = 32 << 20
    rows, cols, k = 200000, 2048, 64          # needs rows*k*4 = 51 MB of scratch
    assert lib.workspace_size(lib.OP_SELECT, rows, cols, 0, k, 1) > limit
    p = ctypes.c_void_p(256)                  # rejected on the host before any use
    st = raw.quads_select_residual_channels_noalloc(p, rows, cols, cols, None, 1, None, p, 0, p, p, k,
                                                    p, None, p, p, 0, p, None)
    assert st == 7 and b"built-in array" in raw.quads_last_error_detail()


def test_noalloc_reports_the_same_status_as_the_workspace_entry_point(lib):
    # bad shapes are refused before the scratch is considered, with the codes
    # the workspace entry point returns for the same arguments
    raw = lib.load()
    p = ctypes.c_void_p(256)
    for rows, cols, k in [(64, 256, 0), (64, 256, 24), (64, 250, 16), (64, 256, 512)]:
        st_ws = raw.quads_select_residual_channels(p, rows, cols, cols, None, 1, None, p, 0, p, p, k,
                                                   p, None, p, p, 0, p, p, 1 << 20, None, None)
        st_na = raw.quads_select_residual_channels_noalloc(p, rows, cols, cols, None, 1, None, p, 0, p,
                                                           p, k, p, None, p, p, 0, p, None)
        assert st_ws == st_na != 0, (rows, cols, k, st_ws, st_na)

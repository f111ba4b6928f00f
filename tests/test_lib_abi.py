"""CPU checks of the C ABI: the library builds and loads without a GPU, exports
every function the header declares, and rejects bad arguments on the host
before touching the device."""
import ctypes

import pytest

from nvfp4_w4a4_quantized_quant_gb300 import build, quads


@pytest.fixture(scope="module")
def lib():
    build.build()
    return quads.load()


def test_exports_every_header_symbol(lib):
    syms = quads.header_symbols()
    assert len(syms) >= 14
    assert [s for s in syms if not hasattr(lib, s)] == []
    assert lib.quads_version() == 100


def test_status_strings_and_sizes(lib):
    assert lib.quads_status_string(0) == b"ok"
    assert lib.quads_status_string(5) == b"device pipeline wait timed out"
    assert [lib.quads_kpad(k) for k in (16, 64, 80, 128, 192, 256, 272)] == [64, 64, 128, 128, 256, 256, 512]
    assert lib.quads_workspace_size(quads.OP_QUANTIZE, 10, 64, 0, 0, 3) == 12
    sel = lib.quads_workspace_size(quads.OP_SELECT, 100, 256, 0, 16, 2)
    assert sel == ((100 * 16 * 4 + 255) // 256) * 256 + 256 + 2 * 256 * 4
    assert lib.quads_workspace_size(quads.OP_MOE_ROUTE, 100, 128, 0, 8, 1) == 4 * 128 * 8 + 16
    g = lib.quads_workspace_size(quads.OP_GEMM, 0, 2048, 6144, 128, 1)
    assert g == ((6144 * 64 + 1023) // 1024) * 1024 + 6144 * 8


def _err(lib):
    return lib.quads_last_error_detail().decode()


def test_host_side_argument_checks_need_no_gpu(lib):
    p = ctypes.c_void_p(16)     # never dereferenced: every call below fails validation first
    st = lib.quads_quantize_nvfp4(p, 8, 15, 16, None, None, 1, None, None, None, p, 8, p, 0, p, None, p, 64, None)
    assert st == 2 and "multiple of 16" in _err(lib)
    st = lib.quads_quantize_nvfp4(None, 8, 16, 16, None, None, 1, None, None, None, p, 8, p, 0, p, None, p, 64, None)
    assert st == 1
    st = lib.quads_quantize_nvfp4(p, 8, 32, 16, None, None, 1, None, None, None, p, 16, p, 0, p, None, p, 64, None)
    assert st == 3                                   # ldx < cols
    st = lib.quads_quantize_nvfp4(p, 8, 32, 32, None, None, 1, None, None, None, p, 16, p, 1, p, None, p, 64, None)
    assert st == 2                                   # tcgen05 layout needs cols % 64
    st = lib.quads_quantize_nvfp4(p, 8, 32, 32, None, None, 1, None, p, p, p, 16, p, 0, p, None, p, 64, None)
    assert st == 1                                   # both tensor_scale_in and tensor_amax_in
    st = lib.quads_quantize_nvfp4(p, 8, 32, 32, None, None, 1, p, None, None, p, 16, p, 0, p, None, p, 64, None)
    assert st == 1 and "group_counts" in _err(lib)   # counts without group offsets
    qsg = lambda rows, cols, ldx, k, ts, am, ws: lib.quads_quantize_select_groups_nvfp4(  # noqa: E731
        p, rows, cols, ldx, p, 4, None, ts, am, k, p, cols // 2, p, 0, p, p, None, p, p, 0, p, p,
        ws, None, None)
    assert qsg(64, 2048, 2048, 64, None, None, 1 << 20) == 2   # cols > 1024 (one channel per thread)
    assert qsg(64, 768, 768, 24, None, None, 1 << 20) == 2     # k % 16
    assert qsg(64, 768, 768, 64, p, p, 1 << 20) == 1           # both tensor_scale_in and tensor_amax_in
    assert qsg(64, 768, 512, 64, None, None, 1 << 20) == 3     # ldx < cols
    assert qsg(64, 768, 768, 64, None, None, 16) == 7          # workspace below rows * k * 4
    assert lib.quads_workspace_size(quads.OP_QUANTIZE_SELECT_GROUPS, 100, 768, 0, 64, 4) == 100 * 64 * 4
    st = lib.quads_w4a4_gemm_comp(64, 100, 256, p, p, p, p, p, p, None, None, None, None, None, None,
                                  None, None, 0, p, 0, 100, None, 0, None)
    assert st == 2 and "N%128" in _err(lib)
    st = lib.quads_w4a4_gemm_comp(64, 128, 256, p, p, p, p, p, p, p, p, None, None, p, p, p, p, 8, p, 0,
                                  128, None, 0, None)
    assert st == 1                                   # k not a multiple of 16
    st = lib.quads_w4a4_gemm_comp(64, 128, 256, p, p, p, p, p, p, None, None, None, None, p, p, p, p, 16,
                                  p, 0, 128, None, 0, None)
    assert st == 1 and "column-major" in _err(lib)   # compensation without the weight copy or Q(W_sel)
    st = lib.quads_w4a4_gemm_comp(64, 128, 256, p, p, p, p, p, p, None, None, p, None, p, p, p, p, 16,
                                  p, 0, 128, None, 0, None)
    assert st == 1 and "both" in _err(lib)           # Q(W_sel) codes without its scales
    q = ctypes.c_void_p(24)
    st = lib.quads_w4a4_gemm_comp(64, 128, 256, p, p, p, p, p, p, None, None, q, p, p, p, p, p, 16,
                                  p, 0, 128, None, 0, None)
    assert st == 3                                   # Q(W_sel) not 16-byte aligned
    st = lib.quads_select_residual_channels(p, 64, 256, 256, None, 1, None, p, 0, p, p, 17, p, None, p, p, 0, p,
                                            p, 1 << 20, None, None)
    assert st == 2
    st = lib.quads_select_residual_channels(p, 64, 256, 256, None, 1, p, p, 0, p, p, 16, p, None, p, p, 0, p,
                                            p, 1 << 20, None, None)
    assert st == 1 and "group_counts" in _err(lib)   # counts without group offsets
    u = ctypes.c_void_p(20)                          # 4-byte but not 16-byte aligned
    st = lib.quads_select_residual_channels(p, 64, 256, 256, None, 1, None, p, 0, p, p, 16, p, None, u, p, 0, p,
                                            p, 1 << 20, None, None)
    assert st == 3 and "r_codes" in _err(lib)
    st = lib.quads_select_residual_channels(p, 64, 256, 256, None, 1, None, p, 0, p, p, 16, p, None, p, p, 0, p,
                                            u, 1 << 20, None, None)
    assert st == 3 and "workspace" in _err(lib)
    st = lib.quads_quantize_select_groups_nvfp4(p, 64, 768, 768, p, 4, None, None, None, 64, p, 384, p, 0, p,
                                                p, None, p, p, 0, p, u, 1 << 20, None, None)
    assert st == 3 and "workspace" in _err(lib)
    st = lib.quads_moe_route(p, 100, 16, 8, p, p, p, p, p, p, 1 << 20, u, 1 << 20, None)
    assert st == 3 and "workspace" in _err(lib)
    st = lib.quads_moe_combine(u, 2048, p, p, 16, 8, 2048, p, 2048, None)
    assert st == 3 and "16-byte" in _err(lib)        # y read as 16-byte words
    st = lib.quads_moe_route(p, 100, 300, 8, p, p, p, p, p, p, 1 << 20, p, 1 << 20, None)
    assert st == 2                                   # > 256 experts
    st = lib.quads_moe_route(p, 100, 16, 8, p, p, p, p, p, p, 10, p, 1 << 20, None)
    assert st == 1 and "rows_capacity" in _err(lib)
    st = lib.quads_moe_route(p, 100, 16, 8, p, p, p, p, p, p, 1 << 20, p, 4, None)
    assert st == 7                                   # workspace too small
    st = lib.quads_moe_gather(p, p, 16, 256, 256, p, p, p, ctypes.c_void_p(20), None)
    assert st == 3 and "out_scales" in _err(lib)     # 16-byte scale words need a 16-byte base
    st = lib.quads_moe_gather(p, p, 16, 200, 256, p, p, p, p, None)
    assert st == 2                                   # rows_capacity % 128
    st = lib.quads_moe_grouped_gemm(4, 1000, 256, 256, p, None, p, p, p, 0, p, p, p, None, None, None,
                                    None, None, None, None, 0, None, 0, 0, 0, p, 1, 256, None, None, 0,
                                    None)
    assert st == 2                                   # rows_capacity % 128
    st = lib.quads_weight_columns(p, p, 2, 100, 256, p, p, None)
    assert st == 2                                   # rows_per_group % 128
    st = lib.quads_select_weight_channels(2, 100, 256, p, p, p, 0, 16, p, p, None)
    assert st == 2                                   # rows_per_group % 128
    st = lib.quads_select_weight_channels(2, 128, 256, p, p, p, 0, 24, p, p, None)
    assert st == 1                                   # k % 16
    st = lib.quads_select_weight_channels(2, 128, 256, p, p, p, 0, 272, p, p, None)
    assert st == 1                                   # k > cols
    st = lib.quads_select_weight_channels(2, 128, 256, p, p, None, 0, 16, p, p, None)
    assert st == 1                                   # no selection
    st = lib.quads_trace_round(p, 4, 24, 24, p, 12, p, p, p, None, None)
    assert st == 2
    st = lib.quads_trace_pack_record(p, 4, 24, 12, p, 3, None)
    assert st == 2                                   # cols % 16
    st = lib.quads_trace_pack_record(p, 4, 32, 16, p, 3, None)
    assert st == 2                                   # ld_bits < cols / 8
    st = lib.quads_trace_round_1bit(p, 4, 32, 24, p, 4, p, p, p, 16, None, None)
    assert st == 3                                   # ldx < cols
    st = lib.quads_mx_quantize(p, 4, 48, 48, p, 24, p, 0, None, 0, None)
    assert st == 2                                   # cols % 32
    st = lib.quads_mx_quantize(p, 4, 96, 96, p, 48, p, 1, None, 0, None)
    assert st == 2                                   # TCGEN05 layout needs cols % 128
    st = lib.quads_mx_gemm(64, 128, 192, p, p, p, p, p, 0, 128, None)
    assert st == 2                                   # K % 128
    st = lib.quads_trace_round_mx(p, 4, 48, 48, p, 24, p, p, None, None)
    assert st == 2                                   # cols % 32
    st = lib.quads_qdq_nvfp4(p, 4, 32, 32, None, 1, p, None, 32, None, 16, None, 0, p, None, 0, None)
    assert st == 1                                   # null y
    st = lib.quads_qdq_nvfp4(p, 4, 32, 32, None, 1, p, p, 24, None, 16, None, 0, p, None, 0, None)
    assert st == 3                                   # ldy < cols


def test_product_path_never_imports_the_oracle():
    import pathlib
    pkg = pathlib.Path(quads.__file__).parent
    for f in list(pkg.glob("*.py")) + list(pkg.glob("csrc/*")):
        text = f.read_text()
        assert "import oracle" not in text and "from oracle" not in text, f


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    """No CPU fallback: with the shared library absent the binding raises
    before any computation instead of answering from another code path."""
    import pytest
    from nvfp4_w4a4_quantized_quant_gb300 import quads as Q
    monkeypatch.setattr(Q, "_lib", None)     # restored after the test
    with pytest.raises(RuntimeError, match="not built"):
        Q.load(str(tmp_path / "missing.so"))

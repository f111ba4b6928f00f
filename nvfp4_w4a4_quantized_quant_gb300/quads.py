"""Thin Python binding of the libquads C ABI (ctypes).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels; PyTorch supplies device memory (output and workspace tensors) and the
current CUDA stream.  There is no CPU or PyTorch fallback -- if the library is
not built, or no CUDA device is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass
from typing import Optional

import torch

from .build import DEBUG_LIB, LIB, ROOT

LINEAR, TCGEN05 = 0, 1
OUT_F32, OUT_BF16 = 0, 1
EPI_NONE, EPI_SWIGLU = 0, 1
OP_QUANTIZE, OP_SELECT, OP_GEMM, OP_MOE_GEMM, OP_MOE_ROUTE, OP_QUANTIZE_SELECT = 0, 1, 2, 3, 4, 5
OP_QUANTIZE_SELECT_GROUPS = 6
SCORE_CHUNK_ROWS = 32
MOE_ROW_ALIGN = 128

_P, _I32, _I64, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t

_SIGS = {
    "quads_version": (ctypes.c_int, []),
    "quads_kernel_launch_count": (ctypes.c_uint64, []),
    "quads_status_string": (ctypes.c_char_p, [_I32]),
    "quads_last_error_detail": (ctypes.c_char_p, []),
    "quads_device_status": (_I32, [_P, ctypes.POINTER(_I32)]),
    "quads_test_gemm_wait_timeout": (None, [_I32]),
    "quads_test_gemm_timeline": (None, [_P]),
    "quads_set_gemm_tile_policy": (ctypes.c_int32, [ctypes.c_int32]),
    "quads_workspace_size": (_SZ, [_I32, _I64, _I64, _I64, _I32, _I32]),
    "quads_kpad": (_I32, [_I32]),
    "quads_quantize_nvfp4": (_I32, [_P, _I64, _I64, _I64, _P, _P, _I32, _P, _P, _P, _P, _I64,
                                    _P, _I32, _P, _P, _P, _SZ, _P]),
    "quads_qdq_nvfp4": (_I32, [_P, _I64, _I64, _I64, _P, _I32, _P, _P, _I64, _P, _I64, _P, _I32,
                               _P, _P, _SZ, _P]),
    "quads_select_residual_channels": (_I32, [_P, _I64, _I64, _I64, _P, _I32, _P, _P, _I32, _P,
                                              _P, _I32, _P, _P, _P, _P, _I32, _P, _P, _SZ, _P,
                                              _P]),
    "quads_select_residual_channels_noalloc": (_I32, [_P, _I64, _I64, _I64, _P, _I32, _P, _P, _I32,
                                                      _P, _P, _I32, _P, _P, _P, _P, _I32, _P, _P]),
    "quads_quantize_select_nvfp4": (_I32, [_P, _I64, _I64, _I64, _I32, _P, _I64, _P, _I32, _P, _P,
                                           _P, _P, _P, _I32, _P, _P, _SZ, _P]),
    "quads_quantize_select_groups_nvfp4": (_I32, [_P, _I64, _I64, _I64, _P, _I32, _P, _P, _P, _I32,
                                                  _P, _I64, _P, _I32, _P, _P, _P, _P, _P, _I32, _P,
                                                  _P, _SZ, _P, _P]),
    "quads_w4a4_gemm_comp": (_I32, [_I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                    _P, _P, _P, _P, _I32, _P, _I32, _I64, _P, _SZ, _P]),
    "quads_moe_grouped_gemm": (_I32, [_I32, _I64, _I64, _I64, _P, _P, _P, _P, _P, _I32, _P, _P,
                                      _P, _P, _P, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _I32,
                                      _P, _I32, _I64, _P, _P, _SZ, _P]),
    "quads_weight_columns": (_I32, [_P, _P, _I32, _I64, _I64, _P, _P, _P]),
    "quads_select_weight_channels": (_I32, [_I32, _I64, _I64, _P, _P, _P, _I32, _I32, _P, _P,
                                            _P]),
    "quads_trace_round": (_I32, [_P, _I64, _I64, _I64, _P, _I64, _P, _P, _P, _P, _P]),
    "quads_trace_pack_record": (_I32, [_P, _I64, _I64, _I64, _P, _I64, _P]),
    "quads_trace_round_1bit": (_I32, [_P, _I64, _I64, _I64, _P, _I64, _P, _P, _P, _I64, _P, _P]),
    "quads_mx_quantize": (_I32, [_P, _I64, _I64, _I64, _P, _I64, _P, _I32, _P, _I64, _P]),
    "quads_mx_gemm": (_I32, [_I64, _I64, _I64, _P, _P, _P, _P, _P, _I32, _I64, _P]),
    "quads_trace_round_mx": (_I32, [_P, _I64, _I64, _I64, _P, _I64, _P, _P, _P, _P]),
    "quads_moe_route": (_I32, [_P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _I64, _P, _SZ, _P]),
    "quads_moe_gather": (_I32, [_P, _P, _I32, _I64, _I64, _P, _P, _P, _P, _P]),
    "quads_moe_combine": (_I32, [_P, _I64, _P, _P, _I32, _I32, _I64, _P, _I64, _P]),
}

_lib = None


def header_symbols() -> list[str]:
    """Every function the public header declares."""
    text = open(os.path.join(ROOT, "include", "quads.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(quads_[a-z0-9_]+)\s*\(", text)))


def load(path: Optional[str] = None):
    """Load libquads.so (no CUDA device needed for loading); the bounds-checked
    build when QUADS_DEBUG_LIB=1, or the library at QUADS_LIB when set."""
    global _lib
    if path is None:
        path = os.environ.get("QUADS_LIB") or (
            DEBUG_LIB if os.environ.get("QUADS_DEBUG_LIB") == "1" else LIB)
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libquads is not built ({path}); run "
                               "nvfp4_w4a4_quantized_quant_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


class QuadsError(RuntimeError):
    pass


def _check(status: int, what: str):
    if status != 0:
        lib = load()
        raise QuadsError(f"{what}: {lib.quads_status_string(status).decode()} -- "
                         f"{lib.quads_last_error_detail().decode()}")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise QuadsError("libquads takes device tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _torch_stream(stream=None):
    return torch.cuda.current_stream() if stream is None else stream


def _stream(stream=None):
    return ctypes.c_void_p(_torch_stream(stream).cuda_stream)


def kpad(k: int) -> int:
    return int(load().quads_kpad(k))


def workspace_size(op, rows=0, cols=0, n=0, k=0, groups=1) -> int:
    return int(load().quads_workspace_size(op, rows, cols, n, k, groups))


def _workspace(nbytes: int, device, ws: Optional[torch.Tensor], stream=None):
    """The caller's workspace, or a temporary one allocated on the stream the
    kernels run on (so that the caching allocator does not hand it to another
    stream's allocation while those kernels may still use it)."""
    if ws is not None:
        if ws.numel() < nbytes:
            raise QuadsError(f"workspace of {ws.numel()} bytes < {nbytes}")
        return ws
    with torch.cuda.stream(_torch_stream(stream)):
        return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


def sf_tc_bytes(rows: int, cols: int) -> int:
    return ((rows + 127) // 128) * 128 * (cols // 16)


def kernel_launch_count() -> int:
    """Kernels launched (or captured) by libquads in this process so far."""
    return int(load().quads_kernel_launch_count())


def device_status(stream=None) -> int:
    code = _I32(0)
    _check(load().quads_device_status(_stream(stream), ctypes.byref(code)), "device_status")
    return int(code.value)


def test_gemm_wait_timeout(enable: bool = True) -> None:
    """Test hook: the next GEMM launch runs with a 1 ms wait limit and an MMA
    issuer that issues nothing, so that its bounded waits run out."""
    load().quads_test_gemm_wait_timeout(1 if enable else 0)


def test_gemm_timeline(buf: torch.Tensor) -> None:
    """Profiling hook: the next GEMM launch writes its first CTA's stage
    timeline (int64 [7, 64], %globaltimer ns) into `buf`."""
    assert buf.dtype == torch.int64 and buf.numel() >= 7 * 64 and buf.is_cuda
    load().quads_test_gemm_timeline(_ptr(buf))


TILES_AUTO, TILES_128, TILES_256 = 0, 1, 2


def set_gemm_tile_policy(policy: int) -> int:
    """GEMM output tile width, process-wide (TILES_AUTO: 128x256 for plain
    products with N % 256 == 0; TILES_128; TILES_256: also compensated
    products).  Returns the previous policy."""
    prev = load().quads_set_gemm_tile_policy(int(policy))
    if prev < 0:
        raise ValueError(f"unknown GEMM tile policy {policy}")
    return prev


@dataclass
class QTensor:
    """NVFP4 tensor: packed codes [rows, cols/2], scale bytes in `layout`, tensor scales [G].
    Weights also carry their column-major copy (codes_t, scales_t) for the W_sel gather."""
    codes: torch.Tensor
    scales: torch.Tensor
    tensor_scale: torch.Tensor
    rows: int
    cols: int
    layout: int
    codes_t: Optional[torch.Tensor] = None
    scales_t: Optional[torch.Tensor] = None


def quantize_nvfp4(x: torch.Tensor, *, group_offsets=None, num_groups: int = 1,
                   group_counts=None, tensor_scale_in=None, tensor_amax_in=None,
                   scale_layout: int = LINEAR, scores: bool = False,
                   row_index=None, rows: Optional[int] = None, workspace=None, out=None,
                   stream=None):
    """x bf16 [rows, cols] -> (QTensor, score partials [ceil(rows/32), cols] or None).
    group_counts (int32 [num_groups], with group_offsets): rows of group g at or
    past offsets[g] + counts[g] are taken as zero rows and not read."""
    lib = load()
    assert x.dtype == torch.bfloat16 and x.dim() == 2
    rows = x.shape[0] if rows is None else rows
    cols = x.shape[1]
    G = num_groups if group_offsets is not None else 1
    dev = x.device
    if out is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
        nsf = sf_tc_bytes(rows, cols) if scale_layout == TCGEN05 else rows * (cols // 16)
        scales = torch.empty(nsf, dtype=torch.uint8, device=dev)
        ts = torch.empty(G, dtype=torch.float32, device=dev)
        part = (torch.empty(((rows + 31) // 32, cols), dtype=torch.float32, device=dev)
                if scores else None)
    else:
        codes, scales, ts, part = out
    ws = _workspace(workspace_size(OP_QUANTIZE, rows, cols, 0, 0, G), dev, workspace, stream)
    _check(lib.quads_quantize_nvfp4(_ptr(x), rows, cols, x.stride(0), _ptr(row_index),
                                    _ptr(group_offsets), G, _ptr(group_counts),
                                    _ptr(tensor_scale_in),
                                    _ptr(tensor_amax_in), _ptr(codes),
                                    codes.stride(0), _ptr(scales), scale_layout, _ptr(ts),
                                    _ptr(part), _ptr(ws), ws.numel(), _stream(stream)),
           "quantize_nvfp4")
    return QTensor(codes, scales, ts, rows, cols, scale_layout), part


def qdq_nvfp4(x: torch.Tensor, *, group_offsets=None, num_groups: int = 1,
              tensor_scale_in=None, want_codes: bool = False, scale_layout: int = LINEAR,
              workspace=None, out=None, stream=None):
    """W4A16 fake quantization: -> (y bf16 = DQ(Q(x)), QTensor of the codes or None)."""
    lib = load()
    assert x.dtype == torch.bfloat16 and x.dim() == 2
    rows, cols = x.shape
    G = num_groups if group_offsets is not None else 1
    dev = x.device
    y = out if out is not None else torch.empty((rows, cols), dtype=torch.bfloat16, device=dev)
    codes = scales = None
    if want_codes:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
        nsf = sf_tc_bytes(rows, cols) if scale_layout == TCGEN05 else rows * (cols // 16)
        scales = torch.empty(nsf, dtype=torch.uint8, device=dev)
    ts = torch.empty(G, dtype=torch.float32, device=dev)
    ws = None
    if tensor_scale_in is None:
        ws = _workspace(workspace_size(OP_QUANTIZE, rows, cols, 0, 0, G), dev, workspace, stream)
    _check(lib.quads_qdq_nvfp4(
        _ptr(x), rows, cols, x.stride(0), _ptr(group_offsets), G, _ptr(tensor_scale_in), _ptr(y),
        y.stride(0), _ptr(codes), cols // 2, _ptr(scales), scale_layout, _ptr(ts), _ptr(ws),
        ws.numel() if ws is not None else 0, _stream(stream)), "qdq_nvfp4")
    q = QTensor(codes, scales, ts, rows, cols, scale_layout) if want_codes else None
    return y, q


def _event(ev, stream):
    """Raw cudaEvent_t of a torch.cuda.Event (created by a first record if needed)."""
    if ev is None:
        return None
    if not ev.cuda_event:
        ev.record(_torch_stream(stream))
    return ctypes.c_void_p(ev.cuda_event)


def quantize_select_nvfp4(x: torch.Tensor, k: int, *, scale_layout: int = LINEAR,
                          r_scale_layout: int = LINEAR, want_scores: bool = False,
                          workspace=None, out=None, stream=None):
    """quantize_nvfp4 (tensor scale from the amax, one group) and
    select_residual_channels in one cooperative launch.
    -> (QTensor of Q(X), sel int32 [1, k], scores [1, cols] or None, QTensor of Q(R_sel))."""
    lib = load()
    assert x.dtype == torch.bfloat16 and x.dim() == 2
    rows, cols = x.shape
    kp = kpad(k)
    dev = x.device
    if out is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
        nsf = sf_tc_bytes(rows, cols) if scale_layout == TCGEN05 else rows * (cols // 16)
        scales = torch.empty(nsf, dtype=torch.uint8, device=dev)
        ts = torch.empty(1, dtype=torch.float32, device=dev)
        sel = torch.empty((1, k), dtype=torch.int32, device=dev)
        rc = torch.empty((rows, kp // 2), dtype=torch.uint8, device=dev)
        nrs = sf_tc_bytes(rows, kp) if r_scale_layout == TCGEN05 else rows * (kp // 16)
        rs = torch.empty(nrs, dtype=torch.uint8, device=dev)
        rts = torch.empty(1, dtype=torch.float32, device=dev)
    else:
        codes, scales, ts, sel, rc, rs, rts = out
    sc = torch.empty((1, cols), dtype=torch.float32, device=dev) if want_scores else None
    ws = _workspace(workspace_size(OP_QUANTIZE_SELECT, rows, cols, 0, k, 1), dev, workspace, stream)
    _check(lib.quads_quantize_select_nvfp4(
        _ptr(x), rows, cols, x.stride(0), k, _ptr(codes), codes.stride(0), _ptr(scales),
        scale_layout, _ptr(ts), _ptr(sel), _ptr(sc), _ptr(rc), _ptr(rs), r_scale_layout, _ptr(rts),
        _ptr(ws), ws.numel(), _stream(stream)), "quantize_select_nvfp4")
    return (QTensor(codes, scales, ts, rows, cols, scale_layout), sel, sc,
            QTensor(rc, rs, rts, rows, kp, r_scale_layout))


def quantize_select_groups_nvfp4(x: torch.Tensor, k: int, group_offsets, num_groups: int, *,
                                 group_counts=None, tensor_scale_in=None, tensor_amax_in=None,
                                 scale_layout: int = LINEAR, r_scale_layout: int = LINEAR,
                                 want_scores: bool = False, rows: Optional[int] = None,
                                 sel_ready_event=None, workspace=None, out=None, stream=None):
    """quantize_nvfp4 (row groups, score partials) and select_residual_channels
    (per group) in one launch, one block per group.
    -> (QTensor of Q(X), sel int32 [G, k], scores [G, cols] or None, QTensor of Q(R_sel)).
    out = (codes, scales, tensor_scale [G], sel, r_codes, r_scales, r_tensor_scale [G])."""
    lib = load()
    assert x.dtype == torch.bfloat16 and x.dim() == 2
    rows = x.shape[0] if rows is None else rows
    cols = x.shape[1]
    G = num_groups
    kp = kpad(k)
    dev = x.device
    if out is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
        nsf = sf_tc_bytes(rows, cols) if scale_layout == TCGEN05 else rows * (cols // 16)
        scales = torch.empty(nsf, dtype=torch.uint8, device=dev)
        ts = torch.empty(G, dtype=torch.float32, device=dev)
        sel = torch.empty((G, k), dtype=torch.int32, device=dev)
        rc = torch.empty((rows, kp // 2), dtype=torch.uint8, device=dev)
        nrs = sf_tc_bytes(rows, kp) if r_scale_layout == TCGEN05 else rows * (kp // 16)
        rs = torch.empty(nrs, dtype=torch.uint8, device=dev)
        rts = torch.empty(G, dtype=torch.float32, device=dev)
    else:
        codes, scales, ts, sel, rc, rs, rts = out
    sc = torch.empty((G, cols), dtype=torch.float32, device=dev) if want_scores else None
    ws = _workspace(workspace_size(OP_QUANTIZE_SELECT_GROUPS, rows, cols, 0, k, G), dev, workspace,
                    stream)
    _check(lib.quads_quantize_select_groups_nvfp4(
        _ptr(x), rows, cols, x.stride(0), _ptr(group_offsets), G, _ptr(group_counts),
        _ptr(tensor_scale_in), _ptr(tensor_amax_in), k, _ptr(codes), codes.stride(0),
        _ptr(scales), scale_layout, _ptr(ts), _ptr(sel), _ptr(sc), _ptr(rc), _ptr(rs),
        r_scale_layout, _ptr(rts), _ptr(ws), ws.numel(), _event(sel_ready_event, stream),
        _stream(stream)), "quantize_select_groups_nvfp4")
    return (QTensor(codes, scales, ts, rows, cols, scale_layout), sel, sc,
            QTensor(rc, rs, rts, rows, kp, r_scale_layout))


def select_residual_channels(x: torch.Tensor, q: QTensor, partials: torch.Tensor, k: int, *,
                             group_offsets=None, num_groups: int = 1, group_counts=None,
                             r_scale_layout: int = LINEAR, want_scores: bool = False,
                             sel_ready_event=None, workspace=None, out=None, stream=None):
    """-> (sel int32 [G, k], scores [G, cols] or None, QTensor of Q(R_sel) [rows, kpad]).
    sel_ready_event (torch.cuda.Event): recorded once sel is written, before R_sel.
    group_counts: as given to quantize_nvfp4 (rows past a group's count are zero rows)."""
    lib = load()
    G = num_groups if group_offsets is not None else 1
    rows, cols = q.rows, q.cols
    kp = kpad(k)
    dev = x.device
    if out is None:
        sel = torch.empty((G, k), dtype=torch.int32, device=dev)
        rc = torch.empty((rows, kp // 2), dtype=torch.uint8, device=dev)
        nsf = sf_tc_bytes(rows, kp) if r_scale_layout == TCGEN05 else rows * (kp // 16)
        rs = torch.empty(nsf, dtype=torch.uint8, device=dev)
        rts = torch.empty(G, dtype=torch.float32, device=dev)
    else:
        sel, rc, rs, rts = out
    sc = torch.empty((G, cols), dtype=torch.float32, device=dev) if want_scores else None
    ws = _workspace(workspace_size(OP_SELECT, rows, cols, 0, k, G), dev, workspace, stream)
    _check(lib.quads_select_residual_channels(
        _ptr(x), rows, cols, x.stride(0), _ptr(group_offsets), G, _ptr(group_counts),
        _ptr(q.scales), q.layout,
        _ptr(q.tensor_scale), _ptr(partials), k, _ptr(sel), _ptr(sc), _ptr(rc), _ptr(rs),
        r_scale_layout, _ptr(rts), _ptr(ws), ws.numel(), _event(sel_ready_event, stream),
        _stream(stream)), "select_residual_channels")
    return sel, sc, QTensor(rc, rs, rts, rows, kp, r_scale_layout)


def select_residual_channels_noalloc(x: torch.Tensor, q: QTensor, partials: torch.Tensor, k: int, *,
                                     group_offsets=None, num_groups: int = 1, group_counts=None,
                                     r_scale_layout: int = LINEAR, want_scores: bool = False,
                                     out=None, stream=None):
    """As select_residual_channels, with the library's built-in scratch array instead of
    a workspace (for callers that cannot allocate)."""
    lib = load()
    G = num_groups if group_offsets is not None else 1
    rows, cols = q.rows, q.cols
    kp = kpad(k)
    dev = x.device
    if out is None:
        sel = torch.empty((G, k), dtype=torch.int32, device=dev)
        rc = torch.empty((rows, kp // 2), dtype=torch.uint8, device=dev)
        nsf = sf_tc_bytes(rows, kp) if r_scale_layout == TCGEN05 else rows * (kp // 16)
        rs = torch.empty(nsf, dtype=torch.uint8, device=dev)
        rts = torch.empty(G, dtype=torch.float32, device=dev)
    else:
        sel, rc, rs, rts = out
    sc = torch.empty((G, cols), dtype=torch.float32, device=dev) if want_scores else None
    _check(lib.quads_select_residual_channels_noalloc(
        _ptr(x), rows, cols, x.stride(0), _ptr(group_offsets), G, _ptr(group_counts),
        _ptr(q.scales), q.layout,
        _ptr(q.tensor_scale), _ptr(partials), k, _ptr(sel), _ptr(sc), _ptr(rc), _ptr(rs),
        r_scale_layout, _ptr(rts), _stream(stream)), "select_residual_channels_noalloc")
    return sel, sc, QTensor(rc, rs, rts, rows, kp, r_scale_layout)


def _wsel_args(r, w, w_sel, size_args, dev, workspace, stream=None):
    """Workspace and Q(W_sel) pointers of a compensated GEMM call."""
    if r is None:
        return None, None, None
    if w_sel is not None:
        return None, _ptr(w_sel.codes), _ptr(w_sel.scales)
    if w.codes_t is None:
        raise QuadsError("compensation needs the weight's column-major copy (weight_columns)")
    return _workspace(workspace_size(*size_args), dev, workspace, stream), None, None


def w4a4_gemm_comp(a: QTensor, w: QTensor, r: Optional[QTensor] = None, sel=None, k: int = 0, *,
                   out_dtype=torch.bfloat16, w_sel: Optional[QTensor] = None, workspace=None,
                   out=None, stream=None):
    """Y [M, N] = Q(A) Q(W)^T (+ Q(R_sel) Q(W_sel)^T when r is given; Q(W_sel) is
    built by the call unless given, from select_weight_channels)."""
    lib = load()
    M, K, N = a.rows, a.cols, w.rows
    y = out if out is not None else torch.empty((M, N), dtype=out_dtype, device=a.codes.device)
    yd = OUT_F32 if y.dtype == torch.float32 else OUT_BF16
    ws, wsc, wss = _wsel_args(r, w, w_sel, (OP_GEMM, 0, K, N, k, 1), y.device, workspace, stream)
    _check(lib.quads_w4a4_gemm_comp(
        M, N, K, _ptr(a.codes), _ptr(a.scales), _ptr(a.tensor_scale), _ptr(w.codes),
        _ptr(w.scales), _ptr(w.tensor_scale), _ptr(w.codes_t), _ptr(w.scales_t), wsc, wss,
        _ptr(r.codes if r else None),
        _ptr(r.scales if r else None), _ptr(r.tensor_scale if r else None), _ptr(sel), k,
        _ptr(y), yd, y.stride(0), _ptr(ws), ws.numel() if ws is not None else 0,
        _stream(stream)), "w4a4_gemm_comp")
    return y


def moe_grouped_gemm(plan: dict, a: QTensor, w: QTensor, num_experts: int, n: int,
                     r: Optional[QTensor] = None, sel=None, k: int = 0, *,
                     a_scale_per_expert: bool = False, r_scale_per_expert: bool = False,
                     sel_per_expert: bool = False, epilogue: int = EPI_NONE,
                     out_dtype=torch.bfloat16, y_amax=None, w_sel: Optional[QTensor] = None,
                     workspace=None, out=None, stream=None):
    """Grouped compensated GEMM over the experts of `plan` (from moe_route)."""
    lib = load()
    cap = plan["rows_capacity"]
    K = a.cols
    ycols = n // 2 if epilogue == EPI_SWIGLU else n
    y = out if out is not None else torch.empty((cap, ycols), dtype=out_dtype, device=a.codes.device)
    yd = OUT_F32 if y.dtype == torch.float32 else OUT_BF16
    ws, wsc, wss = _wsel_args(r, w, w_sel, (OP_MOE_GEMM, 0, K, n, k, num_experts), y.device,
                              workspace, stream)
    _check(lib.quads_moe_grouped_gemm(
        num_experts, cap, n, K, _ptr(plan["offsets"]), _ptr(plan["counts"]), _ptr(a.codes),
        _ptr(a.scales), _ptr(a.tensor_scale), int(a_scale_per_expert), _ptr(w.codes),
        _ptr(w.scales), _ptr(w.tensor_scale), _ptr(w.codes_t), _ptr(w.scales_t), wsc, wss,
        _ptr(r.codes if r else None), _ptr(r.scales if r else None),
        _ptr(r.tensor_scale if r else None), int(r_scale_per_expert), _ptr(sel),
        int(sel_per_expert), k, epilogue, _ptr(y), yd, y.stride(0), _ptr(y_amax), _ptr(ws),
        ws.numel() if ws is not None else 0, _stream(stream)),
        "moe_grouped_gemm")
    return y


def trace_round(x_train: torch.Tensor, rollout: QTensor, *, counters=None, out=None, stream=None):
    """-> (codes [rows, cols/2], counters int64 [3]: rtn mismatches, trace mismatches, rtn off-by-one)."""
    lib = load()
    rows, cols = x_train.shape
    if rollout.layout != LINEAR:
        raise QuadsError("trace_round takes LINEAR rollout scales")
    codes = out if out is not None else torch.empty((rows, cols // 2), dtype=torch.uint8,
                                                    device=x_train.device)
    if counters is None:
        counters = torch.zeros(3, dtype=torch.int64, device=x_train.device)
    _check(lib.quads_trace_round(_ptr(x_train), rows, cols, x_train.stride(0),
                                 _ptr(rollout.codes), rollout.codes.stride(0),
                                 _ptr(rollout.scales), _ptr(rollout.tensor_scale), _ptr(codes),
                                 _ptr(counters), _stream(stream)), "trace_round")
    return codes, counters


def trace_pack_record(rollout: QTensor, *, out=None, stream=None) -> torch.Tensor:
    """Mantissa bits of the rollout codes, [rows, cols/8] bytes (element 8i+j in bit j)."""
    lib = load()
    rows, cols = rollout.rows, rollout.cols
    bits = out if out is not None else torch.empty((rows, cols // 8), dtype=torch.uint8,
                                                   device=rollout.codes.device)
    _check(lib.quads_trace_pack_record(_ptr(rollout.codes), rows, cols, rollout.codes.stride(0),
                                       _ptr(bits), bits.stride(0), _stream(stream)),
           "trace_pack_record")
    return bits


def trace_round_1bit(x_train: torch.Tensor, mantissa_bits: torch.Tensor, rollout: QTensor, *,
                     counters=None, out=None, stream=None):
    """-> (codes [rows, cols/2], counters int64 [2]: changed vs RTN, record-bit mismatches).
    Uses the rollout's LINEAR scales and tensor scale; its codes are not read."""
    lib = load()
    rows, cols = x_train.shape
    if rollout.layout != LINEAR:
        raise QuadsError("trace_round_1bit takes LINEAR rollout scales")
    codes = out if out is not None else torch.empty((rows, cols // 2), dtype=torch.uint8,
                                                    device=x_train.device)
    if counters is None:
        counters = torch.zeros(2, dtype=torch.int64, device=x_train.device)
    _check(lib.quads_trace_round_1bit(_ptr(x_train), rows, cols, x_train.stride(0),
                                      _ptr(mantissa_bits), mantissa_bits.stride(0),
                                      _ptr(rollout.scales), _ptr(rollout.tensor_scale),
                                      _ptr(codes), codes.stride(0), _ptr(counters),
                                      _stream(stream)), "trace_round_1bit")
    return codes, counters


def mx_quantize(x: torch.Tensor, *, scale_layout: int = LINEAR, want_qdq: bool = False,
                out=None, stream=None):
    """MXFP4 (32-element blocks, E8M0 scales) -> (QTensor with tensor_scale None, bf16 QDQ or None)."""
    lib = load()
    assert x.dtype == torch.bfloat16 and x.dim() == 2
    rows, cols = x.shape
    dev = x.device
    if out is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
        nsf = ((rows + 127) // 128 * 128 if scale_layout == TCGEN05 else rows) * (cols // 32)
        scales = torch.empty(nsf, dtype=torch.uint8, device=dev)
    else:
        codes, scales = out
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device=dev) if want_qdq else None
    _check(lib.quads_mx_quantize(_ptr(x), rows, cols, x.stride(0), _ptr(codes), codes.stride(0),
                                 _ptr(scales), scale_layout, _ptr(y), cols, _stream(stream)),
           "mx_quantize")
    return QTensor(codes, scales, None, rows, cols, scale_layout), y


def mx_gemm(a: QTensor, w: QTensor, *, out_dtype=torch.bfloat16, out=None, stream=None):
    """Y [M, N] = DQ(A) DQ(W)^T for MXFP4 operands (TCGEN05 scale layout)."""
    lib = load()
    if a.layout != TCGEN05 or w.layout != TCGEN05:
        raise QuadsError("mx_gemm takes TCGEN05 scale layouts")
    M, K, N = a.rows, a.cols, w.rows
    y = out if out is not None else torch.empty((M, N), dtype=out_dtype, device=a.codes.device)
    yd = OUT_F32 if y.dtype == torch.float32 else OUT_BF16
    _check(lib.quads_mx_gemm(M, N, K, _ptr(a.codes), _ptr(a.scales), _ptr(w.codes),
                             _ptr(w.scales), _ptr(y), yd, y.stride(0), _stream(stream)), "mx_gemm")
    return y


def trace_round_mx(x_train: torch.Tensor, rollout: QTensor, *, counters=None, out=None,
                   stream=None):
    """TRACE rounding under an MXFP4 rollout (LINEAR E8M0 scales)."""
    lib = load()
    rows, cols = x_train.shape
    if rollout.layout != LINEAR:
        raise QuadsError("trace_round_mx takes LINEAR rollout scales")
    codes = out if out is not None else torch.empty((rows, cols // 2), dtype=torch.uint8,
                                                    device=x_train.device)
    if counters is None:
        counters = torch.zeros(3, dtype=torch.int64, device=x_train.device)
    _check(lib.quads_trace_round_mx(_ptr(x_train), rows, cols, x_train.stride(0),
                                    _ptr(rollout.codes), rollout.codes.stride(0),
                                    _ptr(rollout.scales), _ptr(codes), _ptr(counters),
                                    _stream(stream)), "trace_round_mx")
    return codes, counters


def moe_rows_capacity(tokens: int, topk: int, experts: int) -> int:
    cap = tokens * topk + experts * (MOE_ROW_ALIGN - 1)
    return (cap + MOE_ROW_ALIGN - 1) // MOE_ROW_ALIGN * MOE_ROW_ALIGN


def weight_columns(w: QTensor, num_groups: int = 1, stream=None) -> QTensor:
    """Attach the column-major copy of an NVFP4 weight (made once per weight update)."""
    lib = load()
    rpg = w.rows // num_groups
    dev = w.codes.device
    w.codes_t = torch.empty(num_groups * w.cols * (rpg // 2), dtype=torch.uint8, device=dev)
    w.scales_t = torch.empty(num_groups * (w.cols // 16) * rpg, dtype=torch.uint8, device=dev)
    _check(lib.quads_weight_columns(_ptr(w.codes), _ptr(w.scales), num_groups, rpg, w.cols,
                                    _ptr(w.codes_t), _ptr(w.scales_t), _stream(stream)),
           "weight_columns")
    return w


def select_weight_channels(w: QTensor, sel: torch.Tensor, k: int, num_groups: int = 1, *,
                           sel_per_group: bool = False, out=None, stream=None) -> QTensor:
    """Q(W_sel): the selected columns of the weight (per group), requantized with
    the group's s_w kept aside; TCGEN05 scales over kpad columns."""
    lib = load()
    if w.codes_t is None:
        raise QuadsError("select_weight_channels needs the column-major copy (weight_columns)")
    rpg, kp, dev = w.rows // num_groups, kpad(k), w.codes.device
    if out is None:
        out = (torch.empty((w.rows, kp // 2), dtype=torch.uint8, device=dev),
               torch.empty(sf_tc_bytes(w.rows, kp), dtype=torch.uint8, device=dev))
    codes, scales = out
    _check(lib.quads_select_weight_channels(num_groups, rpg, w.cols, _ptr(w.codes_t),
                                            _ptr(w.scales_t), _ptr(sel), int(sel_per_group), k,
                                            _ptr(codes), _ptr(scales), _stream(stream)),
           "select_weight_channels")
    return QTensor(codes, scales, None, w.rows, kp, TCGEN05)


def moe_route(logits: torch.Tensor, topk: int, *, rows_capacity: Optional[int] = None,
              out=None, workspace=None, stream=None) -> dict:
    lib = load()
    T, E = logits.shape
    cap = rows_capacity or moe_rows_capacity(T, topk, E)
    dev = logits.device
    if out is None:
        out = dict(idx=torch.empty((T, topk), dtype=torch.int32, device=dev),
                   gates=torch.empty((T, topk), dtype=torch.float32, device=dev),
                   counts=torch.empty(E, dtype=torch.int32, device=dev),
                   offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   row_token=torch.empty(cap, dtype=torch.int32, device=dev),
                   token_row=torch.empty((T, topk), dtype=torch.int32, device=dev))
    ws = _workspace(workspace_size(OP_MOE_ROUTE, T, E, 0, topk, 1), dev, workspace, stream)
    _check(lib.quads_moe_route(_ptr(logits), T, E, topk, _ptr(out["idx"]), _ptr(out["gates"]),
                               _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["row_token"]),
                               _ptr(out["token_row"]), cap, _ptr(ws), ws.numel(),
                               _stream(stream)), "moe_route")
    out.update(rows_capacity=cap, tokens=T, experts=E, topk=topk)
    return out


def moe_gather(plan: dict, q: QTensor, *, out=None, stream=None) -> QTensor:
    lib = load()
    cap, cols = plan["rows_capacity"], q.cols
    dev = q.codes.device
    if out is None:
        oc = torch.empty((cap, cols // 2), dtype=torch.uint8, device=dev)
        osf = torch.empty(sf_tc_bytes(cap, cols), dtype=torch.uint8, device=dev)
    else:
        oc, osf = out
    _check(lib.quads_moe_gather(_ptr(plan["row_token"]), _ptr(plan["offsets"]), plan["experts"],
                                cap, cols, _ptr(q.codes), _ptr(q.scales), _ptr(oc), _ptr(osf),
                                _stream(stream)), "moe_gather")
    return QTensor(oc, osf, q.tensor_scale, cap, cols, TCGEN05)


def moe_combine(y: torch.Tensor, plan: dict, *, out=None, stream=None) -> torch.Tensor:
    lib = load()
    T, topk, H = plan["tokens"], plan["topk"], y.shape[1]
    o = out if out is not None else torch.empty((T, H), dtype=torch.bfloat16, device=y.device)
    _check(lib.quads_moe_combine(_ptr(y), y.stride(0), _ptr(plan["token_row"]),
                                 _ptr(plan["gates"]), T, topk, H, _ptr(o), o.stride(0),
                                 _stream(stream)), "moe_combine")
    return o


def swiglu_row_index(experts: int, ffn: int, hidden: int, device) -> torch.Tensor:
    """Row order of the stacked W1 [E*2F, H] that puts 64 gate rows and the
    matching 64 up rows in every 128-row tile (what the SwiGLU epilogue reads)."""
    assert ffn % 64 == 0
    l = torch.arange(2 * ffn, dtype=torch.int64)
    tile, within = l // 128, l % 128
    src = torch.where(within < 64, tile * 64 + within, ffn + tile * 64 + (within - 64))
    full = (torch.arange(experts, dtype=torch.int64)[:, None] * (2 * ffn) + src[None, :]).reshape(-1)
    return full.to(torch.int32).to(device)


def quantize_expert_weights(w: torch.Tensor, *, swiglu_interleave: bool = False,
                            stream=None) -> QTensor:
    """Stacked expert weights bf16 [E, N, K] -> NVFP4 with one tensor scale per
    expert and tensor-core scale layout (N % 128 == 0)."""
    E, N, K = w.shape
    flat = w.reshape(E * N, K)
    offs = torch.arange(0, E * N + 1, N, dtype=torch.int32, device=w.device)
    ri = swiglu_row_index(E, N // 2, K, w.device) if swiglu_interleave else None
    q, _ = quantize_nvfp4(flat, group_offsets=offs, num_groups=E, scale_layout=TCGEN05,
                          row_index=ri, stream=stream)
    return weight_columns(q, E, stream=stream)

"""The two rollout-side layers built from libquads calls, with every buffer
allocated once so a forward pass only enqueues kernels (and can be captured
in a CUDA graph).

CompensatedLinear   Y = Q(X) Q(W)^T + Q(R_sel) Q(W_sel)^T
MoEExpertLayer      route -> quantize X (+select) -> gather -> grouped GEMM1
                    (+SwiGLU) -> quantize h per expert (+select) -> grouped
                    GEMM2 -> combine

[QUADS technical summary] 2.2 B "Residual Activation Compensation (Rollout
Side)"; [TRACE digest] "MoE 专家路由敏感性".
"""
from __future__ import annotations

from typing import Optional

import torch

from . import quads as Q


class CompensatedLinear:
    """One compensated W4A4 projection with pre-quantized weights (weights are
    quantized once, as after a weight sync; activations every call)."""

    def __init__(self, w: torch.Tensor, k: int, max_rows: int, out_dtype=torch.bfloat16,
                 compensate: bool = True):
        self.N, self.K = w.shape
        self.k, self.compensate = k, compensate
        dev = w.device
        self.wq, _ = Q.quantize_nvfp4(w, scale_layout=Q.TCGEN05)
        Q.weight_columns(self.wq)
        self.max_rows = max_rows
        kp = Q.kpad(k)
        self.bufs = dict(
            codes=torch.empty((max_rows, self.K // 2), dtype=torch.uint8, device=dev),
            scales=torch.empty(Q.sf_tc_bytes(max_rows, self.K), dtype=torch.uint8, device=dev),
            ts=torch.empty(1, dtype=torch.float32, device=dev),
            part=torch.empty(((max_rows + 31) // 32, self.K), dtype=torch.float32, device=dev),
            sel=torch.empty((1, k), dtype=torch.int32, device=dev),
            rc=torch.empty((max_rows, kp // 2), dtype=torch.uint8, device=dev),
            rs=torch.empty(Q.sf_tc_bytes(max_rows, kp), dtype=torch.uint8, device=dev),
            rts=torch.empty(1, dtype=torch.float32, device=dev),
            y=torch.empty((max_rows, self.N), dtype=out_dtype, device=dev),
            wsc=torch.empty((self.N, kp // 2), dtype=torch.uint8, device=dev),
            wss=torch.empty(Q.sf_tc_bytes(self.N, kp), dtype=torch.uint8, device=dev),
        )
        self.ws_q = torch.empty(Q.workspace_size(Q.OP_QUANTIZE, max_rows, self.K), dtype=torch.uint8,
                                device=dev)
        self.ws_s = torch.empty(Q.workspace_size(Q.OP_SELECT, max_rows, self.K, 0, k),
                                dtype=torch.uint8, device=dev)
        # Q(W_sel) is built on a side stream as soon as the selection is known,
        # next to the residual slice (forked and joined by events)
        self.side = torch.cuda.Stream(device=dev)
        self.ev_sel, self.ev_w = torch.cuda.Event(), torch.cuda.Event()
        # the weight preparation above ran on the current stream; forward() may
        # run on other streams that do not wait for it (and the allocator may
        # already hand its freed scratch to other buffers), so finish it here
        torch.cuda.current_stream(dev).synchronize()

    def forward(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        b = self.bufs
        M = x.shape[0]
        assert M <= self.max_rows
        xq, part = Q.quantize_nvfp4(x, scale_layout=Q.TCGEN05, scores=self.compensate,
                                    workspace=self.ws_q, stream=stream,
                                    out=(b["codes"][:M], b["scales"], b["ts"],
                                         b["part"][: (M + 31) // 32] if self.compensate else None))
        y = b["y"][:M]
        if not self.compensate:
            return Q.w4a4_gemm_comp(xq, self.wq, out=y, stream=stream)
        main = torch.cuda.current_stream() if stream is None else stream
        sel, _, r = Q.select_residual_channels(x, xq, part, self.k, r_scale_layout=Q.TCGEN05,
                                               workspace=self.ws_s, sel_ready_event=self.ev_sel,
                                               stream=stream,
                                               out=(b["sel"], b["rc"][:M], b["rs"], b["rts"]))
        self.side.wait_event(self.ev_sel)
        wsel = Q.select_weight_channels(self.wq, sel, self.k, stream=self.side,
                                        out=(b["wsc"], b["wss"]))
        self.ev_w.record(self.side)
        main.wait_event(self.ev_w)
        return Q.w4a4_gemm_comp(xq, self.wq, r, sel, self.k, out=y, w_sel=wsel, stream=stream)


class MoEExpertLayer:
    """Routed expert FFN (gate+up, SwiGLU, down) with NVFP4 W4A4 GEMMs and
    residual compensation on both GEMMs."""

    def __init__(self, w1: torch.Tensor, w2: torch.Tensor, topk: int, k1: int, k2: int,
                 max_tokens: int, compensate: bool = True, fused_activation_side: bool = False,
                 fused_expert_side: Optional[bool] = None):
        """fused_activation_side: GEMM1's activation side (quantization,
        selection, R_sel) as one cooperative launch (quantize_select_nvfp4)
        instead of the quantizer and the selection call.  Off by default: the
        cooperative grid holds every SM while it runs, so the routing on the
        side stream cannot overlap it.
        fused_expert_side: GEMM2's activation side (h's per-expert
        quantization, selection and R_sel) as one launch with a block per
        expert (quantize_select_groups_nvfp4) instead of the quantizer and the
        selection call; the same outputs bit for bit.  None (default): used
        when the experts average at most 256 rows (decode-sized and mid-sized
        batches, where it saves launches); with more rows per expert, one
        block per expert quantizes slower than the quantizer spread over
        every SM, and Q(W_sel) could no longer overlap R_sel."""
        self.E, twoF, self.H = w1.shape
        self.F = twoF // 2
        assert w2.shape == (self.E, self.H, self.F)
        self.topk, self.k1, self.k2, self.compensate = topk, k1, k2, compensate
        self.fused = fused_activation_side
        if fused_expert_side is None:
            fused_expert_side = max_tokens * topk <= 256 * w1.shape[0]
        self.fused_h = fused_expert_side
        dev = w1.device
        self.w1q = Q.quantize_expert_weights(w1, swiglu_interleave=True)
        self.w2q = Q.quantize_expert_weights(w2)
        T, E, H, F = max_tokens, self.E, self.H, self.F
        cap = Q.moe_rows_capacity(T, topk, E)
        self.cap, self.max_tokens = cap, T
        kp1, kp2 = Q.kpad(k1), Q.kpad(k2)
        u8, f32, i32 = torch.uint8, torch.float32, torch.int32
        e = lambda *s, dt=u8: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
        # h and y: rows past the last expert's group (and y's padding rows) are
        # never written by the kernels; zeroed once here so that whole-buffer
        # reads see zeros rather than stale memory
        z = lambda *s, dt: torch.zeros(*s, dtype=dt, device=dev)  # noqa: E731
        self.b = dict(
            route=dict(idx=e((T, topk), dt=i32), gates=e((T, topk), dt=f32), counts=e(E, dt=i32),
                       offsets=e(E + 1, dt=i32), row_token=e(cap, dt=i32),
                       token_row=e((T, topk), dt=i32)),
            xc=e((T, H // 2)), xs=e(T * (H // 16)), xts=e(1, dt=f32), xpart=e(((T + 31) // 32, H), dt=f32),
            sel1=e((1, k1), dt=i32), r1c=e((T, kp1 // 2)), r1s=e(T * (kp1 // 16)), r1ts=e(1, dt=f32),
            a1c=e((cap, H // 2)), a1s=e(Q.sf_tc_bytes(cap, H)),
            g1c=e((cap, kp1 // 2)), g1s=e(Q.sf_tc_bytes(cap, kp1)),
            h=z((cap, F), dt=torch.bfloat16),
            hc=e((cap, F // 2)), hs=e(Q.sf_tc_bytes(cap, F)), hts=e(E, dt=f32),
            hpart=e((cap // 32, F), dt=f32),
            sel2=e((E, k2), dt=i32), r2c=e((cap, kp2 // 2)), r2s=e(Q.sf_tc_bytes(cap, kp2)),
            r2ts=e(E, dt=f32), hamax=e(E, dt=f32),
            y=z((cap, H), dt=torch.bfloat16), out=e((T, H), dt=torch.bfloat16),
            w1sc=e((E * 2 * F, kp1 // 2)), w1ss=e(Q.sf_tc_bytes(E * 2 * F, kp1)),
            w2sc=e((E * H, kp2 // 2)), w2ss=e(Q.sf_tc_bytes(E * H, kp2)),
        )
        self.ws = dict(
            rt=e(Q.workspace_size(Q.OP_MOE_ROUTE, T, E, 0, topk)),
            q1=e(Q.workspace_size(Q.OP_QUANTIZE, T, H)),
            s1=e(Q.workspace_size(Q.OP_SELECT, T, H, 0, k1)),
            qs1=e(Q.workspace_size(Q.OP_QUANTIZE_SELECT, T, H, 0, k1) if fused_activation_side else 16),
            q2=e(Q.workspace_size(Q.OP_QUANTIZE, cap, F, 0, 0, E)),
            s2=e(Q.workspace_size(Q.OP_SELECT, cap, F, 0, k2, E)),
            qs2=e(Q.workspace_size(Q.OP_QUANTIZE_SELECT_GROUPS, cap, F, 0, k2, E)),
        )
        # Work that does not wait on its neighbours runs on two side streams,
        # forked and joined by events (so this also holds inside a captured
        # graph): routing, then the gather of X's rows (needs only X's codes),
        # on `side`; Q(W_sel) of each GEMM (needs only the selection, not
        # R_sel) on `wside`.
        self.side = torch.cuda.Stream(device=dev)
        self.wside = torch.cuda.Stream(device=dev)
        (self.ev_fork, self.ev_xq, self.ev_a1, self.ev_sel1, self.ev_w1, self.ev_sel2,
         self.ev_w2, self.ev_plan) = (torch.cuda.Event() for _ in range(8))
        # the weight preparation and buffer fills above ran on the current
        # stream; forward() runs on streams that do not wait for it (and the
        # allocator may already have handed that work's freed scratch to the
        # routing buffers), so finish it here
        torch.cuda.current_stream(dev).synchronize()

    def forward(self, x: torch.Tensor, logits: torch.Tensor, stream=None) -> dict:
        b, ws, T = self.b, self.ws, x.shape[0]
        assert T == self.max_tokens, "buffers are sized for a fixed token count"
        E, H, F = self.E, self.H, self.F
        comp = self.compensate
        main = torch.cuda.current_stream() if stream is None else stream
        self.ev_fork.record(main)
        self.side.wait_event(self.ev_fork)
        plan = Q.moe_route(logits, self.topk, rows_capacity=self.cap, out=b["route"],
                           workspace=ws["rt"], stream=self.side)
        self.ev_plan.record(self.side)
        r1 = sel1 = w1sel = xr = None
        if comp and self.fused:
            # X's activation side in one cooperative launch: quantization,
            # channel scores, top-k and the second quantization of R_sel
            xq, sel1, _, xr = Q.quantize_select_nvfp4(
                x, self.k1, workspace=ws["qs1"], stream=stream,
                out=(b["xc"], b["xs"], b["xts"], b["sel1"], b["r1c"], b["r1s"], b["r1ts"]))
            self.ev_sel1.record(main)
        else:
            xq, xpart = Q.quantize_nvfp4(x, scores=comp, workspace=ws["q1"], stream=stream,
                                         out=(b["xc"], b["xs"], b["xts"], b["xpart"] if comp else None))
        self.ev_xq.record(main)
        self.side.wait_event(self.ev_xq)
        a1 = Q.moe_gather(plan, xq, out=(b["a1c"], b["a1s"]), stream=self.side)
        self.ev_a1.record(self.side)
        if comp and not self.fused:
            sel1, _, xr = Q.select_residual_channels(x, xq, xpart, self.k1, workspace=ws["s1"],
                                                     sel_ready_event=self.ev_sel1, stream=stream,
                                                     out=(b["sel1"], b["r1c"], b["r1s"], b["r1ts"]))
        if comp:
            self.wside.wait_event(self.ev_sel1)
            w1sel = Q.select_weight_channels(self.w1q, sel1, self.k1, E, stream=self.wside,
                                             out=(b["w1sc"], b["w1ss"]))
            self.ev_w1.record(self.wside)
        if comp:
            # R_sel's rows need only the plan, not the gather of X's rows
            main.wait_event(self.ev_plan)
            r1 = Q.moe_gather(plan, xr, out=(b["g1c"], b["g1s"]), stream=stream)
            main.wait_event(self.ev_w1)
        main.wait_event(self.ev_a1)
        # GEMM1's epilogue also leaves each expert's max |h| for h's tensor scale
        h = Q.moe_grouped_gemm(plan, a1, self.w1q, E, 2 * F, r1, sel1, self.k1,
                               epilogue=Q.EPI_SWIGLU, y_amax=b["hamax"], w_sel=w1sel,
                               out=b["h"], stream=stream)
        # h's padding rows (past each expert's count) are zero: not read
        r2 = sel2 = w2sel = None
        if comp and self.fused_h:
            # one block per expert: h's quantization, channel scores, top-k
            # and the second quantization of R_sel
            hq, sel2, _, r2 = Q.quantize_select_groups_nvfp4(
                h, self.k2, plan["offsets"], E, group_counts=plan["counts"],
                tensor_amax_in=b["hamax"], scale_layout=Q.TCGEN05, r_scale_layout=Q.TCGEN05,
                rows=self.cap, sel_ready_event=self.ev_sel2, workspace=ws["qs2"], stream=stream,
                out=(b["hc"], b["hs"], b["hts"], b["sel2"], b["r2c"], b["r2s"], b["r2ts"]))
        else:
            hq, hpart = Q.quantize_nvfp4(h, group_offsets=plan["offsets"], num_groups=E,
                                         group_counts=plan["counts"],
                                         tensor_amax_in=b["hamax"], scale_layout=Q.TCGEN05,
                                         scores=comp, rows=self.cap,
                                         workspace=ws["q2"], stream=stream,
                                         out=(b["hc"], b["hs"], b["hts"], b["hpart"] if comp else None))
        if comp and not self.fused_h:
            sel2, _, r2 = Q.select_residual_channels(h, hq, hpart, self.k2,
                                                     group_offsets=plan["offsets"], num_groups=E,
                                                     group_counts=plan["counts"],
                                                     r_scale_layout=Q.TCGEN05, workspace=ws["s2"],
                                                     sel_ready_event=self.ev_sel2, stream=stream,
                                                     out=(b["sel2"], b["r2c"], b["r2s"], b["r2ts"]))
        if comp:
            self.wside.wait_event(self.ev_sel2)
            w2sel = Q.select_weight_channels(self.w2q, sel2, self.k2, E, sel_per_group=True,
                                             stream=self.wside, out=(b["w2sc"], b["w2ss"]))
            self.ev_w2.record(self.wside)
            main.wait_event(self.ev_w2)
        y = Q.moe_grouped_gemm(plan, hq, self.w2q, E, H, r2, sel2, self.k2,
                               a_scale_per_expert=True, r_scale_per_expert=True,
                               sel_per_expert=True, w_sel=w2sel, out=b["y"], stream=stream)
        out = Q.moe_combine(y, plan, out=b["out"], stream=stream)
        self._a1, self._r1, self._w1sel = a1, r1, w1sel
        return dict(out=out, plan=plan, xq=xq, sel1=sel1, a1=a1, r1=r1, h=h, hq=hq, sel2=sel2,
                    r2=r2, y=y)

"""Benchmark of the NVFP4 W4A4 residual-compensation MoE expert layer on GB300.

One step = one pass of the rollout-side hot path over one batch: router top-8
and dispatch plan, NVFP4 quantization of the tokens with residual-energy
partials, top-k residual channel selection and second quantization, gather
into expert order, grouped compensated GEMM1 with the SwiGLU epilogue,
per-expert quantization and selection of h, grouped compensated GEMM2, and
the gate-weighted combine (weights are pre-quantized once, as after a weight
sync).  Workload: 8192 tokens, hidden 2048, 128 experts, top-8, expert FFN 768,
k = 64 selected channels per GEMM, seeded synthetic inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  `value` is the whole-job MoE GEMM throughput in TFLOP/s
(algorithmic FLOPs of both grouped GEMMs, main + correction, over real rows)
divided by the device-timed step; `e2e` is the same metric through the C ABI
from pinned host buffers with the copies inside the timed region.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = dict(tokens=8192, hidden=2048, experts=128, topk=8, ffn=768, k1=64, k2=64)
METRIC = "W4A4+residual-comp MoE GEMM TFLOPS (% FP4 peak); quantizer GB/s (% HBM)"
FP4_OVER_BF16 = 13.5 / 2.25          # nominal dense ratio used to scale the measured bf16 peak


def moe_flops(w=WORKLOAD) -> float:
    rows = w["tokens"] * w["topk"]
    H, F = w["hidden"], w["ffn"]
    g1 = 2.0 * rows * (2 * F) * (H + w["k1"])
    g2 = 2.0 * rows * H * (F + w["k2"])
    return g1 + g2


def gemm1_bytes(w=WORKLOAD) -> float:
    """Algorithmic HBM bytes of one grouped GEMM1 launch: NVFP4 weights of all
    experts (0.5625 B/element), NVFP4 A rows, the correction operands, bf16 h."""
    rows, H, F, E = w["tokens"] * w["topk"], w["hidden"], w["ffn"], w["experts"]
    kp = 64 if w["k1"] <= 64 else 128
    return (E * 2 * F * H * 0.5625 + rows * H * 0.5625 + rows * kp * 0.5625
            + E * 2 * F * kp * 0.5625 + rows * F * 2)


# DRAM traffic (read + write) of one GEMM1 launch at this workload, from the
# committed ncu capture of GEMM1; reset to None whenever gemm_kernel changes
# until a new capture is taken.
GEMM1_TRAFFIC_BYTES = 320.355072e6 + 92.516096e6


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index, self.proc, self.path = index, None, None

    def start(self):
        try:
            self.path = os.path.join(tempfile.gettempdir(), f"quads_clocks_{os.getpid()}.csv")
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names[1:], parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------- oracle leg
ORACLE_SAMPLE_EXPERTS = 2
REFERENCE_TOKENS = 2048        # per reference-arm step: a quarter of the batch


def oracle_sample(seed=0, tokens=None):
    """The oracle on a bounded sample of the workload: routing and activation
    quantization/selection of `tokens` tokens (default all), then the full
    expert FFN (both compensated GEMMs) of the first experts, with the router
    restricted to them.  Returns (flops, seconds)."""
    import numpy as np
    from nvfp4_w4a4_quantized_quant_gb300 import inputs
    from oracle import moe as M
    w = WORKLOAD
    d = inputs.moe_layer(seed, tokens=tokens or w["tokens"], hidden=w["hidden"],
                         experts=w["experts"], topk=w["topk"], ffn=w["ffn"], k=w["k1"],
                         with_weights=False)
    rng = inputs.make_rng(seed + 1)
    E, H, F = ORACLE_SAMPLE_EXPERTS, w["hidden"], w["ffn"]
    w1 = (rng.standard_normal((E, 2 * F, H), dtype=np.float32) * np.float32(0.02))
    w2 = (rng.standard_normal((E, H, F), dtype=np.float32) * np.float32(0.02))
    x = inputs.bf16_bits_to_f32(d["x"])
    w1q, w2q = M.quantize_weights(w1), M.quantize_weights(w2)
    logits = d["logits"][:, :E]             # routing restricted to the sampled experts
    t0 = time.perf_counter()
    res = M.moe_layer(x, logits, w1q, w2q, w["k1"], w["k2"], topk=min(w["topk"], E),
                      experts_subset=list(range(E)))
    dt = time.perf_counter() - t0
    rows = sum(len(res["tokens"][e]) for e in range(E))
    fl = 2.0 * rows * (2 * F) * (H + w["k1"]) + 2.0 * rows * H * (F + w["k2"])
    return fl, dt


def cpu_baseline(threads=None):
    threads = threads or len(os.sched_getaffinity(0))
    env = dict(os.environ, OMP_NUM_THREADS=str(threads), OPENBLAS_NUM_THREADS=str(threads),
               MKL_NUM_THREADS=str(threads), CUDA_VISIBLE_DEVICES="")
    code = ("import json,sys; sys.path.insert(0, %r); import bench; f,t=bench.oracle_sample(); "
            "print(json.dumps(dict(flops=f, seconds=t)))" % ROOT)
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=900)
    if out.returncode != 0:
        return {"value": None, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                "error": out.stderr.strip().splitlines()[-1:] }
    r = json.loads(out.stdout.strip().splitlines()[-1])
    return {"value": r["flops"] / r["seconds"] / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "seconds": round(r["seconds"], 2),
            "sample": f"all {WORKLOAD['tokens']} tokens routed/quantized/selected; expert FFN of "
                      f"{ORACLE_SAMPLE_EXPERTS} experts (router restricted to them), numpy float32/float64"}


# ----------------------------------------------------------------- GPU leg
def build_layer(torch, seed=0):
    import numpy as np
    from nvfp4_w4a4_quantized_quant_gb300 import inputs
    from nvfp4_w4a4_quantized_quant_gb300.layer import MoEExpertLayer
    w = WORKLOAD
    d = inputs.moe_layer(seed, tokens=w["tokens"], hidden=w["hidden"], experts=w["experts"],
                         topk=w["topk"], ffn=w["ffn"], k=w["k1"], with_weights=False)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    E, H, F = w["experts"], w["hidden"], w["ffn"]
    w1 = (torch.randn((E, 2 * F, H), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    w2 = (torch.randn((E, H, F), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    layer = MoEExpertLayer(w1, w2, w["topk"], w["k1"], w["k2"], w["tokens"])
    del w1, w2
    x_host = torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    l_host = torch.from_numpy(d["logits"]).pin_memory()
    return layer, x_host, l_host


def secondary(torch, Q, steps, flush, stream):
    """The other configurations of the scope table, each captured in a CUDA
    graph and timed like the step (L2 flushed before every replay):
    dense projection 4096x2048 x W 6144x2048 (k=128, bf16 Y) compensated and
    plain, the 512-token decode layer, TRACE rounding of 16384x2048 and the
    trainer-side W4A16 fake quantization of the expert gate/up weights."""
    import numpy as np
    from nvfp4_w4a4_quantized_quant_gb300 import inputs
    from nvfp4_w4a4_quantized_quant_gb300.layer import CompensatedLinear, MoEExpertLayer

    def check(tag):
        code = Q.device_status(stream)
        if code:
            raise RuntimeError(f"{tag}: device status {code}: "
                               f"{Q.load().quads_last_error_detail().decode()}")

    def graph_ms(fn):
        # inputs prepared on the default stream must be complete before `stream`
        # (which does not wait for the default stream) uses them
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            torch.cuda.synchronize()
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            ms = timed(torch, g.replay, steps, flush, stream) / steps
        check("secondary")
        return ms

    out = {}
    d = inputs.dense_projection(0)
    x = torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).cuda()
    w = torch.from_numpy(d["w"].view(np.int16)).view(torch.bfloat16).cuda()
    M, K = x.shape
    N = w.shape[0]
    k = 128
    dense = {}
    for comp in (True, False):
        lin = CompensatedLinear(w, k, M, compensate=comp)
        ms = graph_ms(lambda: lin.forward(x, stream=stream))
        fl = 2.0 * M * N * (K + (k if comp else 0))
        dense["comp" if comp else "plain"] = {"ms": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 1)}
        del lin
    dense["overhead_pct"] = round(100.0 * (dense["comp"]["ms"] / dense["plain"]["ms"] - 1.0), 1)
    dense["shape"] = {"M": M, "K": K, "N": N, "k": k, "y": "bf16"}
    out["dense_projection"] = dense

    # MXFP4 variant on the same shapes: quantizer of X, plain W4A4 GEMM
    wx, _ = Q.mx_quantize(w, scale_layout=Q.TCGEN05)
    ax, _ = Q.mx_quantize(x, scale_layout=Q.TCGEN05)
    ymx = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ms_q = graph_ms(lambda: Q.mx_quantize(x, scale_layout=Q.TCGEN05, out=(ax.codes, ax.scales),
                                          stream=stream))
    ms_g = graph_ms(lambda: Q.mx_gemm(ax, wx, out=ymx, stream=stream))
    qb = M * K * (2 + 0.5 + 1.0 / 32)
    out["mxfp4_dense_projection"] = {
        "quantize_ms": round(ms_q, 4), "quantize_gbs": round(qb / (ms_q * 1e-3) / 1e9, 1),
        "gemm_ms": round(ms_g, 4), "gemm_tflops": round(2.0 * M * N * K / (ms_g * 1e-3) / 1e12, 1),
        "shape": {"M": M, "K": K, "N": N, "y": "bf16"}}
    del x, w, wx, ax, ymx

    # the headline step without compensation (plain W4A4 both GEMMs): the
    # overhead of the residual compensation on the MoE layer
    wm = WORKLOAD
    dm = inputs.moe_layer(0, tokens=wm["tokens"], hidden=wm["hidden"], experts=wm["experts"],
                          topk=wm["topk"], ffn=wm["ffn"], k=wm["k1"], with_weights=False)
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    E, H, F = wm["experts"], wm["hidden"], wm["ffn"]
    w1 = (torch.randn((E, 2 * F, H), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    w2 = (torch.randn((E, H, F), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    xm = torch.from_numpy(dm["x"].view(np.int16)).view(torch.bfloat16).cuda()
    lm = torch.from_numpy(dm["logits"]).cuda()
    moe = {}
    for name, comp, fused, fused_h in (("plain", False, False, None), ("comp", True, False, None),
                                       ("comp_fused_activation_side", True, True, None),
                                       ("comp_fused_expert_side", True, False, True)):
        lay = MoEExpertLayer(w1, w2, wm["topk"], wm["k1"], wm["k2"], wm["tokens"], compensate=comp,
                             fused_activation_side=fused, fused_expert_side=fused_h)
        ms = graph_ms(lambda: lay.forward(xm, lm, stream=stream))
        moe[name] = {"ms": round(ms, 4)}
        del lay
    rows = wm["tokens"] * wm["topk"]
    fl_plain = 2.0 * rows * (2 * F) * H + 2.0 * rows * H * F
    moe["plain"]["tflops"] = round(fl_plain / (moe["plain"]["ms"] * 1e-3) / 1e12, 1)
    moe["comp"]["tflops"] = round(moe_flops() / (moe["comp"]["ms"] * 1e-3) / 1e12, 1)
    moe["overhead_pct"] = round(100.0 * (moe["comp"]["ms"] / moe["plain"]["ms"] - 1.0), 1)
    out["moe_step_plain_vs_comp"] = moe
    del w1, w2, xm, lm

    # quantizer (with residual-energy partials) over growing inputs, up to 2 GiB
    # of bf16: the asymptotic fraction of HBM bandwidth
    sweep = []
    for rows_q in (8192, 65536, 262144, 524288):
        Hq = 2048
        xq_in = torch.empty((rows_q, Hq), dtype=torch.bfloat16, device="cuda").normal_()
        wsq = torch.empty(Q.workspace_size(Q.OP_QUANTIZE, rows_q, Hq), dtype=torch.uint8, device="cuda")
        qo, po = Q.quantize_nvfp4(xq_in, scores=True, workspace=wsq)
        ms = graph_ms(lambda: Q.quantize_nvfp4(xq_in, scores=True, workspace=wsq,
                                               out=(qo.codes, qo.scales, qo.tensor_scale, po),
                                               stream=stream))
        # the quantize pass alone, with the tensor scale given (as when the
        # producer already knows the amax): x is read once
        ms1 = graph_ms(lambda: Q.quantize_nvfp4(xq_in, scores=True, workspace=wsq,
                                                tensor_scale_in=qo.tensor_scale,
                                                out=(qo.codes, qo.scales, qo.tensor_scale, po),
                                                stream=stream))
        # plain quantization (no residual-energy partials), tensor scale given
        ms0 = graph_ms(lambda: Q.quantize_nvfp4(xq_in, workspace=wsq,
                                                tensor_scale_in=qo.tensor_scale,
                                                out=(qo.codes, qo.scales, qo.tensor_scale, None),
                                                stream=stream))
        qb = rows_q * Hq * (2 + 0.5 + 1.0 / 16) + (rows_q // 32) * Hq * 4
        qb0 = rows_q * Hq * (2 + 0.5 + 1.0 / 16)
        sweep.append({"rows": rows_q, "cols": Hq, "input_mib": rows_q * Hq * 2 >> 20,
                      "ms": round(ms, 4), "gbs": round(qb / (ms * 1e-3) / 1e9, 1),
                      "ms_scale_given": round(ms1, 4),
                      "gbs_scale_given": round(qb / (ms1 * 1e-3) / 1e9, 1),
                      "ms_no_scores_scale_given": round(ms0, 4),
                      "gbs_no_scores_scale_given": round(qb0 / (ms0 * 1e-3) / 1e9, 1)})
        del xq_in, wsq, qo, po
    out["quantizer_sweep"] = sweep

    wl = dict(WORKLOAD, tokens=512)
    dd = inputs.moe_layer(0, tokens=512, hidden=wl["hidden"], experts=wl["experts"], topk=wl["topk"],
                          ffn=wl["ffn"], k=wl["k1"], with_weights=False)
    g = torch.Generator(device="cuda")
    g.manual_seed(1)
    E, H, F = wl["experts"], wl["hidden"], wl["ffn"]
    w1 = (torch.randn((E, 2 * F, H), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    w2 = (torch.randn((E, H, F), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    layer = MoEExpertLayer(w1, w2, wl["topk"], wl["k1"], wl["k2"], 512)
    layer2 = MoEExpertLayer(w1, w2, wl["topk"], wl["k1"], wl["k2"], 512, fused_expert_side=False)
    del w1, w2
    xd = torch.from_numpy(dd["x"].view(np.int16)).view(torch.bfloat16).cuda()
    ld = torch.from_numpy(dd["logits"]).cuda()
    ms = graph_ms(lambda: layer.forward(xd, ld, stream=stream))
    ms2 = graph_ms(lambda: layer2.forward(xd, ld, stream=stream))
    wbytes = E * (2 * F * H + H * F) * (0.5 + 1.0 / 16)
    out["moe_decode_512"] = {"ms": round(ms, 4), "weight_gbs": round(wbytes / (ms * 1e-3) / 1e9, 1),
                             "weight_bytes": int(wbytes), "frac_hbm": None,
                             "ms_expert_side_two_calls": round(ms2, 4)}
    del layer, layer2

    t = inputs.trace_rounding(0)
    xr = torch.from_numpy(t["x_rollout"].view(np.int16)).view(torch.bfloat16).cuda()
    xt = torch.from_numpy(t["x_train"].view(np.int16)).view(torch.bfloat16).cuda()
    rq, _ = Q.quantize_nvfp4(xr)
    codes = torch.empty((xt.shape[0], xt.shape[1] // 2), dtype=torch.uint8, device="cuda")
    cnt = torch.zeros(3, dtype=torch.int64, device="cuda")
    ms = graph_ms(lambda: Q.trace_round(xt, rq, counters=cnt, out=codes, stream=stream))
    tb = xt.numel() * (2 + 0.5 + 0.5 + 1.0 / 16)
    out["trace_16384x2048"] = {"ms": round(ms, 4), "gbs": round(tb / (ms * 1e-3) / 1e9, 1),
                               "algorithmic_bytes": int(tb)}
    # mantissa-only mode: pack the 1.5-bit record, then round from it
    bits = Q.trace_pack_record(rq)
    cnt1 = torch.zeros(2, dtype=torch.int64, device="cuda")
    ms_p = graph_ms(lambda: Q.trace_pack_record(rq, out=bits, stream=stream))
    ms_r = graph_ms(lambda: Q.trace_round_1bit(xt, bits, rq, counters=cnt1, out=codes,
                                               stream=stream))
    n = xt.numel()
    pb, rb = n * (0.5 + 1.0 / 8), n * (2 + 1.0 / 8 + 1.0 / 16 + 0.5)
    out["trace_1bit_16384x2048"] = {
        "pack_ms": round(ms_p, 4), "pack_gbs": round(pb / (ms_p * 1e-3) / 1e9, 1),
        "round_ms": round(ms_r, 4), "gbs": round(rb / (ms_r * 1e-3) / 1e9, 1),
        "algorithmic_bytes": int(rb), "record_bits_per_value": 1.5}
    del xr, xt, rq, codes, bits

    # trainer-side W4A16 fake quantization of the 128 experts' gate/up weights
    # (one tensor scale per expert; codes and scales written for the rollout copy)
    E, H, F = WORKLOAD["experts"], WORKLOAD["hidden"], WORKLOAD["ffn"]
    g = torch.Generator(device="cuda")
    g.manual_seed(2)
    wq = (torch.randn((E * 2 * F, H), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    offs = torch.arange(0, E * 2 * F + 1, 2 * F, dtype=torch.int32, device="cuda")
    yq = torch.empty_like(wq)
    ws = torch.empty(Q.workspace_size(Q.OP_QUANTIZE, wq.shape[0], H, 0, 0, E), dtype=torch.uint8,
                     device="cuda")
    ms = graph_ms(lambda: Q.qdq_nvfp4(wq, group_offsets=offs, num_groups=E, want_codes=True,
                                      workspace=ws, out=yq, stream=stream))
    qb = wq.numel() * (2 + 2 + 0.5 + 1.0 / 16)
    out["w4a16_qdq_w1"] = {"ms": round(ms, 4), "gbs": round(qb / (ms * 1e-3) / 1e9, 1),
                           "algorithmic_bytes": int(qb), "shape": [E * 2 * F, H],
                           "note": "bytes: x read once, bf16 y, codes + scales; the amax pass re-reads x"}
    return out


def timed(torch, fn, steps, flush, stream):
    """Sum of per-step device times (ms) with an L2 flush before each step."""
    tot = 0.0
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        tot += a.elapsed_time(b)
    return tot


def max_over_ranks(dist, values, device="cuda"):
    """Element-wise max of per-rank timings (the slowest rank sets the job
    time).  `dist` is torch.distributed (initialised) or None for one process."""
    if dist is None:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def run_gpu(args):
    import torch
    from nvfp4_w4a4_quantized_quant_gb300 import quads as Q
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    Q.load()
    pk = peaks()
    layer, x_host, l_host = build_layer(torch, seed=rank)
    x = x_host.cuda()
    logits = l_host.cuda()
    stream = torch.cuda.Stream()
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    flush = lambda: flush_buf.random_(0, 255)  # noqa: E731  (writes 256 MB > L2)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            layer.forward(x, logits)
        torch.cuda.synchronize()
        n0 = Q.kernel_launch_count()
        layer.forward(x, logits)
        torch.cuda.synchronize()
        launches_per_step = Q.kernel_launch_count() - n0
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            layer.forward(x, logits)
        torch.cuda.synchronize()
        code = Q.device_status(stream)
        assert code == 0, f"device status {code}: {Q.load().quads_last_error_detail().decode()}"

    def step():
        graph.replay()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        clocks = ClockSampler(local)
        clocks.start()
        time.sleep(0.3)
        torch.cuda.synchronize()
        t_ms = timed(torch, step, args.steps, flush, stream)
        clk = clocks.stop()

        # per-kernel timing of the dominant kernel (grouped GEMM1) inside the same stream
        plan = layer.b["route"]
        def g1():
            Q.moe_grouped_gemm(dict(plan, rows_capacity=layer.cap, experts=layer.E), layer._a1,
                               layer.w1q, layer.E, 2 * layer.F, layer._r1, layer.b["sel1"],
                               layer.k1, epilogue=Q.EPI_SWIGLU, w_sel=layer._w1sel,
                               out=layer.b["h"], stream=stream)
        # captured in a graph so that host-side launch work stays out of the timing
        g1_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1_graph, stream=stream):
            g1()
        g1_ms = timed(torch, g1_graph.replay, args.steps, flush, stream) / args.steps

        # quantizer alone on the layer input (scores on): algorithmic bytes
        xpart = torch.empty(((x.shape[0] + 31) // 32, x.shape[1]), dtype=torch.float32, device="cuda")
        xq_out = (layer.b["xc"], layer.b["xs"], layer.b["xts"], xpart)
        def qx():
            Q.quantize_nvfp4(x, scores=True, workspace=layer.ws["q1"], out=xq_out, stream=stream)
        q_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(q_graph, stream=stream):
            qx()
        q_ms = timed(torch, q_graph.replay, args.steps, flush, stream) / args.steps

        # GEMM1's whole activation side (quantize + select) in one cooperative launch
        b = layer.b
        qs_out = (b["xc"], b["xs"], b["xts"], b["sel1"], b["r1c"], b["r1s"], b["r1ts"])
        qs_ws = torch.empty(Q.workspace_size(Q.OP_QUANTIZE_SELECT, x.shape[0], x.shape[1], 0, layer.k1),
                            dtype=torch.uint8, device="cuda")
        def qs():
            Q.quantize_select_nvfp4(x, layer.k1, workspace=qs_ws, out=qs_out, stream=stream)
        qs_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(qs_graph, stream=stream):
            qs()
        qs_ms = timed(torch, qs_graph.replay, args.steps, flush, stream) / args.steps

        # end to end: every step copies its inputs from pinned host memory and
        # its output back; the copies of step i+1 (in) and i (out) run on their
        # own streams while step i+1 / i computes, with two input/output buffer
        # sets and one captured graph per set
        out_host = [torch.empty(layer.b["out"].shape, dtype=torch.bfloat16).pin_memory()
                    for _ in range(2)]
        xs, ls = [x, torch.empty_like(x)], [logits, torch.empty_like(logits)]
        outs = [layer.b["out"], torch.empty_like(layer.b["out"])]
        graphs = [graph, torch.cuda.CUDAGraph()]
        layer.b["out"] = outs[1]
        with torch.cuda.graph(graphs[1], stream=stream):
            layer.forward(xs[1], ls[1])
        layer.b["out"] = outs[0]
        torch.cuda.synchronize()
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()  # noqa: E731
        ev_in, ev_done, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        def e2e_run(n):
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(h2d)
            for i in range(n):
                b = i % 2
                if i >= 2:
                    h2d.wait_event(ev_done[b])        # step i-2 has read set b's inputs
                with torch.cuda.stream(h2d):
                    xs[b].copy_(x_host, non_blocking=True)
                    ls[b].copy_(l_host, non_blocking=True)
                ev_in[b].record(h2d)
                stream.wait_event(ev_in[b])
                if i >= 2:
                    stream.wait_event(ev_out[b])      # step i-2's output has left set b
                graphs[b].replay()
                ev_done[b].record(stream)
                d2h.wait_event(ev_done[b])
                with torch.cuda.stream(d2h):
                    out_host[b].copy_(outs[b], non_blocking=True)
                ev_out[b].record(d2h)
            t1.record(d2h)
            t1.synchronize()
            return t0.elapsed_time(t1)
        e2e_run(2)
        e2e_ms = e2e_run(args.steps)
    torch.cuda.synchronize()
    sec = secondary(torch, Q, args.steps, flush, stream) if rank == 0 else None

    ms = t_ms / args.steps
    e_ms = e2e_ms / args.steps
    ms, e_ms = max_over_ranks(dist, [ms, e_ms])
    if rank != 0:
        return
    if sec:
        dec = sec["moe_decode_512"]
        dec["frac_hbm"] = round(dec["weight_bytes"] / (dec["ms"] * 1e-3) / 1e9 / pk["hbm"], 4)
        tr = sec["trace_16384x2048"]
        tr["frac_hbm"] = round(tr["gbs"] / pk["hbm"], 4)
        t1 = sec["trace_1bit_16384x2048"]
        t1["frac_hbm"] = round(t1["gbs"] / pk["hbm"], 4)
        wq = sec["w4a16_qdq_w1"]
        wq["frac_hbm"] = round(wq["gbs"] / pk["hbm"], 4)
        for row in sec["quantizer_sweep"]:
            row["frac_hbm"] = round(row["gbs"] / pk["hbm"], 4)
            row["frac_hbm_scale_given"] = round(row["gbs_scale_given"] / pk["hbm"], 4)
            row["frac_hbm_no_scores_scale_given"] = round(row["gbs_no_scores_scale_given"] / pk["hbm"], 4)
    fl = moe_flops()
    value = world * fl / (ms * 1e-3) / 1e12
    e2e_val = world * fl / (e_ms * 1e-3) / 1e12
    T, H, E = WORKLOAD["tokens"], WORKLOAD["hidden"], WORKLOAD["experts"]
    q_bytes = T * H * 2 + T * H * 0.5 + T * H / 16 + (T // 32) * H * 4
    kp1 = 64 if WORKLOAD["k1"] <= 64 else 128
    qs_bytes = T * H * 2 + T * H * 0.5625 + T * kp1 * 0.5625     # x once, Q(X), Q(R_sel)
    # the timed region is a series of sub-millisecond graph replays, not a
    # seconds-long loop: the burst peak applies
    fp4_peak = pk["bf16"] * FP4_OVER_BF16
    g1_bytes = gemm1_bytes()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 (e2m1 codes, e4m3 block scales, fp32 tensor scale; fp32 accumulate)",
        "data": "synthetic (seeded: Student-t(4) tokens, N(0,1) router logits, N(0,0.02) weights)",
        "config": {"workload": "moe_expert_layer", **WORKLOAD, "l2": "flushed (256 MB write) before every step",
                   "graph": "CUDA graph replay of the whole step", "parallelism": "replicas" if world > 1 else "1 GPU"},
        "frac_of_fp4_peak": round(value / fp4_peak, 4),
        "fp4_peak_tflops": round(fp4_peak, 1),
        "fp4_peak_source": f"{pk['src']} bf16 burst {pk['bf16']} x nominal fp4/bf16 ratio {FP4_OVER_BF16}",
        "roofline": {
            "kernel": "grouped compensated GEMM1 (gate+up, SwiGLU epilogue)",
            "bound": "hbm",
            "achieved": round(g1_bytes / (g1_ms * 1e-3) / 1e9, 1),
            "peak": pk["hbm"],
            "unit": "GB/s",
            "frac": round(g1_bytes / (g1_ms * 1e-3) / 1e9 / pk["hbm"], 4),
            "traffic": GEMM1_TRAFFIC_BYTES,
            "ms": round(g1_ms, 4),
            "tflops": round(2.0 * T * WORKLOAD["topk"] * 2 * WORKLOAD["ffn"] * (H + WORKLOAD["k1"]) / (g1_ms * 1e-3) / 1e12, 1),
            "algorithmic_bytes": int(g1_bytes),
            "peak_source": pk["src"],
        },
        "secondary": sec,
        "quantizer": {"gbs": round(q_bytes / (q_ms * 1e-3) / 1e9, 1), "frac_hbm": round(q_bytes / (q_ms * 1e-3) / 1e9 / pk["hbm"], 4),
                      "ms": round(q_ms, 4), "shape": [T, H], "algorithmic_bytes": int(q_bytes),
                      "note": "amax pass + quantize pass with score partials (two launches)",
                      "fused_quantize_select_ms": round(qs_ms, 4),
                      "fused_quantize_select_gbs": round(qs_bytes / (qs_ms * 1e-3) / 1e9, 1),
                      "fused_note": "amax, quantization, scores, top-k, R_sel and its quantization in one "
                                    "cooperative launch (GEMM1's activation side; x read from HBM once)"},
        "e2e": {"value": round(e2e_val, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(x_host.numel() * 2 + l_host.numel() * 4),
                "d2h_bytes_per_step": int(out_host[0].numel() * 2), "ms_per_step": round(e_ms, 4),
                "timing": "pipelined: copies of step i+1 in / step i out overlap compute; "
                          "no L2 flush (weights and activations exceed L2)"},
        "gpu_launches": int(launches_per_step * args.steps),
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_profile(args):
    """Plain sequences of eager calls (no graph, no flush, no clock sampling)
    for an ncu launch list or a single-kernel capture:
      moe     the MoE expert layer step (8192 tokens)
      dense   the compensated dense projection 4096x2048 x 6144x2048, k = 128
      decode  the MoE expert layer on 512 tokens
      streams the streaming kernels: TRACE rounding, record packing and 1-bit
              rounding on 16384x2048; quantization of 8192x2048 with score
              partials (amax + quantize); plain quantization of 262144x2048
              with the tensor scale given"""
    import numpy as np
    import torch
    from nvfp4_w4a4_quantized_quant_gb300 import inputs
    from nvfp4_w4a4_quantized_quant_gb300 import quads as Q
    from nvfp4_w4a4_quantized_quant_gb300.layer import CompensatedLinear, MoEExpertLayer
    torch.cuda.set_device(0)
    Q.load()
    if args.profile == "dense":
        d = inputs.dense_projection(0)
        x = torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).cuda()
        w = torch.from_numpy(d["w"].view(np.int16)).view(torch.bfloat16).cuda()
        lin = CompensatedLinear(w, 128, x.shape[0])
        step = lambda: lin.forward(x)  # noqa: E731
    elif args.profile == "streams":
        t = inputs.trace_rounding(0)
        xr = torch.from_numpy(t["x_rollout"].view(np.int16)).view(torch.bfloat16).cuda()
        xt = torch.from_numpy(t["x_train"].view(np.int16)).view(torch.bfloat16).cuda()
        rq, _ = Q.quantize_nvfp4(xr)
        codes = torch.empty((xt.shape[0], xt.shape[1] // 2), dtype=torch.uint8, device="cuda")
        cnt = torch.zeros(3, dtype=torch.int64, device="cuda")
        bits = Q.trace_pack_record(rq)
        cnt1 = torch.zeros(2, dtype=torch.int64, device="cuda")
        g = torch.Generator(device="cuda")
        g.manual_seed(3)
        xs = torch.randn((8192, 2048), generator=g, device="cuda").to(torch.bfloat16)
        xl = torch.randn((262144, 2048), generator=g, device="cuda").to(torch.bfloat16)
        ws = torch.empty(Q.workspace_size(Q.OP_QUANTIZE, 262144, 2048), dtype=torch.uint8,
                         device="cuda")
        qs, ps = Q.quantize_nvfp4(xs, scores=True, workspace=ws)
        ql, _ = Q.quantize_nvfp4(xl, workspace=ws)

        def step():
            Q.trace_round(xt, rq, counters=cnt, out=codes)
            Q.trace_pack_record(rq, out=bits)
            Q.trace_round_1bit(xt, bits, rq, counters=cnt1, out=codes)
            Q.quantize_nvfp4(xs, scores=True, workspace=ws,
                             out=(qs.codes, qs.scales, qs.tensor_scale, ps))
            Q.quantize_nvfp4(xl, workspace=ws, tensor_scale_in=ql.tensor_scale,
                             out=(ql.codes, ql.scales, ql.tensor_scale, None))
    else:
        w = dict(WORKLOAD, tokens=512) if args.profile == "decode" else WORKLOAD
        d = inputs.moe_layer(0, tokens=w["tokens"], hidden=w["hidden"], experts=w["experts"],
                             topk=w["topk"], ffn=w["ffn"], k=w["k1"], with_weights=False)
        g = torch.Generator(device="cuda")
        g.manual_seed(0)
        E, H, F = w["experts"], w["hidden"], w["ffn"]
        w1 = (torch.randn((E, 2 * F, H), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
        w2 = (torch.randn((E, H, F), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
        layer = MoEExpertLayer(w1, w2, w["topk"], w["k1"], w["k2"], w["tokens"])
        x = torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).cuda()
        logits = torch.from_numpy(d["logits"]).cuda()
        step = lambda: layer.forward(x, logits)  # noqa: E731
    torch.cuda.synchronize()
    for _ in range(args.warmup + args.steps):
        step()
    torch.cuda.synchronize()
    assert Q.device_status() == 0
    print(json.dumps({"profile": args.profile, "profile_steps": args.warmup + args.steps,
                      "launches": Q.kernel_launch_count()}))


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    fl_tot, t_tot = 0.0, 0.0
    for _ in range(args.warmup):
        pass                      # the oracle has no warm-up state; warm-up steps are not repeated
    for s in range(args.steps):
        fl, dt = oracle_sample(seed=s, tokens=REFERENCE_TOKENS)
        fl_tot += fl
        t_tot += dt
    v = fl_tot / t_tot / 1e12
    threads = len(os.sched_getaffinity(0))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_tot / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4 values in float32/float64 (numpy)", "data": "synthetic",
        "config": {"workload": "moe_expert_layer", **WORKLOAD},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step: {REFERENCE_TOKENS} tokens routed/quantized/selected, expert FFN of {ORACLE_SAMPLE_EXPERTS} experts (router restricted to them)"},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="libquads", choices=["libquads", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", nargs="?", const="moe", default=None,
                    choices=["moe", "dense", "decode", "streams"],
                    help="eager steps only (MoE step, dense projection, decode layer or the "
                         "streaming kernels), for ncu")
    args = ap.parse_args()
    if args.warmup < 3 and not args.profile:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.profile:
        run_profile(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()

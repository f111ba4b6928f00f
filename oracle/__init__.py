"""CPU oracle for the NVFP4 W4A4 residual-compensation path (test infrastructure).

This package is the slow, plain reference that the CUDA path is checked
against.  It is test infrastructure only: the test suite, the smoke check and
the benchmark's CPU-baseline leg may import it; the library and its Python
binding never do, and the two share no code, tables or helpers.

Everything is written with numpy in float32 where the method fixes float32
rounding (so that integer decisions -- codes, scale bytes, selected channels
-- are taken in the same precision as on the GPU), and in float64 where a
plain mathematical value is wanted (GEMM accumulation, softmax, SwiGLU).

Sources (page title, then the section used):
  [QUADS]  "Technical Summary: QUADS - Stabilizing NVFP4 Reinforcement Learning
           for MoE via Quantization-error Alignment" (gist.science), sections 1
           "Problem Statement", 2.1 "Error Analysis and Diagnosis", 2.2 B
           "Residual Activation Compensation (Rollout Side)", 4 "Experimental
           Results".
  [QUADS-news] "阿里:QUADS稳定MoE强化学习" (yfxerp.com news digest), "重点思路".
  [TRACE]  "TRACE: Rollout-Guided Quantization-Aware Training for FP4
           Reinforcement Learning of MoE Language Models" (paper.rainbus.top
           digest), sections "NVFP4 与 E2M1 码本" (the NVFP4 / E2M1 codebook),
           "研究动机" (motivation, worked boundary example), "核心方法" (core
           method, Eq. (3)), "方法步骤详情" (method steps), "MoE 专家路由敏感性"
           (MoE routing sensitivity).

Parity status: every function here is pinned by a CPU test (tests/test_oracle_*)
against values the pages print, a library routine, closed forms, invariants or
brute force.  The cross-path differences the TRACE digest quotes for QUADS
(0.09 -> 0, 0 -> 0.10, 0.99) come from inputs the pages do not give and are
not reproduced; the function computing that quantity is pinned by a closed form.
"""

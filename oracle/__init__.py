"""CPU oracle for the low-bit routed-expert FFN.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import this package.  The product path (the CUDA library
and its Python binding) never imports, links or executes anything here, and
this package shares no code with it: the two meet only at the seeded input
generators in ``bit_moe_expert_top_gb300.synth``, which hold no arithmetic of
the method.

The oracle is a plain, slow, obviously-correct restatement of what the layer
computes, written from the pages' problem statement:

  * 2-bit codebook {-4,-1,1,4} experts with one fp16 scale per 32 weights
    (blog "这个项目我们能学到什么?" on vLLM-Moet; vLLM-Moet README, line table,
    "2-bit experts on vLLM v0.24.0");
  * MXFP4 experts, E2M1 values with one E8M0 scale per 32 (OCP Microscaling
    Formats v1.0; vLLM-Moet README, "MoET hybrid": "the checkpoint's MXFP4
    bytes"), used as an FP4 "delta cache" of hot experts;
  * MXFP4 -> FP8 online conversion into a reused workspace ("国产GPU完成MoE大模型
    Day-0适配", §四);
  * top-k softmax routing, per-expert grouping, FC1 (gate/up) + SwiGLU, FC2
    (vLLM-Moet README, release v2026.11.03-r23 notes: "FC1 + SwiGLU + MXFP8
    quant, FC2"), and a weighted combine.

Floating point: every dot product is accumulated in fp64 and rounded once to
fp32 where the definition stores an fp32 value (g, u, routing weights,
output); the bf16 / e4m3 / MXFP8 rounding points of the precision profiles are
applied exactly where the definition places them.

Functions without an independent pin say "parity unpinned" in their
docstring; at present every public function is pinned by ``tests/test_oracle_*``.
"""
from . import codecs, moe  # noqa: F401

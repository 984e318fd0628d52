"""Oracle for the MoE layer hot path: a plain, slow, CPU-only restatement of
what the layer computes, in fp64 wherever the computation is floating point.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import this package.  The CUDA library never
calls it, and it shares no code with the CUDA library.

Sources (page titles as published):
  [EP]   "Expert parallelism" (zerotofrontier.app, MoE chapter, section 13.x)
  [EPS]  "Expert Parallelism at Scale" (study notes on DeepSeek-V2/V3)
  [EPM]  "05 - Expert Parallelism (MoE)" (inference-engineering roadmap notes)
  [SPR]  "Spreading the Experts" (parallelism plate 9 of 11)

Parity status: every function here is pinned by a CPU test against values or
identities that do not come from this module (tests/test_oracle_pins.py): the
pages' hand dispatch and load-imbalance examples, brute-force routing on tiny
inputs, library routines for the special cases (single expert = one SwiGLU MLP,
k = E softmax = dense softmax), a dense-mask brute force of the whole layer and
the pages' byte model.  The pages' capacity-padding percentages (7 %, 0.5 %,
under 3 %) are not reproduced: their workload is not printed (parity unpinned
for those figures; no function here claims them).

A second statement of the forward path, one token at a time in plain C (fp64,
counting sorts, per-token expert loops), lives in moe_loop.c and is reached
through oracle.loop; it is pinned by tests/test_oracle_loop.py (the hand
dispatch, brute-force routing, closed forms, planted mistakes) and agrees with
the numpy statement to 1e-12.
"""
from .moe_ref import *  # noqa: F401,F403

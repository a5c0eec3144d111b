"""CPU oracle for the FP8 up-projection hot path -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct numpy code (fp64 where the method does not fix the
precision).  Only the tests, the smoke check and the bench's CPU-baseline leg may
import it; the library's product path never does, and this package imports nothing
from the library.

Sources (the three web pages on FP8 mixed-precision training):

* "FP8 stability guardrails" page (zenaique), section "Why FP8 is tempting and why it
  is fragile": E4M3 = 4 exponent + 3 mantissa bits with maximum 448, E5M2 = 5 + 2 bits
  with maximum about 57344; values above the maximum overflow or saturate, values far
  below it underflow to zero.  Same page, "Real products, models, and research":
  fine-grained tile and block scaling (DeepSeek-V3), delayed scaling with an amax
  history (Transformer Engine).  "What an interviewer would ask next": E4M3 and E5M2
  in one run (forward operands vs the backward signal).
* "#84 FP8 Precision" speedrun page, sections "Explanation" and "Hardware precision":
  weights divided by a scale before the E4M3 cast, a scaled FP8 matmul with per-operand
  scales, an FP8 copy of the bf16 master weight re-quantised after every optimizer step.

Modules: ``fp8`` (formats, cast), ``quant`` (amax, scales, counters, tile/block,
delayed state), ``gemm`` (scaled matmuls and the error bound), ``linear``
(forward/backward compositions and the delayed-scaling training loop).

Parity status per function is stated in each module header.  Functions whose
definition the pages leave open follow a stated reading; the delayed-scaling state
machine (``quant.DelayedState``) is "parity unpinned" by the pages beyond its
invariants.
"""

"""CPU oracle for mixed-precision quantized KV-cache decode (TEST INFRASTRUCTURE ONLY).

A plain, slow, obviously-correct restatement of what the decode hot path
computes, written from the three pages it follows:

  * "EchoKV: watching a language model decide its own precision" — the FP16
    K_ref ring, the canary KL, the EMA and the lowest-bit-under-tau pick, and
    forward-only (admit-time) tier changes; the KIVI-style asymmetric
    quantizer (`quant.quantize_asym`); the controller variants and the
    majority vote over ranks (`controller`);
  * "Behavior-Guided KV-Cache Quantization" — K quantized per channel, V per
    token, symmetric; packed low-bit storage; GQA head mapping; the
    static-artifact mode (percentile clipping thresholds, role-specific
    candidate scores, AutoK layer allocation: `artifacts`);
  * "KV-Kaizen" — symmetric uniform quantization, bits-per-token accounting.

Only `tests/`, `__graft_entry__.smoke()` and `bench.py`'s CPU-baseline leg
may import this package.  The product (the CUDA library and its binding)
never does; it shares no code with this package.

Numerics: quantization is restated exactly (fp32 division, RNE to the fp16
scale, RNE to the integer code, clamp); attention and KL are accumulated in
fp64.  Every function names the passage it follows.  Functions whose values
have no independent pin say "parity unpinned" in their docstring.
"""
from . import quant, pages, attention, canary, controller, decoder, sizes, artifacts  # noqa: F401

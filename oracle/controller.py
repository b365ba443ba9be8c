"""EMA smoothing and lowest-bit-under-tau tier pick (oracle).

Follows "EchoKV: watching a language model decide its own precision",
"Show the math": the EMA equation EMA_{t+1} = (1-alpha) EMA_t + alpha delta,
and the pick b_l = min{ b in {2,4,8} : EMA_{l,b} < tau }, recomputed from
scratch on every firing (promote and demote, "Bidirectional adjustment").

Readings:
  * alpha comes from the workload (0.25); the page's 0.1 is its own setting;
  * the first observation sets the EMA (no zero start, which would bias the
    first readings low by 1/alpha);
  * if no candidate is under tau the layer takes the widest candidate, 8 bits
    (the page shows layers "upgraded" to INT8 and workloads that "cascade" to
    INT8; FP16 is only the display state before the first firing);
  * the EMA is evaluated in fp32 as t1 = (1-alpha)*ema, t2 = alpha*delta,
    ema = t1 + t2, each operation rounded separately (no fused multiply-add);
  * a frozen controller (the page's freeze_controller) changes nothing.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
BITS = (2, 4, 8)


def ema_step(ema, delta, alpha: float):
    """One EMA update in fp32; `ema` None means first observation."""
    delta = np.asarray(delta, dtype=F32)
    if ema is None:
        return delta.copy()
    a = F32(alpha)
    one_minus = F32(F32(1.0) - a)
    t1 = (one_minus * np.asarray(ema, dtype=F32)).astype(F32)
    t2 = (a * delta).astype(F32)
    return (t1 + t2).astype(F32)


def pick(ema, tau: float) -> int:
    t = F32(tau)
    for i, b in enumerate(BITS):
        if F32(ema[i]) < t:
            return b
    return BITS[-1]


class Controller:
    """Per-layer EMA state and tiers; update() applies one canary firing."""

    def __init__(self, tiers, alpha: float, tau: float):
        self.tiers = [int(t) for t in tiers]
        self.ema = [None] * len(self.tiers)
        self.alpha = alpha
        self.tau = tau

    def update(self, deltas, mask=None, freeze: bool = False):
        if freeze:
            return
        for l, dl in enumerate(deltas):
            if mask is not None and not mask[l]:
                continue
            self.ema[l] = ema_step(self.ema[l], dl, self.alpha)
            self.tiers[l] = pick(self.ema[l], self.tau)

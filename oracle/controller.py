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

Variants ("The tau(L) scaling"; the hysteresis and multi-firing vote the
page proposes against seed drift, "Why does the controller drift across
seeds"), each off by default:
  * tau_ctx0 > 0: budget = tau * sqrt(L / tau_ctx0), L = (sum of the lengths of
    the layer's sequences that hold tokens) / (their count), every operation in
    fp32 with one rounding (L is the context length the page's formula takes;
    a batch shares the layer's tier, so its mean length stands in);
  * hysteresis h: a pick of fewer bits than the current tier must satisfy
    ema_b < budget * (1 - h) (reading: demotions need margin, promotions do not);
  * vote k: the tier changes only after k consecutive firings picked the same
    new tier; a firing that picks the current tier resets the count.
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


def pick(ema, tau: float, cur: int | None = None, hysteresis: float = 0.0) -> int:
    t = F32(tau)
    lower = F32(t * F32(F32(1.0) - F32(hysteresis)))
    for i, b in enumerate(BITS):
        thr = lower if cur is not None and b < cur else t
        if F32(ema[i]) < thr:
            return b
    return BITS[-1]


def budget(tau: float, tau_ctx0: int, lengths) -> np.float32:
    """The pick's threshold: tau, or tau * sqrt(mean length / tau_ctx0)."""
    t = F32(tau)
    if tau_ctx0 <= 0:
        return t
    act = [int(x) for x in lengths if int(x) > 0]
    if not act:
        return t
    mean = F32(F32(sum(act)) / F32(len(act)))
    return F32(t * np.sqrt(F32(mean / F32(tau_ctx0)), dtype=F32))


class Controller:
    """Per-layer EMA state and tiers; update() applies one canary firing."""

    def __init__(self, tiers, alpha: float, tau: float, tau_ctx0: int = 0,
                 hysteresis: float = 0.0, vote: int = 1):
        self.tiers = [int(t) for t in tiers]
        self.ema = [None] * len(self.tiers)
        self.alpha = alpha
        self.tau = tau
        self.tau_ctx0, self.hysteresis, self.vote = tau_ctx0, hysteresis, max(1, vote)
        self.cand = [0] * len(self.tiers)
        self.count = [0] * len(self.tiers)

    def update(self, deltas, mask=None, freeze: bool = False, lengths=None):
        """`lengths[l]`: the cached lengths of layer l's sequences (tau_ctx0 > 0)."""
        if freeze:
            return
        for l, dl in enumerate(deltas):
            if mask is not None and not mask[l]:
                continue
            self.ema[l] = ema_step(self.ema[l], dl, self.alpha)
            b = budget(self.tau, self.tau_ctx0, [] if lengths is None else lengths[l])
            new = pick(self.ema[l], b, self.tiers[l], self.hysteresis)
            if new == self.tiers[l]:
                self.count[l] = 0
                continue
            n = self.count[l] + 1 if self.cand[l] == new else 1
            if n >= self.vote:
                self.tiers[l] = new
                n = 0
            self.cand[l] = new
            self.count[l] = n


def majority_vote(tier_vectors):
    """Consolidation across ranks before the freeze ("Measurement protocol",
    phase 2: "majority vote per layer").  Reading: the most frequent tier of
    each layer; among tied tiers, the widest."""
    L = len(tier_vectors[0])
    result = []
    for l in range(L):
        column = [int(v[l]) for v in tier_vectors]
        best, best_n = None, -1
        for b in sorted(set(column), reverse=True):     # widest first: wins ties
            n = column.count(b)
            if n > best_n:
                best, best_n = b, n
        result.append(best)
    return result

"""Static-artifact mode: offline calibration that freezes clipping thresholds
(theta*) and per-layer K bits (b*), and the read-only online configuration.

Follows "Behavior-Guided KV-Cache Quantization": the framework figure
("Freeze & allocate": theta* and b* are fixed artifacts; "Online inference":
load them read-only, pack the cache, decode), "Calibration protocol" (scores
of candidate parameters on a fixed calibration set, then frozen), "K/V
Role-Aware Low-Bit Quantization" (Key candidates scored by attention KL, Value
candidates by the perturbation of the attention output) and
"Sensitivity-Driven Budget Allocation" (AutoK protects the fewest most
sensitive layers that reach a fraction of the total sensitivity).

Every step runs in the library: thresholds by its percentile select, Key
scores by its canary (which quantizes with the layer's thresholds), Value
scores by its append and decode attention, AutoK by its host allocator.  The
calibration set is synthetic: each sequence's prefill tokens of the workload
and the first decode step's queries.

Definitions:
  * threshold = nearest-rank quantile of |x| (rank max(1, ceil(q n))), K per
    (KV head, channel) over all calibration tokens, V per KV head over all
    calibration tokens and channels;
  * Key score of a candidate = the canary's KL at `low` bits over each
    sequence's newest 64 calibration keys with the candidate's K thresholds;
  * Value score = sum ||o(K, Vhat) - o(K, V)||^2 / sum ||o(K, V)||^2, o the
    decode attention with 16-bit K over the whole calibration context and V
    at the layer's bits with the candidate's V thresholds (exactly 0 at 16 bits);
  * the lowest score wins, equal scores go to the larger percentile;
  * sensitivity = the Key score of the chosen candidate; AutoK over the
    sensitivities gives the protected layers (`high` K bits), the rest `low`.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import ekv, workloads

RING = 64
CANARY_BITS = (2, 4, 8)


@dataclasses.dataclass
class Artifact:
    """Frozen calibration output of one model shape."""
    k_bits: list            # [L] K bits (b*)
    v_bits: list            # [L] V bits
    k_clip: np.ndarray      # [L, Hkv, d] float32 K thresholds (+inf: none)
    v_clip: np.ndarray      # [L, Hkv] float32 V thresholds
    k_percentile: list      # [L] chosen Key candidate
    v_percentile: list      # [L] chosen Value candidate
    sensitivity: list       # [L] Key score at the chosen candidate
    frac: float
    low: int
    high: int

    def save(self, path) -> None:
        np.savez(path, k_bits=np.asarray(self.k_bits, np.int32),
                 v_bits=np.asarray(self.v_bits, np.int32),
                 k_clip=np.asarray(self.k_clip, np.float32),
                 v_clip=np.asarray(self.v_clip, np.float32),
                 k_percentile=np.asarray(self.k_percentile, np.float64),
                 v_percentile=np.asarray(self.v_percentile, np.float64),
                 sensitivity=np.asarray(self.sensitivity, np.float64),
                 alloc=np.asarray([self.frac, self.low, self.high], np.float64))

    @classmethod
    def load(cls, path) -> "Artifact":
        """Read an artifact; its arrays come back read-only."""
        with np.load(path) as z:
            a = {k: z[k].copy() for k in z.files}
        for v in a.values():
            v.setflags(write=False)
        frac, low, high = a["alloc"].tolist()
        return cls([int(b) for b in a["k_bits"]], [int(b) for b in a["v_bits"]], a["k_clip"],
                   a["v_clip"], a["k_percentile"].tolist(), a["v_percentile"].tolist(),
                   a["sensitivity"].tolist(), frac, int(low), int(high))

    def apply(self, cache: ekv.Cache, stream=None) -> None:
        """Load b* as the tiers and theta* as every layer's thresholds."""
        L = len(self.k_bits)
        if cache.num_layers != L:
            raise ValueError("artifact and cache disagree on the layer count")
        if list(cache.v_bits) != list(self.v_bits):
            raise ValueError("the cache's V bits are not the artifact's")
        cache.set_tiers(self.k_bits, stream)
        for l in range(L):
            cache.set_clip(l, self.k_clip[l], self.v_clip[l], stream)

    def workload(self, w: workloads.Workload) -> workloads.Workload:
        """`w` run in static mode: b* as the initial tiers, no canary firings."""
        return w.scaled(k_bits_init=list(self.k_bits), v_bits=list(self.v_bits),
                        canary_period=0)


def cache_for(art: Artifact, w: workloads.Workload, device=None) -> ekv.Cache:
    """A cache for `w` configured read-only from the artifact."""
    c = ekv.cache_for(art.workload(w), device=device)
    art.apply(c)
    return c


def _choose(candidates, scores) -> int:
    return min(range(len(candidates)), key=lambda i: (float(scores[i]), -float(candidates[i])))


def calibrate(w: workloads.Workload, candidates=(1.0, 0.999, 0.99), frac: float = 0.9,
              low: int = 4, high: int = 8, device=None):
    """Run the offline calibration on the workload's synthetic draws.

    Returns (Artifact, scores) with scores = {"k_score", "v_score": [L][n_cand]
    fp64, "k_choice", "v_choice": [L] candidate indices, "order": AutoK order,
    "n_protected": k}."""
    if low not in CANARY_BITS or high not in (4, 8, 16) or high <= low:
        raise ValueError("need low in {2, 4, 8} and a wider high")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    L, B, H, d = w.num_layers, w.batch, w.num_kv_heads, w.head_dim
    slots = torch.arange(B, dtype=torch.int32, device=dev)
    bi = CANARY_BITS.index(low)
    T = list(w.prefill)
    pages = sum((t + 15) // 16 for t in T) * H

    def one_layer(kb, vb):
        return ekv.Cache(1, B, w.num_q_heads, H, d, max(T), {(kb, vb): pages}, [kb], [vb],
                         device=dev)

    def fill(c, kk, vv):
        for s in range(B):
            c.reset(s)
            c.append(0, slots[s:s + 1], kk[s][None], vv[s][None])

    out = {"k_score": [], "v_score": [], "k_choice": [], "v_choice": []}
    k_clip, v_clip, sens = [], [], []
    delta = torch.zeros(3, dtype=torch.float32, device=dev)
    o = torch.empty(B, w.num_q_heads, d, dtype=torch.float16, device=dev)
    oq = torch.empty_like(o)
    ref = one_layer(16, 16)          # raw K/V: its ring is the Key window, its output o(K, V)
    try:
        for l in range(L):
            ks, vs = [], []
            for s in range(B):
                k, v = w.prefill_kv(l, [s], device=dev, n_tok=T[s])
                ks.append(k[0])
                vs.append(v[0])
            K, V = torch.cat(ks), torch.cat(vs)
            Q = w.step_q(l, 0, 1, device=dev)[:, 0].contiguous()
            kc = [ekv.k_thresholds(K, q) for q in candidates]
            vc = [ekv.v_thresholds(V, q) for q in candidates]
            fill(ref, ks, vs)
            kscore = []
            for c in kc:             # Key: the canary over each sequence's newest 64 keys
                ref.set_clip(0, c.cpu(), None)
                ref.canary_kl(0, slots, Q, delta)
                kscore.append(float(delta[bi].item()))
            vb = w.v_bits[l]
            if vb == 16:
                vscore = [0.0] * len(candidates)
            else:                    # Value: attention output, 16-bit K, V at the layer's bits
                ref.decode_attn(0, slots, Q, o)
                quant = one_layer(16, vb)
                try:
                    vscore = []
                    for c in vc:
                        quant.set_clip(0, None, c.cpu())
                        fill(quant, ks, vs)
                        quant.decode_attn(0, slots, Q, oq)
                        num, den = ekv.output_error(oq, o)      # fp64 sums on the GPU
                        vscore.append(num / den if den > 0 else 0.0)
                    quant.sync()
                finally:
                    quant.close()
            i, j = _choose(candidates, kscore), _choose(candidates, vscore)
            k_clip.append(kc[i].cpu().numpy())
            v_clip.append(vc[j].cpu().numpy())
            sens.append(kscore[i])
            out["k_score"].append(kscore)
            out["v_score"].append(vscore)
            out["k_choice"].append(i)
            out["v_choice"].append(j)
        ref.sync()
    finally:
        ref.close()
    k, order = ekv.autok(sens, frac)
    top = set(order[:k])
    bits = [high if l in top else low for l in range(L)]
    out["order"], out["n_protected"] = order, k
    art = Artifact(bits, list(w.v_bits), np.stack(k_clip).astype(np.float32),
                   np.stack(v_clip).astype(np.float32),
                   [candidates[i] for i in out["k_choice"]],
                   [candidates[j] for j in out["v_choice"]], sens, frac, low, high)
    return art, out

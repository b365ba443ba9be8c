"""Static-artifact mode: percentile clipping thresholds, the AutoK allocator and
the offline calibration that produces them (oracle; TEST INFRASTRUCTURE ONLY).

Follows "Behavior-Guided KV-Cache Quantization":
  * "Calibration protocol": candidate quantization parameters are scored on a
    fixed calibration set, and the selected scales, clipping thresholds and
    layer sensitivity readings are frozen before use;
  * "K/V Role-Aware Low-Bit Quantization": the percentile candidates for Key
    are scored by the KL between reference and quantized attention
    distributions, those for Value by the perturbation of the attention
    output;
  * "Sensitivity-Driven Budget Allocation": the most sensitive layers get a
    higher-precision path; AutoK picks the smallest number of protected layers
    whose sensitivities reach a given fraction of the total;
  * the framework figure ("Freeze & allocate", "Online inference"): the
    artifacts theta* (thresholds) and b* (per-layer bits) are loaded read-only,
    then the cache is packed and decoded with them.

Readings (the pages give no formulas for these steps):
  * a threshold is the nearest-rank percentile of |x|: with the n values
    sorted ascending, the value of 1-based rank max(1, ceil(q * n)) (q * n in
    IEEE fp64), so it is always one of the data's own magnitudes;
  * K thresholds are per (KV head, channel) over every calibration token, V
    thresholds per KV head over every calibration token and channel (K is
    quantized per channel, V per token; a per-token threshold cannot be
    frozen, a per-head one can);
  * the Key score of a candidate is the canary's KL at the low bit-width over
    each sequence's newest 64 calibration keys (the same window and quantizer
    the online canary uses), with the candidate's thresholds; the Value score
    is sum ||o(K, Vhat) - o(K, V)||^2 / sum ||o(K, V)||^2 over every query head
    and sequence, o the decode attention over the whole calibration context
    with raw fp16 K;
  * the lowest score wins; equal scores go to the larger percentile (less
    clipping);
  * a layer's sensitivity is its Key score at the chosen candidate;
  * AutoK orders layers by sensitivity, largest first (equal sensitivities:
    lower layer first), and protects the shortest prefix whose fp64 sum,
    accumulated in that order, is >= frac times the sum of all of them; the
    protected layers take `high` K bits, the rest `low`.
"""
from __future__ import annotations

import math

import numpy as np

from . import attention, canary, quant

F16 = np.float16
F32 = np.float32
RING = 64


def nearest_rank(n: int, q: float) -> int:
    """1-based rank of the q-th quantile among n sorted values."""
    if n < 1 or not (0.0 <= q <= 1.0):
        raise ValueError("need n >= 1 and 0 <= q <= 1")
    return min(max(math.ceil(q * n), 1), n)


def abs_percentile(x16, q: float) -> F32:
    """Nearest-rank q-quantile of |x| over every element of fp16 `x16`."""
    a = np.sort(np.abs(np.asarray(x16, dtype=F16).astype(F32)).ravel())
    return F32(a[nearest_rank(a.size, q) - 1])


def k_thresholds(k16, q: float) -> np.ndarray:
    """Per (head, channel) thresholds [H, d] from calibration keys [T, H, d]."""
    k16 = np.asarray(k16, dtype=F16)
    _, H, d = k16.shape
    return np.array([[abs_percentile(k16[:, h, c], q) for c in range(d)] for h in range(H)],
                    dtype=F32)


def v_thresholds(v16, q: float) -> np.ndarray:
    """Per head thresholds [H] from calibration values [T, H, d]."""
    v16 = np.asarray(v16, dtype=F16)
    return np.array([abs_percentile(v16[:, h, :], q) for h in range(v16.shape[1])], dtype=F32)


def sensitivity_order(s) -> list:
    """Layers by sensitivity, largest first; equal values keep layer order."""
    s = [float(x) for x in s]
    if any(math.isnan(x) or x < 0 for x in s):
        raise ValueError("sensitivities must be >= 0")
    return sorted(range(len(s)), key=lambda l: (-s[l], l))


def autok(s, frac: float) -> int:
    """Smallest k such that the k most sensitive layers hold >= frac of the total."""
    if not (0.0 <= frac <= 1.0):
        raise ValueError("frac must lie in [0, 1]")
    order = sensitivity_order(s)
    prefix = [0.0]
    for l in order:
        prefix.append(prefix[-1] + float(s[l]))
    target = frac * prefix[-1]
    return next(k for k, p in enumerate(prefix) if p >= target)


def allocate(s, k: int, low: int, high: int) -> list:
    """K bits per layer: the k most sensitive layers `high`, the rest `low`."""
    top = set(sensitivity_order(s)[:k])
    return [high if l in top else low for l in range(len(s))]


def choose(candidates, scores) -> int:
    """Index of the lowest score; equal scores go to the larger percentile."""
    return min(range(len(candidates)), key=lambda i: (float(scores[i]), -float(candidates[i])))


def v_perturbation(Q16, ks, vs, vb: int, vclip) -> float:
    """Value score: relative squared change of the attention output when V is
    quantized at vb bits with per-head thresholds vclip [Hkv] (K raw fp16).

    Q16 [B, Hq, d]; ks[s], vs[s] = [T_s, Hkv, d] fp16."""
    num = den = 0.0
    for s, q in enumerate(np.asarray(Q16)):
        k = ks[s].astype(F32)
        v = vs[s].astype(F32)
        if vb == 16:
            vh = v
        else:
            qq, sc = quant.quantize(vs[s], vb, axis=2, clip=vclip)
            vh = quant.dequantize(qq, sc, axis=2)
        o = attention.decode_attention(q, k, v)
        oh = attention.decode_attention(q, k, vh)
        num += float(((oh - o) ** 2).sum())
        den += float((o ** 2).sum())
    return num / den if den > 0 else 0.0


def calibration_data(w, l: int):
    """Layer l's calibration set: every sequence's prefill K/V [T_s, Hkv, d]
    and the step-0 queries [B, Hq, d] (the workload's seeded draws)."""
    ks, vs = [], []
    for s in range(w.batch):
        k, v = w.prefill_kv(l, [s], n_tok=w.prefill[s])
        ks.append(k[0].numpy())
        vs.append(v[0].numpy())
    Q = w.step_q(l, 0, 1)[:, 0].numpy()
    return ks, vs, Q


def calibrate(w, candidates, frac: float, low: int, high: int) -> dict:
    """The offline calibration over the workload's layers -> the artifact fields
    and every score (fp64): k_bits, v_bits, k_clip [L, Hkv, d], v_clip [L, Hkv],
    k_choice, v_choice (candidate indices), k_score, v_score [L, n_cand],
    sensitivity [L]."""
    if low not in canary.BITS:
        raise ValueError("low must be 2, 4 or 8 bits")
    bi = canary.BITS.index(low)
    L = w.num_layers
    out = {"k_clip": [], "v_clip": [], "k_choice": [], "v_choice": [], "k_score": [],
           "v_score": [], "sensitivity": []}
    for l in range(L):
        ks, vs, Q = calibration_data(w, l)
        K = np.concatenate(ks)
        V = np.concatenate(vs)
        kc = [k_thresholds(K, q) for q in candidates]
        vc = [v_thresholds(V, q) for q in candidates]
        wins = [k[-RING:].transpose(1, 0, 2) for k in ks]
        kscore = [canary.layer_delta(Q, wins, clip=c)[bi] for c in kc]
        vscore = [v_perturbation(Q, ks, vs, w.v_bits[l], c) for c in vc]
        i, j = choose(candidates, kscore), choose(candidates, vscore)
        out["k_clip"].append(kc[i])
        out["v_clip"].append(vc[j])
        out["k_choice"].append(i)
        out["v_choice"].append(j)
        out["k_score"].append(kscore)
        out["v_score"].append(vscore)
        out["sensitivity"].append(kscore[i])
    k = autok(out["sensitivity"], frac)
    out["n_protected"] = k
    out["k_bits"] = allocate(out["sensitivity"], k, low, high)
    out["v_bits"] = list(w.v_bits)
    out["k_clip"] = np.stack(out["k_clip"])
    out["v_clip"] = np.stack(out["v_clip"])
    return out

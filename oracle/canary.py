"""The EchoKV canary: KL between FP16 and quantized attention over the K_ref ring (oracle).

Follows "EchoKV: watching a language model decide its own precision",
section "Show the math — what the canary actually computes" (the KL
equation) and "Do we store the whole cache in FP16? — No." (the ring):

    delta_{l,b} = KL( softmax(Q K^T) || softmax(Q quant_b(K)^T) ),  b in {2, 4, 8}

summed over the key axis and averaged over all queries of the step.

Readings where the page leaves a step open:
  (i)   the logits carry the layer's attention scale sigma = 1/sqrt(d);
  (ii)  quant_b is the cache's own symmetric quantizer, per channel over
        consecutive 16-row groups of the window starting at the oldest row
        (the page calls its quantizer KIVI-style asymmetric; the workloads fix
        the symmetric one);
  (iii) the window is the newest min(count, 64) K's of the (layer, sequence,
        KV head), oldest first, including this step's K;
  (iv)  the queries are this step's Q for every query head of every sequence;
  (v)   log-probabilities come from log-softmax, so no 0 * log 0 appears.
Computed in fp64.
"""
from __future__ import annotations

import numpy as np

from . import quant

BITS = (2, 4, 8)
GROUP = 16
RING = 64


def window_dequant(w16: np.ndarray, b: int, clip=None, asym: bool = False) -> np.ndarray:
    """quant_b then dequant of a window [n, d] fp16, per channel over 16-row
    groups (clip: the head's per-channel thresholds [d], or None; asym: the
    KIVI-style asymmetric quantizer the page names for quant_b)."""
    w16 = np.asarray(w16, dtype=np.float16)
    n = w16.shape[0]
    out = np.zeros(w16.shape, dtype=np.float32)
    for g0 in range(0, n, GROUP):
        grp = w16[g0:g0 + GROUP]
        if asym:
            u, s, z = quant.quantize_asym(grp, b, axis=0)
            out[g0:g0 + GROUP] = quant.dequantize_asym(u, s, z, axis=0)
        else:
            q, s = quant.quantize(grp, b, axis=0, clip=clip)
            out[g0:g0 + GROUP] = quant.dequantize(q, s, axis=0)
    return out


def _log_softmax(z: np.ndarray) -> np.ndarray:
    m = z.max(axis=-1, keepdims=True)
    return z - m - np.log(np.exp(z - m).sum(axis=-1, keepdims=True))


def kl_per_query(q16: np.ndarray, w16: np.ndarray, b: int, scale: float | None = None,
                 clip=None, asym: bool = False) -> np.ndarray:
    """KL(p || p_hat_b) for each query row of q16 [G, d] against window w16 [n, d]."""
    q = np.asarray(q16).astype(np.float64)
    d = q.shape[-1]
    sigma = 1.0 / np.sqrt(d) if scale is None else float(scale)
    w = np.asarray(w16, dtype=np.float16).astype(np.float64)
    wq = window_dequant(w16, b, clip, asym).astype(np.float64)
    lp = _log_softmax(sigma * (q @ w.T))
    lph = _log_softmax(sigma * (q @ wq.T))
    return (np.exp(lp) * (lp - lph)).sum(axis=-1)


def layer_delta(Q16: np.ndarray, windows, scale: float | None = None, clip=None,
                asym: bool = False) -> np.ndarray:
    """delta[b] for one layer: Q16 [B, Hq, d], windows[s] = [Hkv, n_s, d] -> fp64 [3].

    clip: the layer's K thresholds [Hkv, d] (the cache's quantizer), or None.

    Query head h of sequence s reads KV head h // (Hq/Hkv) of sequence s.
    """
    Q16 = np.asarray(Q16)
    B, Hq, d = Q16.shape
    Hkv = windows[0].shape[0]
    G = Hq // Hkv
    tot = np.zeros(len(BITS), dtype=np.float64)
    for s in range(B):
        for g in range(Hkv):
            for i, b in enumerate(BITS):
                tot[i] += kl_per_query(Q16[s, g * G:(g + 1) * G], windows[s][g], b, scale,
                                       None if clip is None else clip[g], asym).sum()
    return tot / (B * Hq)

"""Single-token decode attention with GQA over dequantized K/V (oracle, fp64).

Definition: for query head h with KV head g = h // G (G = Hq / Hkv, the
contiguous grouping; "GQA head mapping" on the Behavior-Guided KV-Cache
Quantization page, "Storage savings, with a conditional speed trade-off"),

    o_h = sum_t softmax_t( sigma * q_h . khat_{g,t} ) vhat_{g,t},   sigma = 1/sqrt(d)

over every cached token t of the sequence ("every decoded token reads the
entire KV cache", KV-Kaizen page, "Background: The KV Cache Bottleneck").
khat/vhat are the stored values: dequantized codes for sealed K blocks and for
V, raw fp16 for the rows of a K block that is still open.

Computed in fp64 from the exact fp32 dequantized values; softmax subtracts
the max.  At 16 bits this is textbook attention (pinned against torch's
scaled_dot_product_attention); at lower bits its values are pinned only
through the quantizer ("parity unpinned" beyond the definition: the pages
print no worked example).
"""
from __future__ import annotations

import numpy as np


def decode_attention(q16: np.ndarray, khat: np.ndarray, vhat: np.ndarray,
                     scale: float | None = None) -> np.ndarray:
    """q16 [Hq, d] fp16; khat, vhat [T, Hkv, d] fp32 -> o [Hq, d] fp64."""
    q = np.asarray(q16).astype(np.float64)
    k = np.asarray(khat).astype(np.float64)
    v = np.asarray(vhat).astype(np.float64)
    Hq, d = q.shape
    T, Hkv, _ = k.shape
    if Hq % Hkv:
        raise ValueError("query heads must be a multiple of KV heads")
    G = Hq // Hkv
    sigma = 1.0 / np.sqrt(d) if scale is None else float(scale)
    o = np.zeros((Hq, d), dtype=np.float64)
    if T == 0:
        return o
    for h in range(Hq):
        g = h // G
        z = sigma * (k[:, g, :] @ q[h])
        z = z - z.max()
        p = np.exp(z)
        p = p / p.sum()
        o[h] = p @ v[:, g, :]
    return o

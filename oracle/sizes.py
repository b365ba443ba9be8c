"""Closed-form byte and bit accounting (oracle).

  * KV bytes per token = L * 2 * n_kv * d * bytes/element (KV-Kaizen page,
    "Background: The KV Cache Bottleneck": 192 KiB per token for Qwen2.5-14B).
  * K_ref ring = L * n_kv * 64 * d fp16, K only (EchoKV page, "Do we store the
    whole cache in FP16? — No.": about 10 MB for Llama-3.1-70B at 128K).
  * cache codes = L * 2 * n_kv * d * T * bits / 8 (EchoKV page, "What the
    controller costs you in memory": about 42 GB FP16 and 10 GB INT cache).
  * tau(L) = tau0 * sqrt(L / L0), tau0 = 0.022 at L0 = 4K (EchoKV page,
    "Show the math", the tau(L) scaling: 0.124 at 128K).
  * cost c(a) = (d + d_R) * b bits per token per layer, C0 = L * 2 n_kv d_h * 16
    (KV-Kaizen page, "Action Space and Cost Model").
  * bytes one decode step reads from a page of format (kb, vb): the whole page
    for sealed blocks (our layout, see `pages`).
"""
from __future__ import annotations

import math

from . import pages


def kv_bytes_per_token(L: int, n_kv: int, d: int, bytes_per_elem: float = 2) -> float:
    return L * 2 * n_kv * d * bytes_per_elem


def ring_bytes(L: int, n_kv: int, d: int, ring: int = 64) -> int:
    return L * n_kv * ring * d * 2


def cache_code_bytes(L: int, n_kv: int, d: int, T: int, bits: int) -> float:
    return L * 2 * n_kv * d * T * bits / 8


def tau_scaled(ctx: int, tau0: float = 0.022, ctx0: int = 4096) -> float:
    return tau0 * math.sqrt(ctx / ctx0)


def kaizen_cost(d: int, d_rope: int, b: int) -> int:
    return (d + d_rope) * b


def kaizen_c0(L: int, n_kv: int, d_h: int) -> int:
    return L * 2 * n_kv * d_h * 16


def page_read_bytes_per_token(kb: int, vb: int, d: int) -> float:
    """Algorithmic bytes per token per KV head read by attention from sealed pages."""
    return pages.page_bytes(kb, vb, d) / pages.BLOCK

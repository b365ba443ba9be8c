"""Byte layout of one cache page (oracle).

A page holds 16 token slots of one (layer, sequence, KV head).  Its format is
the pair (K bits, V bits); K bits are the layer's tier when the page was
allocated ("already-allocated blocks are never modified", EchoKV page, "What
happens to old blocks when a layer changes tier?"), V bits are the layer's
fixed V width.  K is quantized per channel over the page's 16 tokens and V per
token over the head's channels (Behavior-Guided KV-Cache Quantization page,
"K/V Role-Aware Low-Bit Quantization": Key per channel, Value per token).

Layout (our storage reading; the pages only say "packed low-bit storage"):

    K part  kb < 16 : codes [16][d*kb/8]  then scales [d]  fp16 (per channel)
            kb = 16 : raw fp16 [16][d]
    V part  vb < 16 : codes [16][d*vb/8]  then scales [16] fp16 (per token)
            vb = 16 : raw fp16 [16][d]
    page  = K part || V part            (little-endian fp16)

A cache built with the KIVI-style asymmetric quantizer stores unsigned codes u
and adds each group's fp16 zero point right after the scales: K zero points
[d] (same order as the K scales) after the K scales, V zero points [16] after
the V scales.  16-bit parts are unchanged.

The K scales of 2- and 4-bit pages are stored in "pair order": within each
group of n = 32/kb channels (the channels of one 32-bit code word), scale
position p holds channel p // 2 + (p % 2) * n / 2, i.e. 0, n/2, 1, n/2+1, ...
(4 bits: 0,4,1,5,2,6,3,7; 2 bits: 0,8,1,9,...,7,15).  8-bit pages keep the
natural channel order.
"""
from __future__ import annotations

import numpy as np

from . import quant

BLOCK = 16


def k_part_bytes(kb: int, d: int, asym: bool = False) -> int:
    return BLOCK * d * 2 if kb == 16 else BLOCK * d * kb // 8 + 2 * d * (2 if asym else 1)


def v_part_bytes(vb: int, d: int, asym: bool = False) -> int:
    return BLOCK * d * 2 if vb == 16 else BLOCK * d * vb // 8 + 2 * BLOCK * (2 if asym else 1)


def page_bytes(kb: int, vb: int, d: int, asym: bool = False) -> int:
    return k_part_bytes(kb, d, asym) + v_part_bytes(vb, d, asym)


def regions(kb: int, vb: int, d: int, asym: bool = False) -> dict:
    """name -> (offset, row_bytes, rows) of each region of the page."""
    r = {}
    if kb == 16:
        r["k_raw"] = (0, 2 * d, BLOCK)
    else:
        r["k_codes"] = (0, d * kb // 8, BLOCK)
        r["k_scales"] = (BLOCK * d * kb // 8, 2 * d, 1)
        if asym:
            r["k_zeros"] = (BLOCK * d * kb // 8 + 2 * d, 2 * d, 1)
    o = k_part_bytes(kb, d, asym)
    if vb == 16:
        r["v_raw"] = (o, 2 * d, BLOCK)
    else:
        r["v_codes"] = (o, d * vb // 8, BLOCK)
        r["v_scales"] = (o + BLOCK * d * vb // 8, 2, BLOCK)
        if asym:
            r["v_zeros"] = (o + BLOCK * d * vb // 8 + 2 * BLOCK, 2, BLOCK)
    return r


def scale_order(kb: int, d: int) -> np.ndarray:
    """Channel stored at each K-scale position of a kb-bit page."""
    if kb not in (2, 4):
        return np.arange(d)
    n = 32 // kb
    p = np.arange(d)
    return (p // n) * n + (p % n) // 2 + (p % 2) * (n // 2)


def sealed_k_bytes(kb: int, k16: np.ndarray, clip=None, asym: bool = False) -> dict:
    """Expected bytes of a full page's K part from its 16 raw fp16 rows [16, d]
    (clip: per-channel thresholds [d] or None; asym: the asymmetric quantizer)."""
    k16 = np.asarray(k16, dtype=np.float16)
    assert k16.shape[0] == BLOCK
    if kb == 16:
        return {"k_raw": k16.view(np.uint8).reshape(BLOCK, -1)}
    if asym:
        if clip is not None:
            raise ValueError("clipping thresholds apply to the symmetric quantizer only")
        u, s, z = quant.quantize_asym(k16, kb, axis=0)
        order = scale_order(kb, k16.shape[1])
        return {"k_codes": quant.pack_unsigned(u, kb),
                "k_scales": s[order].astype(np.float16).view(np.uint8)[None, :],
                "k_zeros": z[order].astype(np.float16).view(np.uint8)[None, :]}
    q, s = quant.quantize(k16, kb, axis=0, clip=clip)   # one group per channel
    s = s[scale_order(kb, k16.shape[1])]
    return {"k_codes": quant.pack(q, kb), "k_scales": s.astype(np.float16).view(np.uint8)[None, :]}


def v_rows_bytes(vb: int, v16: np.ndarray, clip=None, asym: bool = False) -> dict:
    """Expected bytes of V rows [n, d] (rows 0..n-1 of the page; clip: the
    head's threshold or None; asym: the asymmetric quantizer)."""
    v16 = np.asarray(v16, dtype=np.float16)
    if vb == 16:
        return {"v_raw": v16.view(np.uint8).reshape(v16.shape[0], -1)}
    if asym:
        if clip is not None:
            raise ValueError("clipping thresholds apply to the symmetric quantizer only")
        u, s, z = quant.quantize_asym(v16, vb, axis=1)
        return {"v_codes": quant.pack_unsigned(u, vb),
                "v_scales": s.astype(np.float16).view(np.uint8).reshape(-1, 2),
                "v_zeros": z.astype(np.float16).view(np.uint8).reshape(-1, 2)}
    q, s = quant.quantize(v16, vb, axis=1, clip=clip)   # one group per token
    return {"v_codes": quant.pack(q, vb),
            "v_scales": s.astype(np.float16).view(np.uint8).reshape(-1, 2)}


def extract(page: np.ndarray, kb: int, vb: int, d: int, name: str, rows: int | None = None,
            asym: bool = False):
    """Slice region `name` out of raw page bytes as [rows, row_bytes] uint8."""
    off, rb, n = regions(kb, vb, d, asym)[name]
    if rows is None:
        rows = n
    return np.asarray(page, dtype=np.uint8)[off:off + rb * n].reshape(n, rb)[:rows]

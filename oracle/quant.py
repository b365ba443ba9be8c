"""Symmetric uniform b-bit quantization and the packed code layout (oracle).

Definition followed (the workloads' quantizer, the reading of "symmetric
uniform quantization" on the KV-Kaizen page, "Three Non-Eviction Compression
Axes", item 3, and of "symmetric INT4" / INT4-RoleAlign on the
Behavior-Guided KV-Cache Quantization page, "K/V Role-Aware Low-Bit
Quantization"):

    qmax = 2**(b-1) - 1
    m    = min( max |x_i|, c )             over the group (exact on fp16 values)
    s    = fp16_rne( fp32(m) / fp32(qmax) ) the stored scale
    q_i  = clamp( rne( fp32(x_i) / fp32(s) ), -qmax, +qmax ),  q_i = 0 if s == 0
    xhat = fp32(q_i) * fp32(s)             (exact in fp32 for b <= 8)

c is the group's clipping threshold, +inf (no clipping) unless a frozen
calibration artifact sets one ("Behavior-Guided KV-Cache Quantization",
"Calibration protocol": the selected scales and clipping thresholds are frozen
and reused by the cache; reading: clipping the group at c before the absmax
makes its range min(absmax, c), and values beyond c take the end codes
+-qmax through the clamp).  With c = +inf the quantizer is the plain one.

All divisions are IEEE fp32 correctly rounded (numpy float32 arithmetic),
rne is round-half-to-even (numpy.rint), and the fp32 -> fp16 conversion is
numpy's round-to-nearest-even.

Stored code (our storage reading; the pages only say "packed low-bit
storage"): u = q + 2**(b-1) (offset binary), b bits per element, elements
packed along the channel axis least-significant-bits first: element c lives
in byte (c*b)//8 at bit (c*b) % 8.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
F16 = np.float16


def qmax(b: int) -> int:
    if b not in (2, 4, 8):
        raise ValueError(f"no integer quantizer for {b} bits")
    return (1 << (b - 1)) - 1


def quantize(x16: np.ndarray, b: int, axis: int, clip=None):
    """Quantize fp16 `x16` in groups along `axis` -> (q int16, s fp16 with `axis` removed).

    `clip` (fp32, broadcast against the groups: the shape of `x16` without
    `axis`, or a scalar) caps each group's absmax; None = no clipping."""
    x16 = np.asarray(x16)
    if x16.dtype != F16:
        raise TypeError("quantizer input must be fp16")
    x = x16.astype(F32)
    qm = F32(qmax(b))
    m = np.max(np.abs(x), axis=axis, keepdims=True)
    if clip is not None:
        c = np.asarray(clip, dtype=F32)
        if np.any(np.isnan(c)) or np.any(c <= 0):
            raise ValueError("clipping thresholds must be positive (+inf: none)")
        m = np.expand_dims(np.minimum(np.squeeze(m, axis=axis), c), axis)
    s32 = (m / qm).astype(F32)
    s16 = s32.astype(F16)
    sf = s16.astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (x / sf).astype(F32)
    q = np.clip(np.rint(r), -qm, qm)
    q = np.where(sf == 0, F32(0), q)
    return q.astype(np.int16), np.squeeze(s16, axis=axis)


def dequantize(q: np.ndarray, s16: np.ndarray, axis: int) -> np.ndarray:
    """xhat = fp32(q) * fp32(s), `s16` broadcast along `axis`."""
    s = np.expand_dims(np.asarray(s16, dtype=F16).astype(F32), axis)
    return (q.astype(F32) * s).astype(F32)


def levels(b: int) -> int:
    if b not in (2, 4, 8):
        raise ValueError(f"no integer quantizer for {b} bits")
    return (1 << b) - 1


def quantize_asym(x16: np.ndarray, b: int, axis: int):
    """KIVI-style asymmetric b-bit quantization of fp16 `x16` in groups along
    `axis` -> (u int16 in [0, 2^b - 1], s fp16, z fp16), `axis` removed.

    Follows "EchoKV: watching a language model decide its own precision",
    "Show the math" (quant_b is KIVI-style asymmetric per-group quantization,
    whose per-group scale is a function of the group's max and min, "Bidirectional
    adjustment"), and the page's per-token KIVI INT2/4/8 cache storage
    ("Upstreaming into vLLM").  Reading (the page gives no formula):

        lo, hi = min x_i, max x_i              (exact on fp16 values)
        s  = fp16_rne( fp32(fp32(hi - lo) / fp32(2^b - 1)) )   the stored scale
        z  = lo                                the stored zero point (fp16, exact)
        u_i = clamp( rne( fp32(fp32(x_i - z) / fp32(s)) ), 0, 2^b - 1 ),  u = 0 if s == 0
        xhat = fp32( fp32(u) * fp32(s) + fp32(z) )   (the product is exact)
    """
    x16 = np.asarray(x16)
    if x16.dtype != F16:
        raise TypeError("quantizer input must be fp16")
    x = x16.astype(F32)
    lv = F32(levels(b))
    lo = np.min(x, axis=axis, keepdims=True)
    hi = np.max(x, axis=axis, keepdims=True)
    s16 = ((hi - lo).astype(F32) / lv).astype(F32).astype(F16)
    sf = s16.astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = ((x - lo).astype(F32) / sf).astype(F32)
    u = np.clip(np.rint(r), F32(0), lv)
    u = np.where(sf == 0, F32(0), u)
    return (u.astype(np.int16), np.squeeze(s16, axis=axis),
            np.squeeze(lo.astype(F16), axis=axis))


def dequantize_asym(u: np.ndarray, s16: np.ndarray, z16: np.ndarray, axis: int) -> np.ndarray:
    """xhat = fp32(u) * fp32(s) + fp32(z), `s16` and `z16` broadcast along `axis`."""
    s = np.expand_dims(np.asarray(s16, dtype=F16).astype(F32), axis)
    z = np.expand_dims(np.asarray(z16, dtype=F16).astype(F32), axis)
    return ((u.astype(F32) * s).astype(F32) + z).astype(F32)


def pack_unsigned(u: np.ndarray, b: int) -> np.ndarray:
    """Pack unsigned codes u in [0, 2^b - 1] (stored as they are, LSB first)."""
    return pack(np.asarray(u, dtype=np.int64) - (1 << (b - 1)), b)


def pack(q: np.ndarray, b: int) -> np.ndarray:
    """Pack int codes along the last axis, offset binary, LSB first -> uint8."""
    q = np.asarray(q, dtype=np.int64)
    n = q.shape[-1]
    if (n * b) % 8:
        raise ValueError("row does not fill whole bytes")
    u = q + (1 << (b - 1))
    if np.any(u < 0) or np.any(u >= (1 << b)):
        raise ValueError("code out of range")
    out = np.zeros(q.shape[:-1] + (n * b // 8,), dtype=np.int64)
    for c in range(n):
        byte, bit = divmod(c * b, 8)
        out[..., byte] |= u[..., c] << bit
    return out.astype(np.uint8)


def unpack(packed: np.ndarray, b: int, n: int) -> np.ndarray:
    """Inverse of `pack`: uint8 rows -> int16 codes q."""
    p = np.asarray(packed, dtype=np.int64)
    q = np.zeros(p.shape[:-1] + (n,), dtype=np.int64)
    for c in range(n):
        byte, bit = divmod(c * b, 8)
        q[..., c] = ((p[..., byte] >> bit) & ((1 << b) - 1)) - (1 << (b - 1))
    return q.astype(np.int16)

"""Seeded, counter-based synthetic inputs (Q, K, V, outlier channels, lengths, bit draws).

This module is the ONE piece shared by the CUDA path's callers (tests, bench)
and the CPU oracle. It holds none of the method's arithmetic: no quantizer,
no attention, no KL, no controller. It only draws numbers.

Every element is a pure function of its coordinates, so any slice (one layer,
one sequence, one KV head, one token range) can be regenerated on the CPU
without materialising the rest, and the same call on a CUDA device gives the
same bits as on the CPU:

  * the hash is integer-only (32-bit arithmetic carried in int64 tensors, with
    every product split so that nothing overflows);
  * the N(0,1) draw is a table lookup: the top 16 bits of the hash index a
    table of the 65,536 standard-normal quantiles at (i + 1/2)/65536, rounded
    once to fp16 (tails reach +-4.33);
  * the only float step after the lookup is one fp32 multiply by a per-channel
    factor (outlier gain x layer gain) and one RNE rounding to fp16, both of
    which are correctly rounded on CPU and GPU alike.

The 32-bit mixer is "lowbias32" from Chris Wellons' hash-prospector
(x ^= x>>16; x *= 0x7feb352d; x ^= x>>15; x *= 0x846ca68b; x ^= x>>16),
written here from that published definition.
"""
from __future__ import annotations

import statistics
from functools import lru_cache

import torch

_M32 = 0xFFFFFFFF

# tensor ids used as hash coordinates
T_Q, T_K, T_V, T_OUTLIER, T_LEN, T_BITS = 1, 2, 3, 4, 5, 6


def _mul32(x: torch.Tensor, m: int) -> torch.Tensor:
    """(x * m) mod 2**32 for x in [0, 2**32), without int64 overflow."""
    lo, hi = m & 0xFFFF, (m >> 16) & 0xFFFF
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & _M32


def mix32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _mix32_int(x: int) -> int:
    x &= _M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & _M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & _M32
    x ^= x >> 16
    return x


def key(*coords: int) -> int:
    """Fold scalar coordinates into one 32-bit key (host-side, exact)."""
    h = 0x9E3779B9
    for c in coords:
        h = _mix32_int(h ^ (int(c) & _M32))
        h = _mix32_int(h + 0x6A09E667)
    return h


def hash_counter(k, counter: torch.Tensor) -> torch.Tensor:
    """Two mixing rounds of (key, counter); counter must lie in [0, 2**32).

    `k` is a host int or an int64 tensor of keys that broadcasts against
    `counter` (one key per sequence, for batched draws).
    """
    if isinstance(k, torch.Tensor):
        k2 = mix32(k ^ 0x85EBCA6B)
    else:
        k2 = _mix32_int(k ^ 0x85EBCA6B)
    return mix32(mix32(counter ^ k) ^ k2)


@lru_cache(maxsize=None)
def _normal_table_cpu() -> torch.Tensor:
    nd = statistics.NormalDist()
    vals = [nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)]
    return torch.tensor(vals, dtype=torch.float64).to(torch.float16)


_TABLES: dict = {}


def normal_table(device) -> torch.Tensor:
    device = torch.device(device)
    t = _TABLES.get(device)
    if t is None:
        t = _normal_table_cpu().to(device)
        _TABLES[device] = t
    return t


def normal16(k: int, counter: torch.Tensor) -> torch.Tensor:
    """fp16 N(0,1) draws, one per counter value."""
    h = hash_counter(k, counter)
    return normal_table(counter.device)[(h >> 16)]


def uniform_int(k: int, counter: torch.Tensor, lo: int, hi: int) -> torch.Tensor:
    """Integers uniform in [lo, hi] (inclusive); modulo bias < 2**-19 for spans < 8192."""
    h = hash_counter(k, counter)
    return lo + (h % (hi - lo + 1))


# ---------------------------------------------------------------------------
# Workload-level draws.  `cfg` is a small integer naming the workload (it keys
# the hash so that two workloads never share draws).
# ---------------------------------------------------------------------------

def outlier_channels(seed: int, cfg: int, layer: int, head: int, d: int, n_out: int,
                     fixed: tuple | None = None) -> list[int]:
    """Channels of one (layer, kv-head) whose K values get the outlier gain."""
    if fixed is not None:
        return sorted(int(c) for c in fixed)
    if n_out <= 0:
        return []
    ch = torch.arange(d, dtype=torch.int64)
    h = hash_counter(key(seed, cfg, T_OUTLIER, layer, head), ch)
    order = torch.argsort(h * d + ch)  # ties impossible: (h, ch) unique
    return sorted(int(c) for c in order[:n_out].tolist())


def k_gain(seed: int, cfg: int, layer: int, n_kv: int, d: int, n_out: int, out_gain: float,
           layer_slope: float, fixed: tuple | None = None) -> torch.Tensor:
    """Per (kv-head, channel) fp32 multiplier for K: outlier gain x (1 + slope*layer)."""
    g = torch.ones(n_kv, d, dtype=torch.float64)
    for h in range(n_kv):
        for c in outlier_channels(seed, cfg, layer, h, d, n_out, fixed):
            g[h, c] = out_gain
    g = g * (1.0 + layer_slope * layer)
    return g.to(torch.float32)


def draw16(seed: int, cfg: int, tensor: int, layer: int, seqs, tok0, n_tok: int,
           n_heads: int, d: int, gain: torch.Tensor | None = None, device="cpu") -> torch.Tensor:
    """fp16 [len(seqs), n_tok, n_heads, d] draws for one layer.

    Row s covers tokens tok0[s] .. tok0[s]+n_tok-1 of sequence seqs[s].  Element
    (s, t, h, c) is keyed by key(seed, cfg, tensor, layer, seqs[s]) and counter
    ((tok0[s]+t)*n_heads + h)*d + c, so any token range of any sequence
    regenerates identically, alone or batched.  `gain` ([n_heads, d] fp32)
    multiplies the N(0,1) draw in fp32 before the single RNE rounding to fp16.
    """
    seqs = [int(x) for x in seqs]
    tok0 = [int(x) for x in tok0]
    if len(tok0) != len(seqs):
        raise ValueError("one tok0 per sequence")
    B = len(seqs)
    if B == 0 or n_tok == 0:
        return torch.empty(B, n_tok, n_heads, d, dtype=torch.float16, device=device)
    if (max(tok0) + n_tok) * n_heads * d > (1 << 32):
        raise ValueError("token range exceeds the 32-bit counter space")
    keys = torch.tensor([key(seed, cfg, tensor, layer, s) for s in seqs],
                        dtype=torch.int64, device=device).view(B, 1)
    offs = torch.tensor(tok0, dtype=torch.int64, device=device).view(B, 1) * (n_heads * d)
    counter = torch.arange(n_tok * n_heads * d, dtype=torch.int64, device=device).view(1, -1) + offs
    h = hash_counter(keys, counter)
    z = normal_table(device)[h >> 16].view(B, n_tok, n_heads, d)
    if gain is None:
        return z
    return (z.to(torch.float32) * gain.to(device)).to(torch.float16)


def seq_lengths(seed: int, cfg: int, n: int, lo: int, hi: int) -> list[int]:
    c = torch.arange(n, dtype=torch.int64)
    return [int(v) for v in uniform_int(key(seed, cfg, T_LEN), c, lo, hi).tolist()]


def shuffled(seed: int, cfg: int, items: list) -> list:
    """Seeded permutation of `items` (sort by hash of position)."""
    c = torch.arange(len(items), dtype=torch.int64)
    h = hash_counter(key(seed, cfg, T_BITS), c)
    order = torch.argsort(h * len(items) + c).tolist()
    return [items[i] for i in order]

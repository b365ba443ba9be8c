"""Stateful reference of the decode loop: append, attention, canary, tiers (oracle).

Step order per decode step t, per layer l (readings of "EchoKV: watching a
language model decide its own precision", section "How EchoKV works", where
the step's K is written into K_ref "before being quantized into the paged
cache", and "What happens to old blocks when a layer changes tier?"):

  1. the new K enters the ring, then K and V enter the cache;
  2. attention reads all cached tokens, the new one included;
  3. on a firing step (t % period == 0) the canary measures delta_l.
After all layers of a firing step the controller updates every layer's EMA
and tier; the new tier governs pages allocated from step t+1 on.

Cache bookkeeping (readings; the pages are silent on the open block):
  * a page is allocated when a block's first token arrives; its K bits are
    the layer's tier at that moment (admit-time bits) and never change;
  * V is quantized per token as it arrives;
  * K rows stay raw fp16 while the block is open and are quantized per
    channel when the 16th token arrives (the block is "sealed"); attention
    reads open rows as fp16.

The state keeps the raw fp16 K/V of every token and derives codes on demand
from the definitions in `quant`; nothing is cached that could drift.
"""
from __future__ import annotations

import numpy as np

from . import attention, canary, controller, pages, quant

BLOCK = 16
RING = 64


class SeqState:
    """Cache of one (layer, sequence) restricted to a list of KV heads.

    Raw fp16 K/V of every token are kept in arrays that grow by doubling.
    Dequantized values of sealed K blocks and of V rows are computed once
    from the raw rows and kept (both are pure functions of rows that never
    change once written).
    """

    def __init__(self, n_heads: int, d: int, vbits: int, kclip=None, vclip=None,
                 asym: bool = False):
        self.H, self.d = n_heads, d
        self.asym = asym           # KIVI-style asymmetric quantizer for K and V
        self.kclip = kclip         # [H, d] fp32 K thresholds or None
        self.vclip = vclip         # [H] fp32 V thresholds or None
        self._k = np.zeros((0, n_heads, d), dtype=np.float16)
        self._v = np.zeros((0, n_heads, d), dtype=np.float16)
        self._kh = np.zeros((0, n_heads, d), dtype=np.float32)   # sealed K, dequantized
        self._vh = np.zeros((0, n_heads, d), dtype=np.float32)   # V, dequantized
        self.n = 0
        self._sealed_upto = 0      # blocks [0, _sealed_upto) hold dequantized K in _kh
        self._vh_upto = 0          # tokens [0, _vh_upto) hold dequantized V in _vh
        self.kbits: list = []      # admit-time K bits per block
        self.vbits = vbits

    @property
    def T(self) -> int:
        return self.n

    @property
    def k(self) -> np.ndarray:
        return self._k[:self.n]

    @property
    def v(self) -> np.ndarray:
        return self._v[:self.n]

    def _grow(self, need: int):
        cap = self._k.shape[0]
        if need <= cap:
            return
        cap = max(need, 2 * cap, 64)
        for name, dt in (("_k", np.float16), ("_v", np.float16), ("_kh", np.float32),
                         ("_vh", np.float32)):
            old = getattr(self, name)
            new = np.zeros((cap, self.H, self.d), dtype=dt)
            new[:old.shape[0]] = old
            setattr(self, name, new)

    def append(self, k16: np.ndarray, v16: np.ndarray, tier: int):
        k16 = np.asarray(k16, dtype=np.float16)
        v16 = np.asarray(v16, dtype=np.float16)
        n = k16.shape[0]
        for p in range(self.n, self.n + n):
            if p % BLOCK == 0:
                self.kbits.append(int(tier))
        self._grow(self.n + n)
        self._k[self.n:self.n + n] = k16
        self._v[self.n:self.n + n] = v16
        self.n += n

    def khat(self) -> np.ndarray:
        """Stored K values [T, H, d] fp32: sealed blocks dequantized, open rows raw."""
        T = self.n
        full = T // BLOCK
        for j in range(self._sealed_upto, full):
            lo, hi = j * BLOCK, (j + 1) * BLOCK
            kb = self.kbits[j]
            if kb == 16:
                self._kh[lo:hi] = self._k[lo:hi].astype(np.float32)
            elif self.asym:
                u, s, z = quant.quantize_asym(self._k[lo:hi], kb, axis=0)
                self._kh[lo:hi] = quant.dequantize_asym(u, s, z, axis=0)
            else:
                q, s = quant.quantize(self._k[lo:hi], kb, axis=0, clip=self.kclip)
                self._kh[lo:hi] = quant.dequantize(q, s, axis=0)
        self._sealed_upto = max(self._sealed_upto, full)
        out = self._kh[:T].copy()
        out[full * BLOCK:T] = self._k[full * BLOCK:T].astype(np.float32)
        return out

    def vhat(self) -> np.ndarray:
        T = self.n
        lo = self._vh_upto
        if T > lo:
            if self.vbits == 16:
                self._vh[lo:T] = self._v[lo:T].astype(np.float32)
            elif self.asym:
                u, s, z = quant.quantize_asym(self._v[lo:T], self.vbits, axis=2)
                self._vh[lo:T] = quant.dequantize_asym(u, s, z, axis=2)
            else:
                q, s = quant.quantize(self._v[lo:T], self.vbits, axis=2, clip=self.vclip)
                self._vh[lo:T] = quant.dequantize(q, s, axis=2)
            self._vh_upto = T
        return self._vh[:T]

    def window(self) -> np.ndarray:
        """The K_ref ring contents [n, H, d], oldest first (n = min(T, 64))."""
        return self.k[max(0, self.n - RING):self.n]

    def page_expect(self, j: int, h: int) -> dict:
        """Expected bytes of the defined regions of page j, head index h."""
        kb = self.kbits[j]
        lo = j * BLOCK
        hi = min(lo + BLOCK, self.n)
        exp = {}
        if hi - lo == BLOCK:
            exp.update(pages.sealed_k_bytes(kb, self._k[lo:hi, h],
                                            None if self.kclip is None else self.kclip[h],
                                            self.asym))
        exp.update(pages.v_rows_bytes(self.vbits, self._v[lo:hi, h],
                                      None if self.vclip is None else self.vclip[h], self.asym))
        return exp


def layer_windows(w, layer: int, step: int, device="cpu") -> list:
    """Ring windows of every sequence after step `step`'s append: [Hkv, n_s, d] each.

    Regenerated from the seeded draws: the newest n_s = min(T_s, 64) K's,
    oldest first.
    """
    wins = []
    for s in range(w.batch):
        T = w.prefill[s] + step + 1
        n_s = min(RING, T)
        k, _ = w.prefill_kv(layer, [s], device=device, tok0=[T - n_s], n_tok=n_s)
        wins.append(k[0].permute(1, 0, 2).cpu().numpy())
    return wins


class Trace:
    """Controller history: tiers in effect at each step's append, deltas, EMAs."""

    def __init__(self):
        self.tiers = []       # tiers[t] = tier vector used by step t's appends
        self.delta = {}       # step -> fp64 [L, 3]
        self.ema = {}         # step -> fp32 [L, 3] after the update
        self.after = {}       # step -> tiers after the update


def controller_trace(w, n_steps: int, device="cpu", clips=None) -> Trace:
    """Run the canary + controller over all layers for steps 0..n_steps-1.

    clips: {layer: (K thresholds [Hkv, d], V thresholds [Hkv])} for layers
    with a frozen clipping artifact (the canary measures the cache's own
    quantizer), or None."""
    ctl = controller.Controller(w.k_bits_init, w.alpha, w.tau)
    tr = Trace()
    for t in range(n_steps):
        tr.tiers.append(list(ctl.tiers))
        if not w.fires(t):
            continue
        deltas = np.zeros((w.num_layers, 3), dtype=np.float64)
        for l in range(w.num_layers):
            Q = w.step_q(l, t, 1, device=device)[:, 0].cpu().numpy()
            kc = None if not clips or l not in clips else clips[l][0]
            deltas[l] = canary.layer_delta(Q, layer_windows(w, l, t, device), clip=kc,
                                           asym=getattr(w, "asym", False))
        tr.delta[t] = deltas
        ctl.update(deltas.astype(np.float32))
        tr.ema[t] = np.array(ctl.ema, dtype=np.float32)
        tr.after[t] = list(ctl.tiers)
    tr.tiers.append(list(ctl.tiers))
    return tr


class ReferenceRun:
    """Attention and page contents for chosen layers, sequences and KV heads.

    Tiers come from a `Trace` (the controller over all layers); K/V/Q are the
    workload's seeded draws for the chosen coordinates only.
    """

    def __init__(self, w, trace: Trace, layers=None, seqs=None, heads=None, device="cpu",
                 clips=None):
        self.w = w
        self.trace = trace
        self.layers = list(range(w.num_layers)) if layers is None else list(layers)
        self.seqs = list(range(w.batch)) if seqs is None else list(seqs)
        self.heads = list(range(w.num_kv_heads)) if heads is None else list(heads)
        self.device = device
        clips = clips or {}
        sel = lambda l, i: (None if l not in clips or clips[l][i] is None
                            else np.asarray(clips[l][i], dtype=np.float32)[self.heads])
        self.state = {(l, s): SeqState(len(self.heads), w.head_dim, w.v_bits[l],
                                       sel(l, 0), sel(l, 1), getattr(w, "asym", False))
                      for l in self.layers for s in self.seqs}
        self.steps_done = 0

    def prefill(self):
        w = self.w
        for l in self.layers:
            for s in self.seqs:
                k, v = w.prefill_kv(l, [s], device=self.device, n_tok=w.prefill[s])
                k = k[0][:, self.heads].cpu().numpy()
                v = v[0][:, self.heads].cpu().numpy()
                self.state[(l, s)].append(k, v, w.k_bits_init[l])

    def q_heads(self) -> list:
        G = self.w.group
        return [g * G + i for g in self.heads for i in range(G)]

    def advance(self):
        """Append decode step t's K/V for the chosen coordinates (no attention)."""
        w, t = self.w, self.steps_done
        tiers = self.trace.tiers[t]
        for l in self.layers:
            k, v = w.step_kv(l, t, 1, seqs=self.seqs, device=self.device)
            for i, s in enumerate(self.seqs):
                self.state[(l, s)].append(k[i][:, self.heads].cpu().numpy(),
                                          v[i][:, self.heads].cpu().numpy(), tiers[l])
        self.steps_done += 1

    def attend(self, l: int, s: int) -> np.ndarray:
        """Attention of the last appended step for (l, s): o [len(heads)*G, d] fp64."""
        t = self.steps_done - 1
        q = self.w.step_q(l, t, 1, seqs=[s], device=self.device)[0, 0][self.q_heads()]
        st = self.state[(l, s)]
        return attention.decode_attention(q.cpu().numpy(), st.khat(), st.vhat())

    def step(self) -> dict:
        """Append step t's K/V and return {(l, s): o [len(heads)*G, d] fp64}."""
        self.advance()
        return {(l, s): self.attend(l, s) for l in self.layers for s in self.seqs}

"""The five synthetic decode workloads and their seeded inputs.

Shapes follow the models the pages quote (Llama-3.1-8B/70B, Qwen2.5-14B):
layers, query heads, KV heads and head_dim only; no weights.  Q, K and V are
fp16 draws from `synth` (N(0,1), K outlier channels scaled, optional
layer-dependent K gain).  Decode-step inputs are fresh draws: with no model,
outputs do not feed back.

Token indexing: a sequence's prefill tokens are 0 .. T0-1; decode step i
appends token T0+i.  The query of decode step i is drawn with token index i.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import torch

from . import synth

BITS = (2, 4, 8, 16)
CANARY_BITS = (2, 4, 8)
BLOCK = 16   # tokens per page block
RING = 64    # K_ref ring length


@dataclass
class Workload:
    name: str
    cfg: int                     # hash namespace of the draws
    num_layers: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    prefill: list                # T0 per sequence
    steps: int
    k_bits_init: list            # per layer
    v_bits: list                 # per layer
    canary_period: int = 0       # 0: no canary; else fire when step % period == 0
    alpha: float = 0.25
    tau: float = 0.05
    outlier_frac: float = 0.0
    outlier_gain: float = 1.0
    outlier_fixed: tuple | None = None
    layer_slope: float = 0.0
    seed: int = 0
    asym: bool = False           # KIVI-style asymmetric quantizer (K, V and canary)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def n_outliers(self) -> int:
        if self.outlier_fixed is not None:
            return len(self.outlier_fixed)
        if self.outlier_frac <= 0:
            return 0
        return max(1, int(round(self.outlier_frac * self.head_dim)))

    @property
    def max_seq_len(self) -> int:
        return max(self.prefill) + self.steps

    def fires(self, step: int) -> bool:
        return self.canary_period > 0 and step % self.canary_period == 0

    def k_gain(self, layer: int) -> torch.Tensor:
        return synth.k_gain(self.seed, self.cfg, layer, self.num_kv_heads, self.head_dim,
                            self.n_outliers, self.outlier_gain, self.layer_slope,
                            self.outlier_fixed)

    # ---- inputs -------------------------------------------------------
    def prefill_kv(self, layer: int, seqs, device="cpu", tok0=None, n_tok=None):
        """K, V fp16 [len(seqs), n, Hkv, d] for prefill tokens (all seqs padded to n)."""
        seqs = list(seqs)
        if tok0 is None:
            tok0 = [0] * len(seqs)
        if n_tok is None:
            n_tok = max(self.prefill[s] for s in seqs)
        g = self.k_gain(layer)
        k = synth.draw16(self.seed, self.cfg, synth.T_K, layer, seqs, tok0, n_tok,
                         self.num_kv_heads, self.head_dim, gain=g, device=device)
        v = synth.draw16(self.seed, self.cfg, synth.T_V, layer, seqs, tok0, n_tok,
                         self.num_kv_heads, self.head_dim, device=device)
        return k, v

    def step_kv(self, layer: int, step0: int, n_steps: int, seqs=None, device="cpu"):
        """K, V fp16 [B, n_steps, Hkv, d] appended at decode steps step0 ..."""
        seqs = list(range(self.batch)) if seqs is None else list(seqs)
        tok0 = [self.prefill[s] + step0 for s in seqs]
        g = self.k_gain(layer)
        k = synth.draw16(self.seed, self.cfg, synth.T_K, layer, seqs, tok0, n_steps,
                         self.num_kv_heads, self.head_dim, gain=g, device=device)
        v = synth.draw16(self.seed, self.cfg, synth.T_V, layer, seqs, tok0, n_steps,
                         self.num_kv_heads, self.head_dim, device=device)
        return k, v

    def step_q(self, layer: int, step0: int, n_steps: int, seqs=None, device="cpu"):
        """Q fp16 [B, n_steps, Hq, d] of decode steps step0 ..."""
        seqs = list(range(self.batch)) if seqs is None else list(seqs)
        return synth.draw16(self.seed, self.cfg, synth.T_Q, layer, seqs, [step0] * len(seqs),
                            n_steps, self.num_q_heads, self.head_dim, device=device)

    # ---- sizing -------------------------------------------------------
    def pool_pages(self) -> dict:
        """Upper bound on pages needed per (k_bits, v_bits) format."""
        need: dict = {}
        P = BLOCK
        for l in range(self.num_layers):
            vb = self.v_bits[l]
            pre = sum(math.ceil(t / P) for t in self.prefill) * self.num_kv_heads
            dec = sum(math.ceil((t + self.steps) / P) - math.ceil(t / P)
                      for t in self.prefill) * self.num_kv_heads
            kb0 = self.k_bits_init[l]
            need[(kb0, vb)] = need.get((kb0, vb), 0) + pre
            tiers = CANARY_BITS if self.canary_period > 0 else (kb0,)
            for kb in set(tiers) | {kb0}:
                need[(kb, vb)] = need.get((kb, vb), 0) + dec
        return need

    def scaled(self, **kw) -> "Workload":
        """A smaller case with the same draws per coordinate (for oracle-sized parity)."""
        w = dataclasses.replace(self, **kw)
        L = w.num_layers
        if len(w.k_bits_init) != L:
            w.k_bits_init = list(self.k_bits_init[:L])
        if len(w.v_bits) != L:
            w.v_bits = list(self.v_bits[:L])
        if len(w.prefill) != w.batch:
            w.prefill = list(self.prefill[:w.batch])
        return w


def tiny() -> Workload:
    """2 layers, batch 1, 4 q / 2 kv heads, d=64, 256 cached + 8 steps, canary every step."""
    return Workload("tiny", 1, 2, 1, 4, 2, 64, [256], 8, [4, 8], [8, 8],
                    canary_period=1, alpha=0.25, tau=0.05, outlier_fixed=(3, 17),
                    outlier_gain=10.0)


def llama8b_layer(bits: int) -> Workload:
    """One Llama-3.1-8B-shaped layer, batch 8, 4K context, uniform K=V bits, 64 steps."""
    return Workload(f"llama8b_layer_b{bits}", 2, 1, 8, 32, 8, 128, [4096] * 8, 64,
                    [bits], [bits], outlier_frac=0.02, outlier_gain=8.0)


def qwen14b_32k() -> Workload:
    """Qwen2.5-14B-shaped 48 layers, batch 1, 40 q / 8 kv heads, 32K, mixed K 2/4/8, V4."""
    kb = synth.shuffled(0, 3, [2] * 12 + [4] * 24 + [8] * 12)
    return Workload("qwen14b_32k", 3, 48, 1, 40, 8, 128, [32768], 128, kb, [4] * 48,
                    outlier_frac=0.01, outlier_gain=10.0)


def llama70b_128k() -> Workload:
    """Llama-3.1-70B-shaped 80 layers, batch 1, 64 q / 8 kv, 128K, canary every 64 steps."""
    return Workload("llama70b_128k", 4, 80, 1, 64, 8, 128, [131072], 512, [4] * 80, [4] * 80,
                    canary_period=64, alpha=0.25, tau=0.05, outlier_frac=0.01,
                    outlier_gain=10.0, layer_slope=0.05)


def llama8b_batch32() -> Workload:
    """Llama-3.1-8B-shaped 32 layers, batch 32, ragged 1K-8K, canary every 64, tau 0.03."""
    lens = synth.seq_lengths(0, 5, 32, 1024, 8192)
    return Workload("llama8b_batch32", 5, 32, 32, 32, 8, 128, lens, 256, [4] * 32, [4] * 32,
                    canary_period=64, alpha=0.25, tau=0.03, outlier_frac=0.01,
                    outlier_gain=10.0)


def all_workloads() -> list:
    return [tiny()] + [llama8b_layer(b) for b in BITS] + [qwen14b_32k(), llama70b_128k(),
                                                          llama8b_batch32()]


def by_name(name: str) -> Workload:
    for w in all_workloads():
        if w.name == name:
            return w
    raise KeyError(name)

"""Shared GPU-vs-oracle harness: run a workload through the C ABI and compare
every output the oracle can produce with it.

Tolerances (the targets the decode path is held to):
  * packed codes, fp16 scale bits, page formats and tiers: bit-exact;
  * attention output: |o_gpu - o_ref| <= 2e-3 + 1e-2 |o_ref| elementwise
    (o_ref in fp64, o_gpu rounded to fp16 from fp32 accumulation);
  * canary readings delta: |delta_gpu - delta_ref| <= 1e-4 (fp32 vs fp64).
A tier that differs from the oracle's is accepted only when the oracle's EMA
of a deciding bit-width lies within 1e-4 of tau (the reading's own
tolerance); the GPU is then set to the oracle's tiers so later pages stay
comparable.  Any other difference fails.
"""
from __future__ import annotations

import numpy as np
import torch

from mixed_precision_quantized_gb300 import ekv, runner, workloads
from oracle import decoder, pages

ATOL, RTOL = 2e-3, 1e-2
KL_TOL = 1e-4
BITS3 = (2, 4, 8)


def check_attn(o_gpu: torch.Tensor, o_ref: np.ndarray, what: str):
    g = o_gpu.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - o_ref)
    bound = ATOL + RTOL * np.abs(o_ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance, "
                           f"max abs err {err.max():.3e}")
    return float(err.max())


def tier_flip_is_ambiguous(ema_ref, tau, t_gpu, t_ref) -> bool:
    """A pick may differ only if an EMA it compared lies within the reading tolerance of tau."""
    top = min(max(t_gpu, t_ref), 8)
    return any(abs(float(ema_ref[i]) - tau) <= KL_TOL for i, b in enumerate(BITS3) if b <= top)


def check_pages(cache: ekv.Cache, ref: decoder.ReferenceRun, l: int, s: int, heads=None):
    """Bit-exact comparison of every defined byte of every page of (l, s)."""
    w = ref.w
    st = ref.state[(l, s)]
    heads = ref.heads if heads is None else heads
    nb = (st.T + 15) // 16
    for hi, h in enumerate(ref.heads):
        if h not in heads:
            continue
        bt = cache.block_table(l, s, h)
        assert len(bt) == nb
        raw = cache.read_pages(l, s, h, 0, nb).cpu().numpy()
        for j in range(nb):
            e = bt[j]
            assert e != -1, f"no page for block {j}"
            fmt = (e >> 28) & 15
            kb, vb = 2 << (fmt >> 2), 2 << (fmt & 3)
            assert kb == st.kbits[j], f"layer {l} seq {s} block {j}: page K bits {kb} != {st.kbits[j]}"
            assert vb == w.v_bits[l]
            exp = st.page_expect(j, hi)
            rows = min(16, st.T - 16 * j)
            for name, want in exp.items():
                got = pages.extract(raw[j], kb, vb, w.head_dim, name,
                                    rows=want.shape[0], asym=getattr(w, "asym", False))
                assert np.array_equal(got, want), (
                    f"layer {l} seq {s} head {h} block {j} ({kb},{vb}) region {name} "
                    f"rows {rows}: {np.argwhere(got != want)[:5].tolist()}")


class Run:
    """A workload on the GPU next to its oracle."""

    def __init__(self, w: workloads.Workload, steps: int, layers=None, seqs=None, heads=None,
                 gen_device="cuda", trace=None, pool_pages=None, fused=False, clips=None,
                 max_seq_len=None):
        """clips: {layer: (K thresholds [Hkv, d], V thresholds [Hkv])} loaded into
        the cache before the prefill and given to the oracle.  max_seq_len: the
        cache's capacity per sequence (default the workload's need)."""
        self.w, self.steps, self.fused = w, steps, fused
        if pool_pages is None and max_seq_len is None:
            self.cache = ekv.cache_for(w)
        else:
            self.cache = ekv.Cache(w.num_layers, w.batch, w.num_q_heads, w.num_kv_heads,
                                   w.head_dim, max_seq_len or w.max_seq_len,
                                   pool_pages or w.pool_pages(), w.k_bits_init,
                                   w.v_bits, alpha=w.alpha, tau=w.tau,
                                   asym=getattr(w, "asym", False))
        for l, (kc, vc) in (clips or {}).items():
            self.cache.set_clip(l, kc, vc)
        self.slots = torch.arange(w.batch, dtype=torch.int32, device="cuda")
        runner.prefill(self.cache, w, self.slots)
        self.cache.sync()
        self.trace = trace if trace is not None else decoder.controller_trace(
            w, steps, device=gen_device, clips=clips)
        self.ref = decoder.ReferenceRun(w, self.trace, layers, seqs, heads, device=gen_device,
                                        clips=clips)
        self.ref.prefill()
        self.inp = runner.Inputs(w, 0, steps)
        self.out = [torch.empty(w.batch, w.num_q_heads, w.head_dim, dtype=torch.float16,
                                device="cuda") for _ in range(w.num_layers)]
        self.t = 0
        self.max_err = 0.0
        self.flips = []

    def step(self, check_attn_now: bool = True):
        w, t = self.w, self.t
        fires = w.fires(t)
        runner.decode_step(self.cache, w, self.slots, self.inp, t, self.out, fires,
                           fused=self.fused)
        self.cache.sync()
        self.ref.advance()
        if check_attn_now:
            qh = self.ref.q_heads()
            for l in self.ref.layers:
                for s in self.ref.seqs:
                    o_ref = self.ref.attend(l, s)
                    e = check_attn(self.out[l][s][qh], o_ref, f"step {t} layer {l} seq {s}")
                    self.max_err = max(self.max_err, e)
        if fires:
            st = self.cache.state()
            dref = self.trace.delta[t]
            dgpu = np.array(st["delta"], dtype=np.float64)
            assert np.all(np.abs(dgpu - dref) <= KL_TOL), (
                f"step {t}: canary readings differ by {np.abs(dgpu - dref).max():.3e}")
            want = self.trace.after[t]
            if st["tiers"] != want:
                for l, (a, b) in enumerate(zip(st["tiers"], want)):
                    if a != b:
                        assert tier_flip_is_ambiguous(self.trace.ema[t][l], w.tau, a, b), (
                            f"step {t} layer {l}: tier {a} != oracle {b}, EMA "
                            f"{self.trace.ema[t][l].tolist()} tau {w.tau}")
                        self.flips.append((t, l, a, b))
                self.cache.set_tiers(want)
        self.t += 1

    def check_all_pages(self):
        for l in self.ref.layers:
            for s in self.ref.seqs:
                check_pages(self.cache, self.ref, l, s)

    def close(self):
        self.cache.close()

"""Issue the decode path of a workload through the C ABI.

One decode step is, per layer l: append the step's K/V (ring write, V
quantization, K staging or seal, page admission at the layer's tier), decode
attention over the whole cache, and on a firing step the canary; after the
last layer of a firing step, the controller updates every layer's EMA and tier.
"""
from __future__ import annotations

import torch

from . import ekv, workloads


class Inputs:
    """Device-resident per-step inputs of a workload (Q, new K, new V per layer)."""

    def __init__(self, w: workloads.Workload, step0: int, n_steps: int, device="cuda"):
        self.q, self.k, self.v = [], [], []
        for l in range(w.num_layers):
            k, v = w.step_kv(l, step0, n_steps, device=device)     # [B, n, Hkv, d]
            q = w.step_q(l, step0, n_steps, device=device)         # [B, n, Hq, d]
            self.k.append(k.transpose(0, 1).contiguous())          # [n, B, Hkv, d]
            self.v.append(v.transpose(0, 1).contiguous())
            self.q.append(q.transpose(0, 1).contiguous())          # [n, B, Hq, d]
        self.step0, self.n = step0, n_steps

    def layer(self, l: int, i: int):
        """(q [B,Hq,d], k [B,1,Hkv,d], v [B,1,Hkv,d]) of local step i."""
        return self.q[l][i], self.k[l][i].unsqueeze(1), self.v[l][i].unsqueeze(1)


def prefill(cache: ekv.Cache, w: workloads.Workload, slots: torch.Tensor, device="cuda",
            chunk_tokens: int = 1 << 16):
    """Append every sequence's prompt K/V, layer by layer (bulk append)."""
    B = w.batch
    same = len(set(w.prefill)) == 1
    for l in range(w.num_layers):
        groups = [list(range(B))] if same else [[s] for s in range(B)]
        for seqs in groups:
            T0 = w.prefill[seqs[0]]
            for t0 in range(0, T0, chunk_tokens):
                n = min(chunk_tokens, T0 - t0)
                k, v = w.prefill_kv(l, seqs, device=device, tok0=[t0] * len(seqs), n_tok=n)
                sl = slots[seqs[0]:seqs[0] + len(seqs)]
                cache.append(l, sl, k, v)
                del k, v


def decode_step(cache: ekv.Cache, w: workloads.Workload, slots: torch.Tensor, inp: Inputs,
                i: int, out: list, fires: bool, delta_out: torch.Tensor | None = None,
                fused: bool = False, combine=None, overlap: bool = True):
    """One decode step over all layers; out[l] ([B,Hq,d]) receives each layer's O.
    With `fused` each layer's append and attention run as one launch, each but the
    first overlapping the previous layer's (`overlap`; valid here because a
    layer's inputs do not come from the previous layer's output).  With
    `combine` (several GPUs, each holding a shard of the batch) the canary
    readings, written to `delta_out` ([L, 3] fp32), are combined over the ranks
    by combine(delta_out) before the tier update."""
    if fires and combine is not None and delta_out is None:
        raise ValueError("combining readings over ranks needs delta_out")
    for l in range(w.num_layers):
        q, k, v = inp.layer(l, i)
        if fused:
            # the previous launch is the fused step of layer l-1 unless this is
            # the first layer or the canary ran after each layer
            cache.append_decode_attn(l, slots, k, v, q, out[l],
                                     after_other_layer=overlap and l > 0 and not fires)
        else:
            cache.append(l, slots, k, v)
            cache.decode_attn(l, slots, q, out[l])
        if fires:
            cache.canary_kl(l, slots, q, None if delta_out is None else delta_out[l])
    if fires:
        if combine is not None:
            combine(delta_out)
            cache.tier_update(delta_out)
        else:
            cache.tier_update()

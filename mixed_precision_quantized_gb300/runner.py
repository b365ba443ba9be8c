"""Issue the decode path of a workload through the C ABI.

One decode step is, per layer l: append the step's K/V (ring write, V
quantization, K staging or seal, page admission at the layer's tier) and
decode attention over the whole cache.  On a firing step the canary of every
layer then runs in one launch (a layer's ring and queries are final once its
append is done, so the readings are those of a canary right after each
layer), and the controller updates every layer's EMA and tier.
"""
from __future__ import annotations

import torch

from . import ekv, workloads


class Inputs:
    """Device-resident per-step inputs of a workload (Q, new K, new V per layer)."""

    def __init__(self, w: workloads.Workload, step0: int, n_steps: int, device="cuda",
                 order=None):
        """`order`: the batch positions' sequences (default 0 .. B-1); position i
        holds sequence order[i], to match a slot list in that order."""
        self.k, self.v = [], []
        L = w.num_layers
        # Q of every layer of a step side by side, [n, L, B, Hq, d], for the
        # canary's all-layer launch
        self.q_all = torch.empty(n_steps, L, w.batch, w.num_q_heads, w.head_dim,
                                 dtype=torch.float16, device=device)
        for l in range(L):
            k, v = w.step_kv(l, step0, n_steps, seqs=order, device=device)  # [B, n, Hkv, d]
            q = w.step_q(l, step0, n_steps, seqs=order, device=device)      # [B, n, Hq, d]
            self.k.append(k.transpose(0, 1).contiguous())          # [n, B, Hkv, d]
            self.v.append(v.transpose(0, 1).contiguous())
            self.q_all[:, l] = q.transpose(0, 1)
        self.q = [self.q_all[:, l] for l in range(L)]              # [n, B, Hq, d] views
        self.step0, self.n = step0, n_steps

    def step_q(self, i: int) -> torch.Tensor:
        """Q of every layer of local step i, [L, B, Hq, d]."""
        return self.q_all[i]

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
                fused: bool = False, combine=None, overlap="dependent"):
    """One decode step over all layers; out[l] ([B,Hq,d]) receives each layer's O.
    With `fused` each layer's append and attention run as one launch.  `overlap`
    lets each launch start before the work before it has finished:
    "dependent" (every layer; as in a model, where a layer's q, k, v come from
    the previous layer's output: the launch streams pages early and reads them
    after that work finishes), "independent" or True (every layer but the first,
    reading its inputs early too: valid here only because the workload's inputs
    are fresh draws, not the previous layer's output), or False/None (none).  With
    `combine` (several GPUs, each holding a shard of the batch) the canary
    readings, written to `delta_out` ([L, 3] fp32), are combined over the ranks
    by combine(delta_out) before the tier update."""
    if fires and combine is not None and delta_out is None:
        raise ValueError("combining readings over ranks needs delta_out")
    L = w.num_layers
    for l in range(L):
        q, k, v = inp.layer(l, i)
        if fused:
            # independent: the previous launch is the fused step of layer l-1
            # unless this is the first layer.  dependent: the previous launch must
            # not append to this layer, so a one-layer workload (whose previous
            # launch is this layer's own last step) does not overlap.
            cache.append_decode_attn(l, slots, k, v, q, out[l],
                                     after_other_layer=(overlap is True or
                                                        overlap == "independent") and l > 0,
                                     after_producer=overlap == "dependent" and L > 1)
        else:
            cache.append(l, slots, k, v)
            cache.decode_attn(l, slots, q, out[l])
    if fires:
        cache.canary_kl_layers(0, slots, inp.step_q(i), delta_out)
        if combine is not None:
            combine(delta_out)
            cache.tier_update(delta_out)
        else:
            cache.tier_update()

"""Multi-GPU decode: one process per GPU.

Attention and the append are independent per (sequence, KV head), so the path
shards two ways.  By batch (`shard`): N GPUs hold N shards of the batch (weak
scaling), each drawing its own sequences from a rank-offset seed.  By KV heads
(`head_shard`, the layout for a batch of one): every GPU holds every sequence
but only Hkv/N of its KV heads and their query heads (strong scaling).  Either
way the one exchange is the controller's: a layer's tier is
shared by the whole batch ("EchoKV: watching a language model decide its own
precision", "Show the math — what the canary actually computes": the KL is
averaged over the step's queries), so at a canary firing the ranks add their
per-layer readings weighted by their query counts (all-reduce of L*3 sums and
one count) and every rank runs the identical tier update on the batch-wide
mean.  The timing collectives are the barrier around each timed region and the
max of its time over ranks.
"""
from __future__ import annotations

import dataclasses
import os

import torch
import torch.distributed as dist


@dataclasses.dataclass(frozen=True)
class Ranks:
    world: int
    rank: int
    local: int


def from_env() -> Ranks:
    """World size, rank and local rank as torchrun exports them (1, 0, 0 alone)."""
    return Ranks(int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
                 int(os.environ.get("LOCAL_RANK", "0")))


def shard(workload, rank: int):
    """This rank's replica: the same shapes, its own sequences (seed offset by rank)."""
    return workload if rank == 0 else workload.scaled(seed=workload.seed + 1000003 * rank)


def head_shard(workload, rank: int, world: int):
    """This rank's part of a split by KV heads (the pages' tensor-parallel layout:
    "EchoKV: watching a language model decide its own precision", "Hardware &
    serving configuration", TP = 4/8): the same sequences, KV heads
    [rank * Hkv / world, (rank + 1) * Hkv / world) and the query heads of their
    groups.  Every draw is the full workload's, sliced to those heads, so the
    ranks together hold exactly the unsplit workload.  Attention and the append
    stay on the rank that owns the heads; the one exchange is again the
    canary's (combine_readings with this rank's B * Hq / world queries)."""
    H, Hq = workload.num_kv_heads, workload.num_q_heads
    if world < 1 or H % world:
        raise ValueError(f"{H} KV heads do not split over {world} ranks")
    if world == 1:
        return workload
    n = H // world
    return HeadShard(**{f.name: getattr(workload, f.name)
                        for f in dataclasses.fields(workload)
                        if f.name not in ("num_kv_heads", "num_q_heads")},
                     num_kv_heads=n, num_q_heads=Hq // world, kv_head0=rank * n,
                     full_kv_heads=H, full_q_heads=Hq)


def barrier(r: Ranks) -> None:
    if r.world > 1:
        dist.barrier()


def max_over_ranks(r: Ranks, seconds: float, device) -> float:
    """The slowest rank's time for a region every rank timed."""
    if r.world == 1:
        return seconds
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(r: Ranks, units_per_rank: int, seconds_max: float) -> float:
    """Units all ranks processed per second of the slowest rank."""
    return r.world * units_per_rank / seconds_max


def total_queries(r: Ranks, n_queries: int, device) -> int:
    """Queries per step over all ranks (once, outside any captured region)."""
    if r.world == 1:
        return n_queries
    n = torch.tensor([n_queries], dtype=torch.int64, device=device)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return int(n.item())


def combine_readings(r: Ranks, delta, n_queries: int, total: int):
    """Batch-wide canary readings from this rank's [L, 3] means over its
    `n_queries` queries: sum over ranks of delta_r * n_r / total, in place (a
    no-op alone).  Only a scale and one all-reduce, so it can be captured in a
    CUDA graph."""
    if r.world == 1:
        return delta
    delta.mul_(n_queries / total)
    dist.all_reduce(delta, op=dist.ReduceOp.SUM)
    return delta


def majority_tiers(vectors) -> list:
    """Per-layer majority of several ranks' tier vectors; a tie goes to the
    widest of the tied tiers (more bits: the conservative choice)."""
    vectors = [list(v) for v in vectors]
    out = []
    for l in range(len(vectors[0])):
        votes: dict = {}
        for v in vectors:
            votes[int(v[l])] = votes.get(int(v[l]), 0) + 1
        top = max(votes.values())
        out.append(max(b for b, n in votes.items() if n == top))
    return out


def consolidate_tiers(r: Ranks, cache, device="cpu") -> list:
    """The pages' consolidation before a freeze ("EchoKV: watching a language
    model decide its own precision", "Measurement protocol", phase 2): every
    rank's per-layer tiers are gathered, each layer takes the ranks' majority,
    and every rank sets that vector.  Returns it (this rank's own alone)."""
    mine = [int(t) for t in cache.state()["tiers"]]
    if r.world == 1:
        return mine
    t = torch.tensor(mine, dtype=torch.int32, device=device)
    got = [torch.zeros_like(t) for _ in range(r.world)]
    dist.all_gather(got, t)
    voted = majority_tiers([g.cpu().tolist() for g in got])
    cache.set_tiers(voted)
    return voted


def share_artifact(r: Ranks, artifact=None):
    """One static artifact for every rank ("Behavior-Guided KV-Cache
    Quantization": theta* and b* are model-level, frozen before inference):
    rank 0 passes the artifact it calibrated, the others None, and all get rank
    0's copy (its arrays read-only).  Alone it returns `artifact`."""
    if r.world == 1:
        return artifact
    if r.rank == 0 and artifact is None:
        raise ValueError("rank 0 must hold the artifact")
    box = [artifact if r.rank == 0 else None]
    dist.broadcast_object_list(box, src=0)
    art = box[0]
    for a in (art.k_clip, art.v_clip):
        a.setflags(write=False)
    return art


def _head_shard_class():
    from . import workloads

    @dataclasses.dataclass
    class HeadShard(workloads.Workload):
        """A workload restricted to a contiguous range of KV heads (and their
        query heads): draws of the full workload, sliced."""
        kv_head0: int = 0
        full_kv_heads: int = 0
        full_q_heads: int = 0

        def full(self):
            base = {f.name: getattr(self, f.name) for f in dataclasses.fields(workloads.Workload)}
            base.update(num_kv_heads=self.full_kv_heads, num_q_heads=self.full_q_heads)
            return workloads.Workload(**base)

        def _kv(self):
            return slice(self.kv_head0, self.kv_head0 + self.num_kv_heads)

        def _q(self):
            G = self.full_q_heads // self.full_kv_heads
            return slice(self.kv_head0 * G, (self.kv_head0 + self.num_kv_heads) * G)

        def k_gain(self, layer: int):
            return self.full().k_gain(layer)[self._kv()]

        def prefill_kv(self, layer, seqs, device="cpu", tok0=None, n_tok=None):
            k, v = self.full().prefill_kv(layer, seqs, device=device, tok0=tok0, n_tok=n_tok)
            return k[:, :, self._kv()].contiguous(), v[:, :, self._kv()].contiguous()

        def step_kv(self, layer, step0, n_steps, seqs=None, device="cpu"):
            k, v = self.full().step_kv(layer, step0, n_steps, seqs=seqs, device=device)
            return k[:, :, self._kv()].contiguous(), v[:, :, self._kv()].contiguous()

        def step_q(self, layer, step0, n_steps, seqs=None, device="cpu"):
            q = self.full().step_q(layer, step0, n_steps, seqs=seqs, device=device)
            return q[:, :, self._q()].contiguous()

    return HeadShard


HeadShard = _head_shard_class()

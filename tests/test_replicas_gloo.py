"""The multi-GPU path: independent replicas, a barrier around each timed region
and the slowest rank's time.  Run as two gloo ranks on CPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from mixed_precision_quantized_gb300 import replicas, workloads


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        R = replicas.from_env()
        replicas.barrier(R)
        t = [0.25, 0.75][rank]                      # rank 1 is the slow one
        tmax = replicas.max_over_ranks(R, t, "cpu")
        rate = replicas.whole_job_rate(R, 32 * 64, tmax)
        w = replicas.shard(workloads.llama8b_batch32(), rank)
        k, _ = w.prefill_kv(0, [0], device="cpu", tok0=[0], n_tok=16)
        gathered = [torch.zeros_like(k) for _ in range(world)]
        dist.all_gather(gathered, k.contiguous())
        out.put((rank, R.world, R.rank, tmax, rate, w.seed, w.name,
                 bool(torch.equal(gathered[0], gathered[1]))))
    finally:
        dist.destroy_process_group()


def test_two_replicas_on_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, k0, t0, v0, s0, n0, same0), (r1, w1, k1, t1, v1, s1, n1, same1) = res
    assert (w0, w1, k0, k1) == (2, 2, 0, 1)
    assert t0 == t1 == 0.75                          # both ranks report the slowest time
    assert v0 == v1 == pytest.approx(2 * 32 * 64 / 0.75)
    assert s0 != s1 and n0 == n1                     # same shapes, own sequences
    assert not same0 and not same1                   # replicas draw different K


def test_single_process_defaults(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    R = replicas.from_env()
    assert (R.world, R.rank, R.local) == (1, 0, 0)
    assert replicas.max_over_ranks(R, 1.5, "cpu") == 1.5
    assert replicas.whole_job_rate(R, 10, 2.0) == 5.0
    w = workloads.tiny()
    assert replicas.shard(w, 0) is w

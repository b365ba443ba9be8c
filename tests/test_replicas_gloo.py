"""The multi-GPU path: a shard of the batch per rank, a barrier around each timed
region, the slowest rank's time, and the one exchange -- the canary readings
combined over the ranks before the tier update.  Run as two gloo ranks on CPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from mixed_precision_quantized_gb300 import replicas, synth, workloads
from oracle import canary


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


def _windows_and_q(B, Hq, Hkv, d, lens):
    """Seeded canary inputs: per sequence a window [Hkv, n_s, d] and Q [B, Hq, d]."""
    wins = [synth.draw16(21, 77, synth.T_K, 0, [s], [0], lens[s], Hkv, d)[0].numpy()
            .transpose(1, 0, 2).copy() for s in range(B)]
    q = synth.draw16(22, 77, synth.T_Q, 0, list(range(B)), [0] * B, 1, Hq, d)[:, 0].numpy()
    return wins, q


def _combine_main(rank: int, world: int, port: int, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        R = replicas.from_env()
        B, Hq, Hkv, d = 5, 8, 2, 64
        wins, q = _windows_and_q(B, Hq, Hkv, d, [9, 64, 33, 64, 17])
        mine = [0, 1, 2] if rank == 0 else [3, 4]          # uneven shards
        L = 2
        delta = torch.zeros(L, 3, dtype=torch.float64)
        for l in range(L):
            delta[l] = torch.from_numpy(canary.layer_delta(q[mine] * (l + 1),
                                                           [wins[s] for s in mine]))
        nq = len(mine) * Hq
        total = replicas.total_queries(R, nq, "cpu")
        replicas.combine_readings(R, delta, nq, total)
        out.put((rank, total, delta.numpy().copy()))
    finally:
        dist.destroy_process_group()


def test_canary_readings_combined_over_ranks():
    """Two ranks holding 3 and 2 of 5 sequences: the combined readings equal the
    oracle's readings over all 5 (mean over all queries), on both ranks."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_combine_main, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted((q.get(timeout=180) for _ in ps), key=lambda x: x[0])
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    B, Hq, Hkv, d = 5, 8, 2, 64
    wins, qq = _windows_and_q(B, Hq, Hkv, d, [9, 64, 33, 64, 17])
    want = np.stack([canary.layer_delta(qq * (l + 1), wins) for l in range(2)])
    for rank, total, got in res:
        assert total == B * Hq
        assert np.allclose(got, want, rtol=1e-12, atol=1e-15), (rank, got, want)
    assert np.array_equal(res[0][2], res[1][2])       # identical on every rank


def test_combine_is_identity_alone(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    R = replicas.from_env()
    x = torch.tensor([[0.1, 0.2, 0.3]], dtype=torch.float64)
    assert replicas.total_queries(R, 40, "cpu") == 40
    assert replicas.combine_readings(R, x, 40, 40) is x and x.tolist() == [[0.1, 0.2, 0.3]]


# ---- consolidation of per-rank tiers before a freeze (majority vote) ---------------


class _FakeCache:
    """Stands in for a GPU cache: holds a tier vector."""

    def __init__(self, tiers):
        self.tiers = list(tiers)

    def state(self):
        return {"tiers": list(self.tiers)}

    def set_tiers(self, tiers):
        self.tiers = list(tiers)


_RANK_TIERS = [[4, 8, 2, 4, 8], [4, 2, 2, 8, 8], [8, 2, 4, 2, 4]]


def _vote_main(rank: int, world: int, port: int, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        c = _FakeCache(_RANK_TIERS[rank])
        voted = replicas.consolidate_tiers(replicas.from_env(), c)
        out.put((rank, voted, c.tiers))
    finally:
        dist.destroy_process_group()


def test_tiers_consolidated_by_majority_on_three_ranks():
    from oracle import controller
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_vote_main, args=(r, 3, port, q)) for r in range(3)]
    for p in ps:
        p.start()
    res = sorted((q.get(timeout=180) for _ in ps), key=lambda x: x[0])
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    want = controller.majority_vote(_RANK_TIERS)
    # layer by layer: 4,4,8 -> 4; 8,2,2 -> 2; 2,2,4 -> 2; 4,8,2 -> tie -> 8; 8,8,4 -> 8
    assert want == [4, 2, 2, 8, 8]
    for rank, voted, tiers in res:
        assert voted == want and tiers == want


def test_majority_matches_oracle_on_random_vectors():
    from oracle import controller
    rng = np.random.default_rng(5)
    for _ in range(200):
        n = int(rng.integers(1, 8))
        vecs = rng.choice([2, 4, 8, 16], size=(n, 12)).tolist()
        assert replicas.majority_tiers(vecs) == controller.majority_vote(vecs)
    assert controller.majority_vote([[2], [8]]) == [8]            # tie -> widest
    assert controller.majority_vote([[2], [2], [8]]) == [2]       # majority beats width


def _artifact_rank(rank: int, world: int, port: int, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from mixed_precision_quantized_gb300 import artifacts
        R = replicas.from_env()
        mine = None
        if rank == 0:
            rng = np.random.default_rng(3)
            mine = artifacts.Artifact([4, 8, 4], [4, 4, 4],
                                      rng.random((3, 2, 64)).astype(np.float32) + 0.5,
                                      rng.random((3, 2)).astype(np.float32) + 0.5,
                                      [1.0, 0.99, 0.9], [1.0, 1.0, 0.99], [0.1, 0.3, 0.2],
                                      0.5, 4, 8)
        got = replicas.share_artifact(R, mine)
        out.put((rank, got.k_bits, got.k_clip.tobytes(), got.v_clip.tobytes(),
                 got.sensitivity, bool(got.k_clip.flags.writeable)))
    finally:
        dist.destroy_process_group()


def test_static_artifact_shared_by_all_ranks():
    """Rank 0's calibrated thresholds and bits reach every rank unchanged, read-only."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_artifact_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, b0, k0, v0, s0, w0), (r1, b1, k1, v1, s1, w1) = res
    assert (r0, r1) == (0, 1)
    assert b0 == b1 == [4, 8, 4] and k0 == k1 and v0 == v1 and s0 == s1
    assert not w0 and not w1


# ---- split by KV heads (batch-1 multi-GPU layout) ---------------------------------


def _head_split_workload():
    # 70B-shaped, two layers, a short context, the canary at every step
    return workloads.llama70b_128k().scaled(num_layers=2, prefill=[150], steps=3,
                                            canary_period=1)


def _head_split_main(rank: int, world: int, port: int, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import controller, decoder
        R = replicas.from_env()
        w = _head_split_workload()
        mine = replicas.head_shard(w, rank, world)
        nq = mine.batch * mine.num_q_heads
        total = replicas.total_queries(R, nq, "cpu")
        ctl = controller.Controller(w.k_bits_init, w.alpha, w.tau)
        tr = decoder.Trace()
        res = {"rank": rank, "heads": (mine.kv_head0, mine.num_kv_heads), "total": total,
               "delta": {}, "tiers": {}, "out": {}, "pages": {}}
        for t in range(w.steps):
            tr.tiers.append(list(ctl.tiers))
            delta = torch.zeros(w.num_layers, 3, dtype=torch.float64)
            for l in range(w.num_layers):
                q = mine.step_q(l, t, 1)[:, 0].numpy()
                delta[l] = torch.from_numpy(canary.layer_delta(q, decoder.layer_windows(mine, l, t)))
            replicas.combine_readings(R, delta, nq, total)     # the one exchange
            res["delta"][t] = delta.numpy().copy()
            ctl.update(delta.numpy().astype(np.float32))
            res["tiers"][t] = list(ctl.tiers)
        tr.tiers.append(list(ctl.tiers))
        run = decoder.ReferenceRun(mine, tr)
        run.prefill()
        for t in range(w.steps):
            o = run.step()
            res["out"][t] = {k: v.copy() for k, v in o.items()}
        st = run.state[(0, 0)]
        res["pages"] = {(j, h): st.page_expect(j, h) for j in range((st.T + 15) // 16)
                        for h in range(mine.num_kv_heads)}
        out.put(res)
    finally:
        dist.destroy_process_group()


def test_kv_head_split_two_ranks_on_gloo():
    """Two ranks owning 4 of the 8 KV heads each (and their 32 query heads): each
    rank's attention outputs and page bytes equal the unsplit oracle's for its
    heads, the canary readings combined over the ranks equal the unsplit
    readings, and both ranks reach the unsplit controller's tiers."""
    from oracle import decoder
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_head_split_main, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted((q.get(timeout=300) for _ in ps), key=lambda x: x["rank"])
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = _head_split_workload()
    G = w.group
    full = decoder.controller_trace(w, w.steps)
    ref = decoder.ReferenceRun(w, full)
    ref.prefill()
    outs = [ref.step() for _ in range(w.steps)]
    st = ref.state[(0, 0)]
    for r in res:
        h0, n = r["heads"]
        assert r["total"] == w.batch * w.num_q_heads
        for t in range(w.steps):
            assert np.allclose(r["delta"][t], full.delta[t], rtol=1e-12, atol=1e-15)
            assert r["tiers"][t] == full.after[t]
            for key, o in r["out"][t].items():
                assert np.array_equal(o, outs[t][key][h0 * G:(h0 + n) * G]), (t, key)
        for (j, h), exp in r["pages"].items():
            want = st.page_expect(j, h0 + h)
            assert exp.keys() == want.keys()
            for name in exp:
                assert np.array_equal(exp[name], want[name]), (j, h, name)
    assert np.array_equal(res[0]["delta"][0], res[1]["delta"][0])


def test_head_shard_slices_the_unsplit_draws():
    w = workloads.tiny()
    with pytest.raises(ValueError):
        replicas.head_shard(w, 0, 3)                      # 2 KV heads over 3 ranks
    assert replicas.head_shard(w, 0, 1) is w
    parts = [replicas.head_shard(w, r, 2) for r in range(2)]
    k, v = w.prefill_kv(1, [0], n_tok=40)
    q = w.step_q(1, 2, 1)
    assert torch.equal(torch.cat([p.prefill_kv(1, [0], n_tok=40)[0] for p in parts], 2), k)
    assert torch.equal(torch.cat([p.prefill_kv(1, [0], n_tok=40)[1] for p in parts], 2), v)
    assert torch.equal(torch.cat([p.step_q(1, 2, 1) for p in parts], 2), q)
    assert torch.equal(torch.cat([p.k_gain(1) for p in parts], 0), w.k_gain(1))
    assert [p.group for p in parts] == [w.group] * 2
    assert parts[1].scaled(steps=2).kv_head0 == 1          # survives scaling

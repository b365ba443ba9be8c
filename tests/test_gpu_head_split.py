"""The split by KV heads through the library, with two ranks emulated one after
the other on one GPU: each rank's cache holds 4 of the 8 KV heads (and their
query heads) of the same sequence.  Per step each rank runs its fused decode
step; at a firing each rank runs its canary, the two readings are combined
weighted by query count (what combine_readings does over NCCL), and both ranks
apply the identical tier update.  Outputs and page bytes of each rank's heads
match the unsplit oracle's, and the tiers match the unsplit controller's."""
import numpy as np
import pytest
import torch

from mixed_precision_quantized_gb300 import build, ekv, replicas, runner, workloads
from oracle import decoder, pages

from gpu_harness import ATOL, RTOL, KL_TOL, tier_flip_is_ambiguous

pytestmark = pytest.mark.gpu


def test_two_head_ranks_match_the_unsplit_oracle():
    build.build()
    w = workloads.llama70b_128k().scaled(num_layers=2, prefill=[700], steps=66)
    shards = [replicas.head_shard(w, r, 2) for r in range(2)]
    L, G = w.num_layers, w.group
    full = decoder.controller_trace(w, w.steps, device="cuda")
    ref = decoder.ReferenceRun(w, full, device="cuda")
    ref.prefill()
    slots = torch.zeros(1, dtype=torch.int32, device="cuda")
    caches = [ekv.cache_for(s) for s in shards]
    try:
        for c, s in zip(caches, shards):
            runner.prefill(c, s, slots)
        inps = [runner.Inputs(s, 0, w.steps) for s in shards]
        outs = [[torch.empty(1, s.num_q_heads, s.head_dim, dtype=torch.float16, device="cuda")
                 for _ in range(L)] for s in shards]
        deltas = [torch.zeros(L, 3, dtype=torch.float32, device="cuda") for _ in shards]
        nq = [s.batch * s.num_q_heads for s in shards]
        for t in range(w.steps):
            for c, s, inp, o in zip(caches, shards, inps, outs):
                runner.decode_step(c, s, slots, inp, t, o, False, fused=True)
            ref.advance()
            if w.fires(t):
                for c, inp, d in zip(caches, inps, deltas):
                    c.canary_kl_layers(0, slots, inp.step_q(t), d)
                comb = sum(d * (n / sum(nq)) for d, n in zip(deltas, nq))
                for c in caches:
                    c.tier_update(comb)
                dref = full.delta[t]
                assert np.all(np.abs(comb.double().cpu().numpy() - dref) <= KL_TOL)
                tiers = [c.state()["tiers"] for c in caches]
                assert tiers[0] == tiers[1]
                if tiers[0] != full.after[t]:
                    for l, (a, b) in enumerate(zip(tiers[0], full.after[t])):
                        if a != b:
                            assert tier_flip_is_ambiguous(full.ema[t][l], w.tau, a, b)
                    for c in caches:
                        c.set_tiers(full.after[t])
            if t in (0, 1, 15, 63, 64, 65):
                for r, (c, s) in enumerate(zip(caches, shards)):
                    c.sync()
                    h0 = s.kv_head0
                    for l in range(L):
                        want = ref.attend(l, 0)[h0 * G:(h0 + s.num_kv_heads) * G]
                        got = outs[r][l][0].float().cpu().numpy().astype(np.float64)
                        err = np.abs(got - want)
                        assert np.all(err <= ATOL + RTOL * np.abs(want)), (t, r, l, err.max())
        # every page byte of each rank's heads against the unsplit oracle
        for r, (c, s) in enumerate(zip(caches, shards)):
            for l in range(L):
                st = ref.state[(l, 0)]
                nb = (st.T + 15) // 16
                for h in range(s.num_kv_heads):
                    bt = c.block_table(l, 0, h)
                    raw = c.read_pages(l, 0, h, 0, nb).cpu().numpy()
                    assert len(bt) == nb
                    for j in range(nb):
                        fmt = (bt[j] >> 28) & 15
                        kb, vb = 2 << (fmt >> 2), 2 << (fmt & 3)
                        assert kb == st.kbits[j]
                        for name, want in st.page_expect(j, s.kv_head0 + h).items():
                            got = pages.extract(raw[j], kb, vb, w.head_dim, name,
                                                rows=want.shape[0])
                            assert np.array_equal(got, want), (r, l, h, j, name)
    finally:
        for c in caches:
            c.close()

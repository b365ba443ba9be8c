"""ekv_stats (the cache's realized precision: pages per format, mean stored K/V
bits per element, page bytes against fp16) against the oracle's admit-time
bookkeeping after canary-driven and forced-tier runs.

The readout is EchoKV's ("EchoKV: watching a language model decide its own
precision": the simulation's "avg bits / element" and "memory saved vs FP16";
"What the controller costs you in memory"); the cost ratio is KV-Kaizen's
c(a) / C0 ("Action Space and Cost Model") with no rank truncation."""
import numpy as np
import pytest
import torch

from mixed_precision_quantized_gb300 import build, ekv, workloads
from oracle import decoder, pages, sizes

from gpu_harness import Run

pytestmark = pytest.mark.gpu

CODE = {2: 0, 4: 1, 8: 2, 16: 3}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ekv.lib()


def expected(ref: decoder.ReferenceRun, layers, asym=False) -> dict:
    """Census of the oracle's cache state: a block's page has the K bits it was
    admitted with and the layer's V bits; the last block is open while the
    sequence's length is not a multiple of 16."""
    w = ref.w
    H, d = w.num_kv_heads, w.head_dim
    sealed, openp, openr = np.zeros(16, np.int64), np.zeros(16, np.int64), np.zeros(16, np.int64)
    kbits = vbits = 0.0
    tokens = 0
    for l in layers:
        vb = w.v_bits[l]
        for s in ref.seqs:
            st = ref.state[(l, s)]
            T, full = st.T, st.T // 16
            tokens += T * H
            for j in range(full):
                sealed[CODE[st.kbits[j]] * 4 + CODE[vb]] += H
                kbits += 16 * H * st.kbits[j]
            if T % 16:
                f = CODE[st.kbits[full]] * 4 + CODE[vb]
                openp[f] += H
                openr[f] += (T % 16) * H
                kbits += (T % 16) * H * 16           # open K rows are held raw
            vbits += T * H * vb
    nbytes = sum((sealed[f] + openp[f]) * pages.page_bytes(2 << (f >> 2), 2 << (f & 3), d,
                                                           asym=asym) for f in range(16))
    out = {"sealed_pages": sealed.tolist(), "open_pages": openp.tolist(),
           "open_rows": openr.tolist(), "tokens": tokens}
    if tokens:
        kb, vb = kbits / tokens, vbits / tokens
        # KV-Kaizen's c(a) of one token of one layer and KV head (K and V at
        # their mean stored bits, no RoPE rank truncation) over its C0
        cost = (sizes.kaizen_cost(d, 0, kb) + sizes.kaizen_cost(d, 0, vb)) / sizes.kaizen_c0(1, 1, d)
        out.update(k_bits=kb, v_bits=vb, cost_vs_c0=cost, page_bytes=float(nbytes),
                   fp16_bytes=tokens * d * 4.0, saved_vs_fp16=1 - nbytes / (tokens * d * 4.0))
    return out


def check(cache, ref, layers, asym=False):
    got = cache.stats(layers[0], len(layers))
    want = expected(ref, layers, asym)
    for k in ("sealed_pages", "open_pages", "open_rows", "tokens"):
        assert got[k] == want[k], f"{k}: {got[k]} != {want[k]}"
    for k in ("k_bits", "v_bits", "cost_vs_c0", "page_bytes", "fp16_bytes", "saved_vs_fp16"):
        assert got[k] == pytest.approx(want.get(k, 0.0), rel=1e-12, abs=1e-12), k
    return got


def test_stats_after_canary_driven_tier_changes():
    """The tiny workload (canary at every step) over 40 steps: layer 1 starts at
    K8 and the controller moves it to K4 at step 1, so its pages hold both
    widths from the block that opens at step 16 on; the census follows the
    oracle's admit-time bits throughout."""
    w = workloads.tiny().scaled(steps=40)
    r = Run(w, 40, fused=True)
    try:
        for t in range(40):
            r.step(check_attn_now=t in (0, 39))
            if t in (0, 1, 15, 16, 17, 39):
                check(r.cache, r.ref, [0, 1])
                check(r.cache, r.ref, [1])
        assert len(set(r.ref.state[(1, 0)].kbits)) > 1, "layer 1 should hold two widths"
    finally:
        r.close()


def test_stats_70b_shape():
    """G = 8, d = 128, 8 KV heads: sealed and open blocks of a 700-token prefill."""
    w = workloads.llama70b_128k().scaled(num_layers=2, prefill=[700], steps=20)
    r = Run(w, 20, fused=True)
    try:
        for t in range(20):
            r.step(check_attn_now=t in (0, 19))
            if t in (0, 3, 4, 19):
                check(r.cache, r.ref, [0, 1])
    finally:
        r.close()


def test_stats_four_formats_and_ragged_batch():
    """Tiers forced 2 -> 16 -> 8 -> 4 (one layer holds four K formats, V16), two
    sequences of different lengths, open and sealed last blocks."""
    w = workloads.Workload("mixed", 10, 1, 2, 8, 2, 128, [40, 23], 70, [2], [16])
    sched = {0: 2, 10: 16, 30: 8, 50: 4}
    tr = decoder.Trace()
    cur = 2
    for t in range(71):
        cur = sched.get(t, cur)
        tr.tiers.append([cur])
    pools = {(kb, 16): 64 for kb in (2, 4, 8, 16)}
    r = Run(w, 70, trace=tr, pool_pages=pools, fused=True)
    try:
        for t in range(70):
            if t in sched:
                r.cache.set_tiers([sched[t]])
            r.step(check_attn_now=False)
            if t in (8, 9, 24, 41, 69):
                got = check(r.cache, r.ref, [0])
        assert sum(1 for n in got["sealed_pages"] if n) >= 3
    finally:
        r.close()


def test_stats_asymmetric_pages_and_empty_cache():
    w = workloads.llama8b_layer(4).scaled(batch=2, prefill=[300, 41], steps=3, asym=True)
    r = Run(w, 3, fused=True)
    try:
        for t in range(3):
            r.step(check_attn_now=False)
        check(r.cache, r.ref, [0], asym=True)
        for s in range(2):
            r.cache.reset(s)
        got = r.cache.stats()
        assert got["tokens"] == 0 and sum(got["sealed_pages"]) == 0
        assert got["k_bits"] == 0.0 and got["saved_vs_fp16"] == 0.0
    finally:
        r.close()


def test_stats_rejects_bad_layers():
    cache = ekv.Cache(2, 1, 4, 2, 64, 64, {(4, 4): 8}, [4, 4], [4, 4])
    try:
        for a, b in ((-1, 1), (0, 0), (1, 2), (0, 3)):
            with pytest.raises(ekv.EkvError) as ei:
                cache.stats(a, b)
            assert ei.value.code == 1
    finally:
        cache.close()

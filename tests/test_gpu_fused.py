"""The fused decode step (ekv_append_decode_attn) against the two separate calls
(ekv_append, then ekv_decode_attn) on twin caches: identical lengths, block
tables and page bytes after every step, outputs within the attention
tolerance, through block seals (row 15), page pops (row 0) and a tier change."""
import ctypes

import numpy as np
import pytest
import torch

from mixed_precision_quantized_gb300 import build, ekv, runner, workloads
from oracle import pages

from gpu_harness import ATOL, RTOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ekv.lib()


def _written_bytes(raw, kb, vb, d, rows):
    """The bytes of a page that hold data once `rows` tokens are in it."""
    out = []
    for name, (off, rb, n) in pages.regions(kb, vb, d).items():
        if name.startswith("k") and rows < 16:
            continue                      # K stays in the staging rows until the seal
        m = n if name == "k_scales" else min(n, rows)
        out.append(raw[off:off + rb * m])
    return np.concatenate(out)


def _compare(a: ekv.Cache, b: ekv.Cache, w, slots_list):
    for l in range(w.num_layers):
        for s in slots_list:
            T = a.seq_len(l, s)
            assert T == b.seq_len(l, s), f"layer {l} seq {s}: lengths differ"
            for h in range(w.num_kv_heads):
                ta, tb = a.block_table(l, s, h), b.block_table(l, s, h)
                nb = (T + 15) // 16
                fa = [(e >> 28) & 15 for e in ta[:nb]]
                fb = [(e >> 28) & 15 for e in tb[:nb]]
                assert fa == fb, f"layer {l} seq {s} head {h}: page formats differ"
                ra = a.read_pages(l, s, h, 0, nb).cpu().numpy()
                rb = b.read_pages(l, s, h, 0, nb).cpu().numpy()
                for j in range(nb):
                    kb, vb = 2 << (fa[j] >> 2), 2 << (fa[j] & 3)
                    rows = min(16, T - 16 * j)
                    assert np.array_equal(_written_bytes(ra[j], kb, vb, w.head_dim, rows),
                                          _written_bytes(rb[j], kb, vb, w.head_dim, rows)), (
                        f"layer {l} seq {s} head {h} block {j}: page bytes differ")


@pytest.mark.parametrize("overlap", ["dependent", "independent", False])
@pytest.mark.parametrize("wname", ["tiny", "d128_v4_batch3"])
def test_fused_equals_separate(wname, overlap):
    """Each overlap mode of consecutive fused launches (a launch starting before
    the previous layer's ends: reading q, k, v after it, or before it, or no
    overlap) gives the separate calls' results."""
    if wname == "tiny":
        w = workloads.tiny().scaled(prefill=[29], steps=40)
    else:
        w = workloads.llama8b_batch32().scaled(num_layers=2, batch=3, prefill=[13, 47, 16],
                                               steps=40)
    caches = [ekv.cache_for(w), ekv.cache_for(w)]
    try:
        slots = torch.arange(w.batch, dtype=torch.int32, device="cuda")
        for c in caches:
            runner.prefill(c, w, slots)
        inp = runner.Inputs(w, 0, w.steps)
        outs = [[torch.empty(w.batch, w.num_q_heads, w.head_dim, dtype=torch.float16,
                             device="cuda") for _ in range(w.num_layers)] for _ in caches]
        for t in range(w.steps):
            if t == 20:                       # later blocks open at another K width
                for c in caches:
                    c.set_tiers([8 if kb != 8 else 2 for kb in w.k_bits_init])
            for c, o, fused in zip(caches, outs, (False, True)):
                runner.decode_step(c, w, slots, inp, t, o, False, fused=fused, overlap=overlap)
            for c in caches:
                c.sync()
            for l in range(w.num_layers):
                x = outs[0][l].float().cpu().numpy().astype(np.float64)
                y = outs[1][l].float().cpu().numpy().astype(np.float64)
                assert np.all(np.abs(x - y) <= ATOL + RTOL * np.abs(x)), (
                    f"step {t} layer {l}: max diff {np.abs(x - y).max():.3e}")
            if t % 5 == 4 or t == w.steps - 1:
                _compare(caches[0], caches[1], w, range(w.batch))
    finally:
        for c in caches:
            c.close()


def test_fused_pool_exhaustion_reports_enomem():
    w = workloads.Workload("oom", 12, 1, 1, 4, 2, 64, [64], 1, [4], [4])
    cache = ekv.Cache(1, 1, 4, 2, 64, 256, {(4, 4): 8}, [4], [4])
    try:
        slots = torch.zeros(1, dtype=torch.int32, device="cuda")
        k, v = w.prefill_kv(0, [0], device="cuda", n_tok=64)   # 4 blocks x 2 heads = 8 pages
        cache.append(0, slots, k, v)
        cache.sync()
        assert cache.pool_free(4, 4) == 0
        k2, v2 = w.prefill_kv(0, [0], device="cuda", tok0=[64], n_tok=1)
        q = w.step_q(0, 0, 1, device="cuda")[:, 0]
        cache.append_decode_attn(0, slots, k2, v2, q)
        with pytest.raises(ekv.EkvError) as ei:
            cache.sync()
        assert ei.value.code == 2
        cache.reset(0)
        cache.sync()
        assert cache.pool_free(4, 4) == 8
    finally:
        cache.close()


def test_fused_invalid_arguments_rejected_on_host():
    cache = ekv.Cache(1, 2, 4, 2, 64, 64, {(4, 4): 16}, [4], [4])
    try:
        slots = torch.zeros(1, dtype=torch.int32, device="cuda")
        q = torch.zeros(1, 4, 64, dtype=torch.float16, device="cuda")
        kv = torch.zeros(1, 2 * 64 + 4, dtype=torch.float16, device="cuda")
        k = kv[:, 4:].view(1, 2, 64)           # 8 bytes past a 16-byte boundary
        with pytest.raises(ekv.EkvError) as ei:
            cache.append_decode_attn(0, slots, k, k, q)
        assert ei.value.code == 1
        good = torch.zeros(1, 2, 64, dtype=torch.float16, device="cuda")
        with pytest.raises(ekv.EkvError) as ei:
            cache.append_decode_attn(3, slots, good, good, q)
        assert ei.value.code == 1
        lib = ekv.lib()
        P = lambda t: ctypes.c_void_p(t.data_ptr())
        assert lib.ekv_append_decode_attn(cache.handle, 0, 1, P(slots), P(good), P(good), P(q),
                                          P(q), 4, None) == 1     # unknown flag bit
        cache.append_decode_attn(0, slots[:0], good[:0], good[:0], q[:0])   # no-op
        cache.sync()
        assert cache.seq_len(0, 0) == 0
    finally:
        cache.close()


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
def test_slot_order_is_only_a_schedule(fused):
    """Listing the slots in another order (longest first) changes which CTAs start
    first, not the results: twin caches fed the same sequences through slot lists
    in two orders hold the same lengths and pages, and each sequence's output
    matches."""
    w = workloads.llama8b_batch32().scaled(num_layers=2, batch=5, prefill=[37, 300, 129, 64, 200],
                                           steps=20)
    order = sorted(range(w.batch), key=lambda s: -w.prefill[s])
    caches = [ekv.cache_for(w), ekv.cache_for(w)]
    try:
        ident = torch.arange(w.batch, dtype=torch.int32, device="cuda")
        for c in caches:
            runner.prefill(c, w, ident)
        slot_lists = [ident, torch.tensor(order, dtype=torch.int32, device="cuda")]
        inps = [runner.Inputs(w, 0, w.steps), runner.Inputs(w, 0, w.steps, order=order)]
        outs = [[torch.empty(w.batch, w.num_q_heads, w.head_dim, dtype=torch.float16,
                             device="cuda") for _ in range(w.num_layers)] for _ in caches]
        for t in range(w.steps):
            for c, sl, inp, o in zip(caches, slot_lists, inps, outs):
                runner.decode_step(c, w, sl, inp, t, o, w.fires(t), fused=fused)
            for c in caches:
                c.sync()
            for l in range(w.num_layers):
                x = outs[0][l][order].float().cpu().numpy().astype(np.float64)
                y = outs[1][l].float().cpu().numpy().astype(np.float64)
                assert np.all(np.abs(x - y) <= ATOL + RTOL * np.abs(x)), (t, l)
        _compare(caches[0], caches[1], w, range(w.batch))
    finally:
        for c in caches:
            c.close()

"""Pins of the oracle's cache bookkeeping (admit-time bits, open block, ring)
and of its byte accounting against the numbers the pages print."""
import json
import os

import numpy as np
import pytest

from mixed_precision_quantized_gb300 import synth, workloads
from oracle import decoder, pages, quant, sizes

from conftest import GOLDEN

F16 = np.float16


def rows(seed, n, H=2, d=64):
    return synth.draw16(seed, 55, synth.T_K, 0, [0], [0], n, H, d)[0].numpy()


def test_admit_time_bits_survive_tier_change():
    st = decoder.SeqState(2, 64, 8)
    st.append(rows(1, 10), rows(2, 10), tier=4)      # block 0 admitted at 4 bits
    st.append(rows(3, 10), rows(4, 10), tier=2)      # tokens 10..19: block 1 admitted at 2
    st.append(rows(5, 20), rows(6, 20), tier=8)      # block 2 at 8 (token 32)
    assert st.kbits == [4, 2, 8]
    kh = st.khat()
    # block 0 sealed at 4 bits, block 1 sealed at 2 bits, block 2 (8 rows) still raw
    q, s = quant.quantize(st.k[0:16], 4, axis=0)
    assert np.array_equal(kh[0:16], quant.dequantize(q, s, axis=0))
    q, s = quant.quantize(st.k[16:32], 2, axis=0)
    assert np.array_equal(kh[16:32], quant.dequantize(q, s, axis=0))
    assert np.array_equal(kh[32:40], st.k[32:40].astype(np.float32))


def test_open_block_rows_are_raw_until_sealed():
    st = decoder.SeqState(1, 64, 4)
    k = rows(7, 16, H=1)
    st.append(k[:15], k[:15], tier=2)
    assert np.array_equal(st.khat(), k[:15].astype(np.float32))
    st.append(k[15:], k[15:], tier=8)                 # 16th token seals at admit bits 2
    assert st.kbits == [2]
    assert not np.array_equal(st.khat(), k.astype(np.float32))
    assert np.max(np.abs(st.khat())) > 0


def test_v_quantized_per_token_immediately():
    st = decoder.SeqState(1, 64, 4)
    v = rows(8, 3, H=1)
    st.append(v, v, tier=4)
    q, s = quant.quantize(v, 4, axis=2)
    assert np.array_equal(st.vhat(), quant.dequantize(q, s, axis=2))


def test_ring_window_is_newest_64_oldest_first():
    st = decoder.SeqState(1, 64, 4)
    k = rows(9, 100, H=1)
    st.append(k[:10], k[:10], 4)
    assert np.array_equal(st.window(), k[:10])
    st.append(k[10:], k[10:], 4)
    assert np.array_equal(st.window(), k[36:100])


def test_page_layout_sizes():
    # d=128 per-token read bytes: K codes d*kb/8 + per-channel scales 2d/16;
    # V codes d*vb/8 + one fp16 scale.
    assert pages.page_bytes(4, 4, 128) == 16 * 64 + 256 + 16 * 64 + 32 == 2336
    assert pages.page_bytes(2, 4, 128) == 16 * 32 + 256 + 16 * 64 + 32
    assert pages.page_bytes(16, 16, 128) == 2 * 16 * 128 * 2
    for kb in (2, 4, 8, 16):
        for vb in (2, 4, 8, 16):
            for d in (64, 128):
                n = pages.page_bytes(kb, vb, d)
                assert n % 32 == 0
                regs = pages.regions(kb, vb, d)
                end = max(o + rb * r for o, rb, r in regs.values())
                assert end == n


def test_page_expect_regions_decode():
    st = decoder.SeqState(2, 64, 8)
    k = rows(10, 16)
    v = rows(11, 16)
    st.append(k, v, 4)
    e = st.page_expect(0, 1)
    q = quant.unpack(e["k_codes"], 4, 64)
    s = np.frombuffer(e["k_scales"].tobytes(), dtype=F16)
    q2, s2 = quant.quantize(k[:, 1], 4, axis=0)
    assert np.array_equal(q, q2)
    # 4-bit pages store each 8-channel group's scales as 0,4,1,5,2,6,3,7
    for grp in range(8):
        want = [8 * grp + c for c in (0, 4, 1, 5, 2, 6, 3, 7)]
        assert np.array_equal(s[8 * grp:8 * grp + 8], s2[want])
    assert e["v_codes"].shape == (16, 64) and e["v_scales"].shape == (16, 2)


def test_scale_pair_order():
    # position p of a group of n = 32/b channels holds channel p//2 + (p%2)*n/2
    assert pages.scale_order(4, 16).tolist() == [0, 4, 1, 5, 2, 6, 3, 7,
                                                   8, 12, 9, 13, 10, 14, 11, 15]
    assert pages.scale_order(2, 16).tolist() == [0, 8, 1, 9, 2, 10, 3, 11,
                                                   4, 12, 5, 13, 6, 14, 7, 15]
    assert pages.scale_order(8, 8).tolist() == list(range(8))
    for b in (2, 4):
        o = pages.scale_order(b, 128)
        assert sorted(o.tolist()) == list(range(128))     # a permutation


def test_tiny_trace_properties():
    w = workloads.tiny()
    tr = decoder.controller_trace(w, w.steps)
    assert tr.tiers[0] == [4, 8]
    assert len(tr.delta) == w.steps           # fires every step
    for t, dl in tr.delta.items():
        assert np.all(dl >= 0)
        assert np.all(dl[:, 0] > dl[:, 2])    # INT2 error dwarfs INT8
        assert all(b in (2, 4, 8) for b in tr.after[t])


def _golden():
    with open(os.path.join(GOLDEN, "paper_numbers.json")) as f:
        return json.load(f)


def _close(val, g):
    if "tol_abs" in g:
        return abs(val - g["value"]) <= g["tol_abs"]
    return abs(val - g["value"]) <= g["tol_rel"] * abs(g["value"])


def test_sizes_against_printed_numbers():
    g = _golden()
    s = g["qwen14b_kv_bytes_per_token"]["shape"]
    assert _close(sizes.kv_bytes_per_token(s["layers"], s["kv_heads"], s["head_dim"], 2),
                  g["qwen14b_kv_bytes_per_token"])
    s = g["qwen14b_32seq_8k_bytes"]["shape"]
    tot = sizes.kv_bytes_per_token(s["layers"], s["kv_heads"], s["head_dim"], 2) * 32 * 8192
    assert _close(tot, g["qwen14b_32seq_8k_bytes"])
    s = g["llama70b_ring_bytes"]["shape"]
    ring = sizes.ring_bytes(s["layers"], s["kv_heads"], s["head_dim"], s["ring"])
    assert _close(ring, g["llama70b_ring_bytes"])
    fp16 = sizes.cache_code_bytes(80, 8, 128, 131072, 16)
    int4 = sizes.cache_code_bytes(80, 8, 128, 131072, 4)
    assert _close(fp16, g["llama70b_fp16_cache_bytes_128k"])
    assert _close(int4, g["llama70b_int_cache_bytes_128k"])
    assert _close(1 - int4 / fp16, g["int4_vs_fp16_saving"])
    assert _close(int4 / ring, g["ring_vs_int_cache_ratio"])
    p = g["tau_128k"]["params"]
    assert _close(sizes.tau_scaled(p["ctx"], p["tau0"], p["ctx0"]), g["tau_128k"])
    # precision-only floor: best compression with b >= 2 against the 16-bit C0
    L, nkv, dh = 28, 4, 128
    c0 = sizes.kaizen_c0(L, nkv, dh)
    best = L * 2 * nkv * dh * 2
    assert _close(c0 / best, g["precision_only_floor"])


def test_pool_sizing_covers_growth():
    w = workloads.llama70b_128k()
    need = w.pool_pages()
    assert need[(4, 4)] == 80 * 8 * (8192 + 32)
    assert need[(2, 4)] == need[(8, 4)] == 80 * 8 * 32


def _ragged_small():
    # three sequences, one shorter than the ring that grows past it during the
    # steps, one whose window straddles the prefill/decode boundary
    return workloads.llama8b_batch32().scaled(num_layers=2, batch=3, prefill=[37, 80, 130],
                                               steps=30)


@pytest.mark.parametrize("make", [workloads.tiny, _ragged_small], ids=["tiny", "ragged"])
def test_layer_windows_equal_the_appended_ring(make):
    # layer_windows regenerates each ring window from the seeded draws; it must
    # equal the ring a step-by-step run holds after each step's append: the
    # newest min(T, 64) K's, oldest first, this step's K included ("EchoKV",
    # "Show the math" and "Do we store the whole cache in FP16? -- No.").
    w = make()
    tr = decoder.Trace()
    tr.tiers = [list(w.k_bits_init)] * (w.steps + 1)
    ref = decoder.ReferenceRun(w, tr)
    ref.prefill()
    for t in range(w.steps):
        ref.advance()
        for l in range(w.num_layers):
            wins = decoder.layer_windows(w, l, t)
            assert len(wins) == w.batch
            for i, s in enumerate(ref.seqs):
                want = ref.state[(l, s)].window().transpose(1, 0, 2)    # [Hkv, n, d]
                assert wins[i].shape == (w.num_kv_heads, min(64, w.prefill[s] + t + 1),
                                         w.head_dim)
                assert np.array_equal(wins[i], want)


def test_layer_windows_newest_is_this_steps_k_and_oldest_is_64_back():
    w = _ragged_small()
    l, t = 1, 5
    wins = decoder.layer_windows(w, l, t)
    k_step, _ = w.step_kv(l, t, 1)                      # [B, 1, Hkv, d]
    for s in range(w.batch):
        T = w.prefill[s] + t + 1
        newest = wins[s][:, -1]                          # [Hkv, d]
        assert np.array_equal(newest, k_step[s, 0].numpy())
        k_first, _ = w.prefill_kv(l, [s], tok0=[max(0, T - 64)], n_tok=1)
        assert np.array_equal(wins[s][:, 0], k_first[0, 0].numpy())
    # a window one step behind, or one that drops this step's K, differs
    behind = decoder.layer_windows(w, l, t - 1)
    for s in range(w.batch):
        assert not np.array_equal(behind[s][:, -1], wins[s][:, -1])
    short = wins[0]                                       # 37 + 6 = 43 tokens, under 64
    assert short.shape[1] == 43
    k_all, _ = w.prefill_kv(l, [0], n_tok=37)
    assert np.array_equal(short[:, :37], k_all[0].permute(1, 0, 2).numpy())

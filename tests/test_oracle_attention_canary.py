"""Pins of the oracle's attention, canary KL and controller against library
routines, closed forms and hand-worked sequences."""
import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

from mixed_precision_quantized_gb300 import synth
from oracle import attention, canary, controller, quant

F16 = np.float16


def draws(seed, n_tok, heads, d, tensor=synth.T_K, gain=1.0):
    z = synth.draw16(seed, 77, tensor, 0, [0], [0], n_tok, heads, d)[0]
    return (z.float() * gain).half().numpy()


# ------------------------------------------------------------------ attention
@pytest.mark.parametrize("Hq,Hkv,d,T", [(4, 2, 64, 37), (32, 8, 128, 300), (40, 8, 128, 17),
                                        (8, 8, 64, 1)])
def test_attention_fp16_equals_sdpa(Hq, Hkv, d, T):
    """16-bit tier: textbook attention, checked against torch SDPA (fp64, GQA expanded)."""
    q = draws(1, 1, Hq, d, synth.T_Q)[0]
    k = draws(2, T, Hkv, d)
    v = draws(3, T, Hkv, d, synth.T_V)
    o = attention.decode_attention(q, k.astype(np.float32), v.astype(np.float32))
    G = Hq // Hkv
    qt = torch.from_numpy(q.astype(np.float64)).view(1, Hq, 1, d)
    kt = torch.from_numpy(k.astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    vt = torch.from_numpy(v.astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    ref = F.scaled_dot_product_attention(qt, kt, vt)[0, :, 0].numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_attention_identical_keys_average_values():
    T, d = 9, 64
    k = np.repeat(draws(4, 1, 1, d), T, axis=0).astype(np.float32)
    v = draws(5, T, 1, d, synth.T_V).astype(np.float32)
    q = draws(6, 1, 3, d, synth.T_Q)[0]
    o = attention.decode_attention(q, k, v)
    np.testing.assert_allclose(o, np.tile(v[:, 0].astype(np.float64).mean(0), (3, 1)), atol=1e-12)


def test_attention_dominant_key_selects_its_value():
    d = 64
    k = np.zeros((5, 1, d), dtype=np.float32)
    k[3, 0, 0] = 1000.0
    q = np.zeros((1, d), dtype=F16)
    q[0, 0] = 1.0
    v = draws(7, 5, 1, d, synth.T_V).astype(np.float32)
    o = attention.decode_attention(q, k, v)
    np.testing.assert_allclose(o[0], v[3, 0], atol=1e-12)


def test_attention_empty_context_is_zero():
    o = attention.decode_attention(np.ones((2, 64), F16), np.zeros((0, 1, 64), np.float32),
                                   np.zeros((0, 1, 64), np.float32))
    assert np.all(o == 0)


# ------------------------------------------------------------------ canary
def test_kl_zero_when_quantization_is_exact():
    # {-1,0,1} at 2 bits (s = 1, codes exact); integers with absmax 127 per
    # (group, channel) at 8 bits (s = 1): the quantized window equals the window.
    rng = np.random.default_rng(0)
    w = rng.integers(-1, 2, size=(64, 64)).astype(F16)
    w[::16] = 1
    q = draws(8, 1, 4, 64, synth.T_Q)[0]
    assert np.all(canary.kl_per_query(q, w, 2) == 0.0)
    w8 = rng.integers(-127, 128, size=(40, 64)).astype(F16)
    w8[0] = 127
    w8[16] = -127
    w8[32] = 127
    assert np.all(canary.kl_per_query(q, w8, 8) == 0.0)


@pytest.mark.parametrize("n", [64, 40, 16, 5, 1])
def test_kl_matches_scipy_and_is_nonnegative(n):
    w = draws(9, n, 1, 128, gain=1.0)[:, 0]
    w[:, 7] = (w[:, 7].astype(np.float32) * 10).astype(F16)
    q = draws(10, 1, 8, 128, synth.T_Q)[0]
    sigma = 1 / np.sqrt(128)
    for b in (2, 4, 8):
        kl = canary.kl_per_query(q, w, b)
        assert np.all(kl >= 0)
        wq = canary.window_dequant(w, b).astype(np.float64)
        z = sigma * q.astype(np.float64) @ w.astype(np.float64).T
        zq = sigma * q.astype(np.float64) @ wq.T
        ref = scipy.special.rel_entr(scipy.special.softmax(z, axis=1),
                                     scipy.special.softmax(zq, axis=1)).sum(axis=1)
        np.testing.assert_allclose(kl, ref, rtol=1e-9, atol=1e-15)


def test_kl_orders_with_bits_on_average():
    tot = np.zeros(3)
    for seed in range(30):
        w = draws(100 + seed, 64, 1, 128)[:, 0]
        q = draws(200 + seed, 1, 4, 128, synth.T_Q)[0]
        tot += [canary.kl_per_query(q, w, b).mean() for b in (2, 4, 8)]
    assert tot[0] > tot[1] > tot[2] > 0


def test_window_groups_start_at_oldest_row():
    # rows 0..15 small (|x| <= 1), rows 16..19 large (127): grouping from the
    # oldest row keeps the small rows in their own group, so at 8 bits their
    # error stays within (1/127)/2; a newest-first grouping would share a
    # scale with the large rows and flush them to zero.
    w = draws(11, 20, 1, 64)[:, 0]
    w[:16] = np.clip(w[:16].astype(np.float32), -1, 1).astype(F16)
    w[:16, :] = np.where(np.arange(16)[:, None] == 0, F16(1.0), w[:16])
    w[16:] = F16(127.0)
    wq = canary.window_dequant(w, 8)
    err = np.abs(wq[:16].astype(np.float64) - w[:16].astype(np.float64))
    assert err.max() <= (1 / 127) / 2 * 1.01
    assert np.all(wq[16:] == 127.0)          # own group: s = 127/127 = 1 exactly


def test_layer_delta_is_mean_over_all_queries():
    B, Hq, Hkv, d = 3, 8, 2, 64
    Q = np.stack([draws(20 + s, 1, Hq, d, synth.T_Q)[0] for s in range(B)])
    wins = [draws(30 + s, 50, Hkv, d).transpose(1, 0, 2) for s in range(B)]
    dl = canary.layer_delta(Q, wins)
    per = np.zeros(3)
    for s in range(B):
        for h in range(Hq):
            for i, b in enumerate((2, 4, 8)):
                per[i] += canary.kl_per_query(Q[s, h:h + 1], wins[s][h // (Hq // Hkv)], b)[0]
    np.testing.assert_allclose(dl, per / (B * Hq), rtol=1e-12)


# ------------------------------------------------------------------ controller
def test_ema_hand_sequence():
    # dyadic values: every fp32 operation below is exact.
    e = controller.ema_step(None, [0.5, 0.25, 0.125], 0.25)
    assert e.tolist() == [0.5, 0.25, 0.125]
    e = controller.ema_step(e, [0.25, 0.25, 0.0], 0.25)
    # 0.75*0.5 + 0.25*0.25 = 0.4375; 0.75*0.25 + 0.25*0.25 = 0.25; 0.75*0.125 = 0.09375
    assert e.tolist() == [0.4375, 0.25, 0.09375]


def test_ema_constant_input_is_fixed_point():
    e = None
    for _ in range(10):
        e = controller.ema_step(e, [0.3, 0.02, 0.001], 0.25)
    np.testing.assert_allclose(e, [0.3, 0.02, 0.001], rtol=1e-6)


def test_pick_rule():
    assert controller.pick([0.01, 0.02, 0.03], 0.05) == 2
    assert controller.pick([0.06, 0.02, 0.03], 0.05) == 4
    assert controller.pick([0.06, 0.05, 0.001], 0.05) == 8      # strict <
    assert controller.pick([0.9, 0.5, 0.06], 0.05) == 8         # nothing under tau: widest
    assert controller.pick([0.05, 0.05, 0.05], 0.05) == 8


def test_bits_monotone_in_tau():
    rng = np.random.default_rng(1)
    for _ in range(200):
        ema = rng.exponential(0.05, 3).astype(np.float32)   # any order, not only sorted
        taus = np.sort(rng.uniform(0, 0.2, 20))
        bits = [controller.pick(ema, t) for t in taus]
        assert all(a >= b for a, b in zip(bits, bits[1:]))


def test_promote_then_demote():
    c = controller.Controller([4], alpha=1.0, tau=0.05)
    c.update([[0.5, 0.04, 0.001]])
    assert c.tiers == [4]
    c.update([[0.5, 0.2, 0.001]])
    assert c.tiers == [8]                  # promote
    c.update([[0.01, 0.002, 0.001]])
    assert c.tiers == [2]                  # demote
    c.update([[0.9, 0.9, 0.9]], freeze=True)
    assert c.tiers == [2]                  # frozen


# ---- controller variants: tau(L), hysteresis, multi-firing vote -------------------


def test_budget_at_128k_matches_the_printed_value():
    import json, os
    from conftest import GOLDEN
    g = json.load(open(os.path.join(GOLDEN, "paper_numbers.json")))["tau_128k"]
    p = g["params"]
    b = float(controller.budget(p["tau0"], p["ctx0"], [p["ctx"]]))
    assert abs(b - g["value"]) <= g["tol_abs"]


def test_budget_exact_cases():
    t = np.float32(0.05)
    assert controller.budget(0.05, 0, [131072]) == t                 # off
    assert controller.budget(0.05, 4096, []) == t                    # no sequence has tokens
    assert controller.budget(0.05, 4096, [0, 0]) == t
    assert controller.budget(0.05, 4096, [4096]) == t                # sqrt(1)
    assert controller.budget(0.05, 4096, [16384]) == np.float32(2) * t  # sqrt(4), exact
    assert controller.budget(0.05, 4096, [1024]) == t / np.float32(2)   # sqrt(1/4), exact
    # mean over the sequences holding tokens only: (8192 + 24576) / 2 = 16384
    assert controller.budget(0.05, 4096, [8192, 0, 24576]) == np.float32(2) * t


def test_hysteresis_needs_margin_to_demote_not_to_promote():
    # tau 0.05, h 0.2 -> fewer bits than the current tier need ema < 0.04
    c = controller.Controller([8], alpha=1.0, tau=0.05, hysteresis=0.2)
    c.update([[0.2, 0.045, 0.001]])
    assert c.tiers == [8]                       # 0.045 is under tau but not under 0.04
    c.update([[0.2, 0.035, 0.001]])
    assert c.tiers == [4]                       # clears the margin
    c.update([[0.2, 0.06, 0.001]])
    assert c.tiers == [8]                       # promotion at plain tau, at once
    plain = controller.Controller([8], alpha=1.0, tau=0.05)
    plain.update([[0.2, 0.045, 0.001]])
    assert plain.tiers == [4]                   # without hysteresis the same reading demotes


def test_vote_needs_consecutive_firings():
    c = controller.Controller([4], alpha=1.0, tau=0.05, vote=2)
    to8, to4, to2 = [0.3, 0.2, 0.001], [0.3, 0.01, 0.001], [0.01, 0.01, 0.001]
    c.update([to8])
    assert c.tiers == [4]                       # one firing for 8
    c.update([to4])
    assert c.tiers == [4]                       # a firing for the current tier resets
    c.update([to8])
    assert c.tiers == [4]
    c.update([to8])
    assert c.tiers == [8]                       # two in a row
    c.update([to2])
    c.update([to4])
    assert c.tiers == [8]                       # 2 then 4: different candidates
    c.update([to4])
    assert c.tiers == [4]

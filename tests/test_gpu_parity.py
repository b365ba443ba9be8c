"""CUDA path vs the oracle through the C ABI, at sizes the oracle finishes in
seconds: every page byte, every attention output, every canary reading and
every tier of the run."""
import numpy as np
import pytest
import torch

from mixed_precision_quantized_gb300 import build, ekv, runner, workloads
from oracle import controller, decoder

from gpu_harness import Run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ekv.lib()


FUSED = pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])


def _full_run(w, steps, attn_steps=None, fused=False):
    r = Run(w, steps, fused=fused)
    try:
        for t in range(steps):
            r.step(check_attn_now=attn_steps is None or t in attn_steps)
        r.check_all_pages()
        return r.max_err, r.flips
    finally:
        r.close()


@FUSED
def test_tiny_config_brute_force(fused):
    """2 layers, d=64, K bits [4,8], V8, canary + controller every step."""
    err, flips = _full_run(workloads.tiny(), 8, fused=fused)
    assert flips == []


@pytest.mark.parametrize("bits", [2, 4, 8, 16])
@FUSED
def test_llama8b_layer_small(bits, fused):
    """Uniform K=V bits, G=4, ragged prefill tail (300 = 18 blocks + 12), crosses a block."""
    w = workloads.llama8b_layer(bits).scaled(batch=2, prefill=[300, 300], steps=6)
    _full_run(w, 6, fused=fused)


@FUSED
def test_qwen14b_mixed_small(fused):
    """G=5 (padding heads), per-layer K bits 2/4/8 mixed across layers, V4."""
    w = workloads.qwen14b_32k()
    w = w.scaled(num_layers=3, prefill=[1000], steps=4,
                 k_bits_init=[2, 4, 8], v_bits=[4, 4, 4])
    _full_run(w, 4, fused=fused)


@FUSED
def test_llama70b_controller_small(fused):
    """Canary every 64 steps changes tiers mid-run: pages of several formats in one layer."""
    w = workloads.llama70b_128k().scaled(num_layers=2, prefill=[700], steps=130)
    err, flips = _full_run(w, 130, attn_steps={0, 1, 15, 63, 64, 65, 100, 127, 128, 129},
                           fused=fused)


@FUSED
def test_llama8b_batch_ragged_small(fused):
    """Ragged batch incl. a sequence shorter than the ring (37 tokens), tau 0.03."""
    w = workloads.llama8b_batch32().scaled(num_layers=2, batch=4, prefill=[37, 300, 129, 64],
                                           steps=70)
    _full_run(w, 70, attn_steps={0, 1, 2, 26, 27, 28, 63, 64, 65, 69}, fused=fused)


@pytest.mark.parametrize("T0,d,Hq,Hkv", [(1, 64, 2, 2), (15, 128, 8, 1), (16, 64, 8, 8),
                                         (17, 128, 16, 2), (33, 128, 40, 8)])
@FUSED
def test_edge_lengths_and_groups(T0, d, Hq, Hkv, fused):
    """Single-token, 15/16/17-token prefills, G = 1, 2, 5, 8."""
    w = workloads.Workload("edge", 9, 1, 1, Hq, Hkv, d, [T0], 20, [4], [8],
                           outlier_frac=0.02, outlier_gain=8.0)
    _full_run(w, 20, fused=fused)


@FUSED
def test_mixed_formats_in_one_layer_forced_tiers(fused):
    """Tiers forced 2 -> 16 -> 8 -> 4 mid-run: one layer holds four K formats (V16)."""
    w = workloads.Workload("mixed", 10, 1, 2, 8, 2, 128, [40, 23], 70, [2], [16])
    sched = {0: 2, 10: 16, 30: 8, 50: 4}
    tr = decoder.Trace()
    cur = 2
    for t in range(71):
        cur = sched.get(t, cur)
        tr.tiers.append([cur])
    pools = {(kb, 16): 64 for kb in (2, 4, 8, 16)}
    r = Run(w, 70, trace=tr, pool_pages=pools, fused=fused)
    try:
        for t in range(70):
            if t in sched:
                r.cache.set_tiers([sched[t]])
            r.step()
        r.check_all_pages()
        assert set(r.ref.state[(0, 0)].kbits) == {2, 16, 8, 4}
    finally:
        r.close()


def test_tier_update_bit_exact_with_injected_readings():
    w = workloads.Workload("ctl", 11, 6, 1, 4, 2, 64, [16], 1, [4] * 6, [4] * 6, alpha=0.25,
                           tau=0.05)
    cache = ekv.cache_for(w)
    try:
        ctl = controller.Controller(w.k_bits_init, w.alpha, w.tau)
        rng = np.random.default_rng(0)
        for it in range(12):
            d = rng.exponential(0.04, size=(6, 3)).astype(np.float32)
            d[:, 0] *= 4
            mask = np.ones(6, dtype=np.uint8)
            if it % 3 == 2:
                mask[rng.integers(0, 6, 2)] = 0
            freeze = it == 7
            dt = torch.from_numpy(d).cuda()
            mt = torch.from_numpy(mask).cuda()
            cache.tier_update(dt, mt, freeze=freeze)
            ctl.update(d, mask=mask, freeze=freeze)
            st = cache.state()
            assert st["tiers"] == ctl.tiers
            ema_gpu = np.array(st["ema"], dtype=np.float32)
            for l in range(6):
                if ctl.ema[l] is not None:
                    assert np.array_equal(ema_gpu[l], ctl.ema[l])
    finally:
        cache.close()


def test_tier_update_variants_bit_exact():
    """tau(L) with the layers' lengths, hysteresis and a 2-firing vote, against the
    oracle controller given the same lengths and readings."""
    w = workloads.Workload("ctlv", 13, 6, 2, 4, 2, 64, [16, 16], 1, [4] * 6, [4] * 6,
                           alpha=0.5, tau=0.05)
    pools = {(4, 4): 128}
    cache = ekv.Cache(6, 2, 4, 2, 64, 256, pools, w.k_bits_init, w.v_bits,
                      alpha=0.5, tau=0.05, tau_ctx0=48, hysteresis=0.25, vote=2)
    try:
        slots = torch.arange(2, dtype=torch.int32, device="cuda")
        lengths = []
        for l in range(6):   # layer l: slot 0 holds 16 + 8l tokens, slot 1 none or 40
            n0 = 16 + 8 * l
            k, v = w.prefill_kv(0, [0], device="cuda", n_tok=n0)
            cache.append(l, slots[:1], k, v)
            if l % 2:
                k, v = w.prefill_kv(0, [1], device="cuda", n_tok=40)
                cache.append(l, slots[1:], k, v)
            lengths.append([n0, 40 if l % 2 else 0])
        cache.sync()
        ctl = controller.Controller(w.k_bits_init, w.alpha, w.tau, tau_ctx0=48, hysteresis=0.25,
                                    vote=2)
        rng = np.random.default_rng(1)
        for it in range(16):
            d = rng.exponential(0.03, size=(6, 3)).astype(np.float32)
            d[:, 0] *= 3
            cache.tier_update(torch.from_numpy(d).cuda())
            ctl.update(d, lengths=lengths)
            st = cache.state()
            assert st["tiers"] == ctl.tiers, (it, st["tiers"], ctl.tiers)
            ema_gpu = np.array(st["ema"], dtype=np.float32)
            for l in range(6):
                assert np.array_equal(ema_gpu[l], ctl.ema[l])
        blob = cache.save_state()                         # the vote state travels too
        c2 = ekv.Cache(6, 2, 4, 2, 64, 256, pools, w.k_bits_init, w.v_bits,
                       alpha=0.5, tau=0.05, tau_ctx0=48, hysteresis=0.25, vote=2)
        try:
            c2.load_state(blob)
            assert c2.save_state() == blob
        finally:
            c2.close()
    finally:
        cache.close()


def test_state_save_load_round_trip():
    w = workloads.tiny()
    cache = ekv.cache_for(w)
    try:
        cache.tier_update(torch.tensor([[0.3, 0.01, 0.001], [0.2, 0.2, 0.001]], device="cuda"))
        blob = cache.save_state()
        s1 = cache.state()
        assert s1["tiers"] == [4, 8]
        cache.tier_update(torch.tensor([[0.0, 0.0, 0.0], [0.0, 0.0, 0.0]], device="cuda"))
        cache.tier_update(torch.tensor([[0.0, 0.0, 0.0], [0.0, 0.0, 0.0]], device="cuda"))
        assert cache.state() != s1
        cache.load_state(blob)
        assert cache.state() == s1
    finally:
        cache.close()


def test_pool_exhaustion_reports_enomem_and_reset_returns_pages():
    w = workloads.Workload("oom", 12, 1, 1, 4, 2, 64, [64], 1, [4], [4])
    cache = ekv.Cache(1, 1, 4, 2, 64, 256, {(4, 4): 8}, [4], [4])
    try:
        slots = torch.zeros(1, dtype=torch.int32, device="cuda")
        k, v = w.prefill_kv(0, [0], device="cuda", n_tok=64)   # 4 blocks x 2 heads = 8 pages
        cache.append(0, slots, k, v)
        cache.sync()
        assert cache.pool_free(4, 4) == 0
        k2, v2 = w.prefill_kv(0, [0], device="cuda", tok0=[64], n_tok=1)
        cache.append(0, slots, k2, v2)
        with pytest.raises(ekv.EkvError) as ei:
            cache.sync()
        assert ei.value.code == 2
        cache.reset(0)
        cache.sync()
        assert cache.pool_free(4, 4) == 8
        assert cache.seq_len(0, 0) == 0
    finally:
        cache.close()


def test_invalid_arguments_rejected_on_host():
    cache = ekv.Cache(1, 2, 4, 2, 64, 64, {(4, 4): 16}, [4], [4])
    try:
        slots = torch.zeros(1, dtype=torch.int32, device="cuda")
        q = torch.zeros(1, 4, 64, dtype=torch.float16, device="cuda")
        with pytest.raises(ekv.EkvError) as ei:
            cache.decode_attn(5, slots, q)       # layer out of range
        assert ei.value.code == 1
        with pytest.raises(ekv.EkvError):
            cache.reset(7)
        # zero sequences is a no-op
        cache.decode_attn(0, slots[:0], q[:0])
        cache.sync()
    finally:
        cache.close()
    with pytest.raises(ekv.EkvError) as ei:
        ekv.Cache(1, 1, 32, 2, 64, 64, {}, [4], [4])   # G = 16 > 8
    assert ei.value.code == 5


def test_empty_sequence_attends_to_zero():
    cache = ekv.Cache(1, 2, 4, 2, 64, 64, {(4, 4): 16}, [4], [4])
    try:
        slots = torch.tensor([1], dtype=torch.int32, device="cuda")
        q = torch.randn(1, 4, 64, device="cuda").half()
        o = cache.decode_attn(0, slots, q)
        cache.sync()
        assert torch.all(o == 0)
    finally:
        cache.close()


def test_all_layer_canary_launch_equals_per_layer_calls():
    """One canary launch over every layer gives each layer exactly the readings
    of its own call (the same CTAs, the same fixed reduction order)."""
    w = workloads.qwen14b_32k().scaled(num_layers=4, batch=2, prefill=[90, 200], steps=2,
                                       k_bits_init=[2, 4, 8, 4], v_bits=[4, 4, 4, 4])
    cache = ekv.cache_for(w)
    try:
        slots = torch.arange(w.batch, dtype=torch.int32, device="cuda")
        runner.prefill(cache, w, slots)
        inp = runner.Inputs(w, 0, 1)
        one = torch.zeros(w.num_layers, 3, dtype=torch.float32, device="cuda")
        for l in range(w.num_layers):
            cache.canary_kl(l, slots, inp.layer(l, 0)[0], one[l])
        allv = torch.zeros_like(one)
        cache.canary_kl_layers(0, slots, inp.step_q(0), allv)
        part = torch.zeros(2, 3, dtype=torch.float32, device="cuda")
        cache.canary_kl_layers(1, slots, inp.step_q(0)[1:3], part)
        cache.sync()
        assert torch.equal(one, allv)
        assert torch.equal(one[1:3], part)
        assert torch.equal(torch.tensor(cache.state()["delta"]), one[:].cpu())
        with pytest.raises(ekv.EkvError):
            cache.canary_kl_layers(3, slots, inp.step_q(0)[:2], part)   # past the last layer
    finally:
        cache.close()


@FUSED
def test_more_units_than_sms_two_ctas_per_sm(fused):
    """20 sequences x 8 KV heads = 160 (sequence, head) units > 152 SMs: the
    launch packs two half-size CTAs per SM; ragged short contexts, d 128, V4."""
    w = workloads.llama8b_batch32().scaled(num_layers=1, batch=20,
                                           prefill=[5 + 13 * i for i in range(20)], steps=6)
    _full_run(w, 6, fused=fused)


@FUSED
def test_two_ctas_per_sm_with_split_merges(fused):
    """160 units with a 40K-token capacity: the page table of a split holds 2,048
    entries in the two-CTA configuration, so each unit takes 3 splits (most of
    them empty for these short sequences) and the split merge runs."""
    w = workloads.llama8b_batch32().scaled(num_layers=1, batch=20,
                                           prefill=[5 + 13 * i for i in range(20)], steps=5)
    r = Run(w, 5, fused=fused, max_seq_len=40000)
    try:
        for _ in range(5):
            r.step()
        r.check_all_pages()
    finally:
        r.close()


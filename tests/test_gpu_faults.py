"""Failure detection without a GPU fault: a bounded device wait that gives up,
and a device allocator that fails inside ekv_create.

The wait is made to give up through the EKV_DEBUG_WAIT_EXPIRY test hook: every
wait still polls until its copy has landed and only then reports expiry, so the
kernel takes the timeout path (stop taking pages, drain the copies in flight,
return) with nothing left in flight.  The context must stay usable: the next
launch without the hook matches the oracle."""
import ctypes

import numpy as np
import pytest
import torch

from mixed_precision_quantized_gb300 import build, ekv, runner, workloads
from oracle import decoder

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2
EKV_ENOMEM, EKV_ETIMEOUT = 2, 4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ekv.lib()


def _check_against_oracle(cache, w, ref, slots, l, q, what):
    o = cache.decode_attn(l, slots, q)
    cache.sync()
    qh = ref.q_heads()
    for s in range(w.batch):
        want = ref.attend(l, s)
        g = o[s][qh].float().cpu().numpy().astype(np.float64)
        err = np.abs(g - want)
        assert np.all(err <= ATOL + RTOL * np.abs(want)), f"{what}: seq {s} max {err.max():.3e}"


@pytest.mark.parametrize("w", [
    workloads.llama70b_128k().scaled(num_layers=1, prefill=[5000], steps=2),
    workloads.llama8b_layer(8).scaled(batch=3, prefill=[300, 17, 1000], steps=2),
], ids=["one_seq_splits", "batch3"])
def test_bounded_wait_expiry_reports_timeout_and_the_context_stays_usable(w):
    cache = ekv.cache_for(w)
    try:
        slots = torch.arange(w.batch, dtype=torch.int32, device="cuda")
        runner.prefill(cache, w, slots)
        cache.sync()
        tr = decoder.Trace()
        tr.tiers = [list(w.k_bits_init)] * 3
        ref = decoder.ReferenceRun(w, tr)
        ref.prefill()
        inp = runner.Inputs(w, 0, 2)
        q, k, v = inp.layer(0, 0)

        # attention alone: the waits give up, the launch returns, the error is reported
        cache.debug_set(ekv.DEBUG_WAIT_EXPIRY, 1)
        cache.decode_attn(0, slots, q)
        with pytest.raises(ekv.EkvError) as ei:
            cache.sync()
        assert ei.value.code == EKV_ETIMEOUT
        cache.sync()                                  # the error word was cleared

        # the fused step under the hook: the append (before the page loop) still
        # happens, attention reports the expiry
        lens = [cache.seq_len(0, s) for s in range(w.batch)]
        cache.append_decode_attn(0, slots, k, v, q)
        with pytest.raises(ekv.EkvError) as ei:
            cache.sync()
        assert ei.value.code == EKV_ETIMEOUT
        assert [cache.seq_len(0, s) for s in range(w.batch)] == [n + 1 for n in lens]

        # hook off: the same handle and context give the oracle's attention
        cache.debug_set(ekv.DEBUG_WAIT_EXPIRY, 0)
        ref.advance()
        _check_against_oracle(cache, w, ref, slots, 0, q, "after the expiry")
        with pytest.raises(ekv.EkvError):
            cache.debug_set(99, 1)                    # unknown knob
    finally:
        cache.close()


def test_allocator_failure_in_create_returns_enomem_and_frees_what_it_took():
    """A dev_alloc that returns NULL at its n-th call: ekv_create fails with
    EKV_ENOMEM and hands every block it got back to dev_free; a misaligned
    block fails the same way."""
    lib = ekv.lib()
    dev = torch.cuda.current_device()
    state = {"n": 0, "fail_at": -1, "skew_at": -1, "live": {}}

    def _alloc(nbytes, ctx):
        i = state["n"]
        state["n"] += 1
        if i == state["fail_at"]:
            return None
        p = torch.cuda.caching_allocator_alloc(int(nbytes) + 256, dev)
        q = p + (8 if i == state["skew_at"] else 0)   # 8: not 16-byte aligned
        state["live"][q] = p
        return q

    def _free(q, ctx):
        p = state["live"].pop(q)
        torch.cuda.caching_allocator_delete(p)

    a, f = ekv.ALLOC_FN(_alloc), ekv.FREE_FN(_free)

    def create(fail_at, skew_at=-1):
        state.update(n=0, fail_at=fail_at, skew_at=skew_at, live={})
        cfg = ekv.EkvConfig()
        cfg.num_layers, cfg.max_seqs, cfg.num_q_heads, cfg.num_kv_heads = 2, 2, 8, 2
        cfg.head_dim, cfg.max_seq_len = 64, 256
        cfg.pool_pages[ekv.fmt_index(4, 8)] = 64
        cfg.ema_alpha, cfg.tau = 0.25, 0.05
        cfg.dev_alloc = ctypes.cast(a, ctypes.c_void_p)
        cfg.dev_free = ctypes.cast(f, ctypes.c_void_p)
        kb = (ctypes.c_uint8 * 2)(4, 4)
        vb = (ctypes.c_uint8 * 2)(8, 8)
        h = ctypes.c_void_p()
        rc = lib.ekv_create(ctypes.byref(cfg), kb, vb, ctypes.byref(h))
        return rc, h

    rc, h = create(-1)                                  # no failure: count the calls
    assert rc == 0
    total = state["n"]
    assert total > 5
    assert lib.ekv_destroy(h) == 0
    assert state["live"] == {}
    for fail_at in sorted({0, 1, total // 2, total - 1}):
        rc, h = create(fail_at)
        assert rc == EKV_ENOMEM, (fail_at, rc)
        assert not h.value
        assert state["live"] == {}, f"fail at call {fail_at}: {len(state['live'])} blocks kept"

    # a misaligned block (16-byte alignment is required) also fails cleanly
    rc, h = create(-1, skew_at=3)
    assert rc == EKV_ENOMEM
    assert not h.value
    assert state["live"] == {}

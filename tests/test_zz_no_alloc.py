"""ekv_decode_attn_noalloc: decode attention for callers that cannot allocate
device memory where they run attention (a process that reserves all device
memory up front, or code that cannot reach the handle's allocator).  Its
split-K scratch lives in a static device array inside the library, so it
must give the same outputs as ekv_decode_attn, call after call, and refuse
requests whose scratch would not fit in that array.

Called through the C ABI directly (ctypes), after the regular entry point has
produced the reference output on the same cache state.  This file is named to
be collected last."""
import ctypes

import numpy as np
import pytest
import torch

from mixed_precision_quantized_gb300 import build, ekv, runner, workloads

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _cache_after_one_step(w):
    cache = ekv.cache_for(w)
    slots = torch.arange(w.batch, dtype=torch.int32, device="cuda")
    runner.prefill(cache, w, slots)
    inp = runner.Inputs(w, 0, 2)   # step 1's queries serve as a second, different query set
    for l in range(w.num_layers):
        _, k, v = inp.layer(l, 0)
        cache.append(l, slots, k, v)
    cache.sync()
    return cache, slots, inp


@pytest.mark.parametrize("w", [
    workloads.llama8b_layer(4).scaled(batch=2, prefill=[300, 300], steps=1),
    workloads.llama70b_128k().scaled(num_layers=1, prefill=[20000], steps=1),
    workloads.tiny(),
], ids=["batch2_int4", "one_seq_many_splits", "tiny_d64"])
def test_noalloc_matches_decode_attn_on_two_calls(w):
    """Two calls in a row with different queries, each against ekv_decode_attn on
    the same query.  The split partials of the first call are still in the
    shared array when the second runs, and the two calls' outputs differ by far
    more than the tolerance, so a second call that read any stale partial
    would fail.  These launches (one CTA per SM, a page ring of two pairs per
    warp or more) give each warp a fixed set of pages and merge in a fixed
    order, so the two entry points' outputs are equal bit for bit."""
    build.build()
    lib = ekv.lib()
    cache, slots, inp = _cache_after_one_step(w)
    try:
        for l in range(w.num_layers):
            outs = []
            for call in range(2):
                q = inp.layer(l, call)[0]
                ref = torch.empty_like(q)
                assert lib.ekv_decode_attn(cache.handle, l, w.batch, _ptr(slots), _ptr(q),
                                           _ptr(ref), _stream()) == 0
                cache.sync()
                r = ref.float().cpu().numpy().astype(np.float64)
                o = torch.full_like(q, float("nan"))
                rc = lib.ekv_decode_attn_noalloc(cache.handle, l, w.batch, _ptr(slots), _ptr(q),
                                                 _ptr(o), _stream())
                assert rc == 0, lib.ekv_status_string(rc)
                cache.sync()
                g = o.float().cpu().numpy().astype(np.float64)
                assert np.all(np.isfinite(g)), f"layer {l} call {call}: unwritten outputs"
                assert torch.equal(o, ref), (
                    f"layer {l} call {call}: max diff {np.abs(g - r).max():.3e}")
                outs.append(g)
            # the test's sensitivity: most outputs of the two query sets lie further
            # apart than the tolerance
            apart = np.abs(outs[0] - outs[1]) > ATOL + RTOL * np.abs(outs[1])
            assert apart.mean() > 0.5, f"layer {l}: the two query sets give close outputs"
    finally:
        cache.close()


@pytest.mark.parametrize("w", [
    workloads.tiny(),
    workloads.llama70b_128k().scaled(num_layers=1, prefill=[3000], steps=1),
], ids=["tiny_d64", "int4_g8_many_splits"])
def test_noalloc_matches_the_oracle(w):
    """The allocation-free attention against the CPU oracle's attention over the
    same pages (prefill plus one appended step), at the attention tolerance."""
    from oracle import decoder
    build.build()
    lib = ekv.lib()
    cache, slots, inp = _cache_after_one_step(w)
    try:
        tr = decoder.Trace()
        tr.tiers = [list(w.k_bits_init)] * 2
        ref = decoder.ReferenceRun(w, tr)
        ref.prefill()
        ref.advance()
        qh = ref.q_heads()
        for l in range(w.num_layers):
            q = inp.layer(l, 0)[0]
            o = torch.full_like(q, float("nan"))
            rc = lib.ekv_decode_attn_noalloc(cache.handle, l, w.batch, _ptr(slots), _ptr(q),
                                             _ptr(o), _stream())
            assert rc == 0, lib.ekv_status_string(rc)
            cache.sync()
            for s in range(w.batch):
                want = ref.attend(l, s)
                g = o[s][qh].float().cpu().numpy().astype(np.float64)
                err = np.abs(g - want)
                assert np.all(err <= ATOL + RTOL * np.abs(want)), (
                    f"layer {l} seq {s}: max diff {err.max():.3e}")
    finally:
        cache.close()


def test_noalloc_rejects_requests_beyond_its_scratch():
    build.build()
    lib = ekv.lib()
    # 128 sequences x 8 KV heads x group 8 x d 128: the partials alone exceed 4 MiB.
    cache = ekv.Cache(1, 128, 64, 8, 128, 16, {}, [4], [4])
    try:
        slots = torch.arange(128, dtype=torch.int32, device="cuda")
        q = torch.zeros(128, 64, 128, dtype=torch.float16, device="cuda")
        o = torch.zeros_like(q)
        assert lib.ekv_decode_attn_noalloc(cache.handle, 0, 128, _ptr(slots), _ptr(q), _ptr(o),
                                           _stream()) == 1          # EKV_EINVAL
        cache.sync()                                                  # nothing was enqueued
        assert lib.ekv_decode_attn_noalloc(cache.handle, 0, 2, _ptr(slots), _ptr(q), _ptr(o),
                                           _stream()) == 0          # small request still fits
        cache.sync()
    finally:
        cache.close()


def test_two_ctas_per_sm_allocation_free_entry_point():
    """The allocation-free attention under the two-CTA configuration matches the
    handle's own (at the attention tolerance: there a CTA's warps take pages
    from a shared counter, so the fp32 summation order varies between
    launches)."""
    w = workloads.llama8b_batch32().scaled(num_layers=1, batch=20,
                                           prefill=[40 + 9 * i for i in range(20)], steps=1)
    cache = ekv.cache_for(w)
    try:
        slots = torch.arange(w.batch, dtype=torch.int32, device="cuda")
        runner.prefill(cache, w, slots)
        q = w.step_q(0, 0, 1, device="cuda")[:, 0].contiguous()
        a = torch.empty_like(q)
        b = torch.empty_like(q)
        cache.decode_attn(0, slots, q, a)
        cache.decode_attn_noalloc(0, slots, q, b)
        cache.sync()
        x = a.float().cpu().numpy().astype(np.float64)
        y = b.float().cpu().numpy().astype(np.float64)
        assert np.all(np.abs(x - y) <= 2e-3 + 1e-2 * np.abs(x))
    finally:
        cache.close()

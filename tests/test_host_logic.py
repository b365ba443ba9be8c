"""Host-side logic of the decode runner and the static-artifact bundle, on CPU:
batch-position order of the step inputs (a slot list in another order sees the
same sequences' draws), the static workload an artifact defines, and the calls
one decode step makes (overlap flags per layer, firing order)."""
import numpy as np
import pytest
import torch

from mixed_precision_quantized_gb300 import artifacts, runner, workloads


def test_inputs_follow_the_batch_order():
    w = workloads.llama8b_batch32().scaled(num_layers=2, batch=4, prefill=[37, 300, 129, 64],
                                           steps=3)
    order = [1, 2, 3, 0]
    base = runner.Inputs(w, 0, 3, device="cpu")
    perm = runner.Inputs(w, 0, 3, device="cpu", order=order)
    for l in range(w.num_layers):
        for i in range(3):
            qa, ka, va = base.layer(l, i)
            qb, kb, vb = perm.layer(l, i)
            for pos, s in enumerate(order):
                assert torch.equal(qb[pos], qa[s]) and torch.equal(kb[pos], ka[s])
                assert torch.equal(vb[pos], va[s])
        # the all-layer block of a step holds each layer's queries side by side
        assert torch.equal(perm.step_q(1)[l], perm.layer(l, 1)[0])
    assert perm.step_q(0).is_contiguous()


def test_artifact_defines_a_static_workload():
    w = workloads.qwen14b_32k().scaled(num_layers=3, prefill=[100], steps=4)
    art = artifacts.Artifact([8, 4, 8], [4, 4, 4], np.ones((3, 8, 128), np.float32),
                             np.ones((3, 8), np.float32), [1.0] * 3, [1.0] * 3, [0.3, 0.1, 0.2],
                             0.9, 4, 8)
    ws = art.workload(w)
    assert ws.k_bits_init == [8, 4, 8] and ws.v_bits == [4, 4, 4]
    assert ws.canary_period == 0 and not any(ws.fires(t) for t in range(64))
    assert (ws.num_layers, ws.prefill, ws.steps) == (w.num_layers, w.prefill, w.steps)


class _RecordingCache:
    """Stands in for ekv.Cache: records the calls a decode step makes."""

    def __init__(self):
        self.calls = []

    def append_decode_attn(self, l, slots, k, v, q, o, after_other_layer=False,
                           after_producer=False):
        self.calls.append(("fused", l, after_other_layer, after_producer))

    def append(self, l, slots, k, v):
        self.calls.append(("append", l))

    def decode_attn(self, l, slots, q, o):
        self.calls.append(("attn", l))

    def canary_kl_layers(self, l0, slots, q, delta_out):
        self.calls.append(("canary",))

    def tier_update(self, delta=None):
        self.calls.append(("tiers", delta is not None))


def _step(L, **kw):
    w = workloads.tiny().scaled(num_layers=L, k_bits_init=[4] * L, v_bits=[8] * L)
    inp = runner.Inputs(w, 0, 1, device="cpu")
    out = [torch.empty(w.batch, w.num_q_heads, w.head_dim, dtype=torch.float16)
           for _ in range(L)]
    c = _RecordingCache()
    runner.decode_step(c, w, torch.zeros(1, dtype=torch.int32), inp, 0, out, **kw)
    return c.calls


def test_decode_step_overlap_flags():
    """Which launches may start before the work before them ends: with dependent
    inputs every layer (never a one-layer step, whose previous launch appends to
    the same layer); with independent inputs every layer but the first; none
    without overlap; the separate calls never."""
    fused = lambda calls: [c for c in calls if c[0] == "fused"]
    assert fused(_step(3, fires=False, fused=True)) == [
        ("fused", l, False, True) for l in range(3)]
    assert fused(_step(1, fires=False, fused=True)) == [("fused", 0, False, False)]
    for ov in ("independent", True):
        assert fused(_step(3, fires=False, fused=True, overlap=ov)) == [
            ("fused", 0, False, False), ("fused", 1, True, False), ("fused", 2, True, False)]
    for ov in (False, None):
        assert fused(_step(3, fires=False, fused=True, overlap=ov)) == [
            ("fused", l, False, False) for l in range(3)]
    assert _step(2, fires=False) == [("append", 0), ("attn", 0), ("append", 1), ("attn", 1)]


def test_decode_step_firing_order():
    """A firing step runs every layer's launches, then one all-layer canary, then
    the tier update (with the combined readings when ranks combine them)."""
    calls = _step(2, fires=True, fused=True)
    assert [c[0] for c in calls] == ["fused", "fused", "canary", "tiers"]
    assert calls[-1] == ("tiers", False)
    seen = []
    delta = torch.zeros(2, 3)
    calls = _step(2, fires=True, fused=True, delta_out=delta, combine=lambda d: seen.append(d))
    assert [c[0] for c in calls] == ["fused", "fused", "canary", "tiers"]
    assert calls[-1] == ("tiers", True) and len(seen) == 1 and seen[0] is delta
    with pytest.raises(ValueError):
        _step(2, fires=True, fused=True, combine=lambda d: d)

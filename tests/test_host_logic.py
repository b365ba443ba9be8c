"""Host-side logic of the decode runner and the static-artifact bundle, on CPU:
batch-position order of the step inputs (a slot list in another order sees the
same sequences' draws) and the static workload an artifact defines."""
import numpy as np
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

"""The KIVI-style asymmetric quantizer on the GPU against the oracle: every
page byte (unsigned codes, fp16 scales and zero points) bit-exact, attention
within the attention tolerance, canary readings within 1e-4 and the tiers they
pick, with the separate calls and the fused step."""
import pytest
import torch

from mixed_precision_quantized_gb300 import build, ekv, workloads
from oracle import decoder

from gpu_harness import Run

pytestmark = pytest.mark.gpu

FUSED = pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ekv.lib()


def _full_run(w, steps, fused, attn_steps=None, **kw):
    r = Run(w, steps, fused=fused, **kw)
    try:
        for t in range(steps):
            r.step(check_attn_now=attn_steps is None or t in attn_steps)
        r.check_all_pages()
        return r
    finally:
        r.close()


@FUSED
def test_tiny_controller_every_step(fused):
    """2 layers, d 64, K 4/8, V8, canary and controller (asymmetric quant_b) every step."""
    _full_run(workloads.tiny().scaled(asym=True), 8, fused)


@pytest.mark.parametrize("bits", [2, 4, 8, 16])
@FUSED
def test_llama8b_layer_small(bits, fused):
    """Uniform K=V bits, G=4, ragged prefill tail, crosses a block."""
    w = workloads.llama8b_layer(bits).scaled(batch=2, prefill=[300, 300], steps=6, asym=True)
    _full_run(w, 6, fused)


@FUSED
def test_qwen14b_mixed_widths_small(fused):
    """G=5 (padding heads), K 2/4/8 across layers, V 2/4/8."""
    w = workloads.qwen14b_32k().scaled(num_layers=3, prefill=[1000], steps=4,
                                       k_bits_init=[2, 4, 8], v_bits=[2, 4, 8], asym=True)
    _full_run(w, 4, fused)


@pytest.mark.parametrize("T0,d,Hq,Hkv", [(1, 64, 2, 2), (17, 128, 16, 2), (33, 128, 40, 8)])
@FUSED
def test_edge_lengths_and_groups(T0, d, Hq, Hkv, fused):
    w = workloads.Workload("edge_asym", 9, 1, 1, Hq, Hkv, d, [T0], 20, [4], [8],
                           outlier_frac=0.02, outlier_gain=8.0, asym=True)
    _full_run(w, 20, fused)


@FUSED
def test_four_k_formats_in_one_layer_v16(fused):
    """Tiers forced 2 -> 16 -> 8 -> 4: asymmetric K pages of every width beside V16."""
    w = workloads.Workload("mixed_asym", 10, 1, 2, 8, 2, 128, [40, 23], 70, [2], [16], asym=True)
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
    finally:
        r.close()


@FUSED
def test_controller_changes_tiers_mid_run(fused):
    """70B shape, 2 layers, canary every 64 steps: several formats in one layer."""
    w = workloads.llama70b_128k().scaled(num_layers=2, prefill=[700], steps=130, asym=True)
    _full_run(w, 130, fused, attn_steps={0, 1, 63, 64, 65, 127, 128, 129})


def test_clipping_thresholds_unsupported_with_the_asymmetric_quantizer():
    cache = ekv.Cache(1, 1, 4, 2, 64, 64, {(4, 4): 8}, [4], [4], asym=True)
    try:
        with pytest.raises(ekv.EkvError) as ei:
            cache.set_clip(0, None, [1.0, 1.0])
        assert ei.value.code == 5
        slots = torch.zeros(1, dtype=torch.int32, device="cuda")
        raw = cache.read_pages(0, 0, 0, 0, 1)
        assert raw.shape[1] == ekv.page_bytes(16, 16, 64, asym=True)
    finally:
        cache.close()


@FUSED
def test_more_units_than_sms_two_ctas_per_sm(fused):
    """160 (sequence, head) units: the packed two-CTA launch on asymmetric pages."""
    w = workloads.llama8b_batch32().scaled(num_layers=1, batch=20,
                                           prefill=[5 + 13 * i for i in range(20)], steps=6,
                                           asym=True)
    _full_run(w, 6, fused)

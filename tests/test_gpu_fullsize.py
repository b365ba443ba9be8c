"""Full-size workloads, run through the C ABI exactly as bench.py runs them
(same library, same split schedule, the fused append + attention launch; the
single-layer sweep uses the separate append and attention calls), checked
against the oracle on sampled outputs the oracle can compute one by one:

  * the controller over ALL layers at every firing: canary readings within
    1e-4 and tiers bit-exact (or a flip inside the reading tolerance of tau);
  * attention of sampled (step, layer, sequence, KV head) within
    2e-3 + 1e-2 |o|, over the full cached context;
  * every byte of every page of sampled (layer, sequence, KV head).
"""
import pytest

from mixed_precision_quantized_gb300 import build, ekv, workloads

from gpu_harness import Run, check_pages

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ekv.lib()


def _sampled(w, steps, layers, seqs, heads, attn_steps, fused=True):
    r = Run(w, steps, layers=layers, seqs=seqs, heads=heads, fused=fused)
    try:
        for t in range(steps):
            r.step(check_attn_now=t in attn_steps)
        for l in layers:
            for s in seqs:
                check_pages(r.cache, r.ref, l, s)
        return r.max_err, r.flips
    finally:
        r.close()


def test_llama70b_128k_full():
    """80 layers x 131072 tokens; canary firings at steps 0, 64, 128 over all layers."""
    w = workloads.llama70b_128k()
    _sampled(w, 130, layers=[0, 79], seqs=[0], heads=[0, 7], attn_steps={0, 64, 129})


def test_qwen14b_32k_full():
    """48 layers x 32768 tokens, per-layer K widths 2/4/8 mixed, V4, G = 5."""
    w = workloads.qwen14b_32k()
    pick = [w.k_bits_init.index(b) for b in (2, 4, 8)]
    _sampled(w, 128, layers=pick, seqs=[0], heads=[0, 3], attn_steps={0, 127})


def test_llama8b_batch32_full():
    """32 layers x 32 ragged sequences (1K-8K), tau 0.03: tiers change mid-run."""
    w = workloads.llama8b_batch32()
    _sampled(w, 256, layers=[0, 31], seqs=[0, 13, 31], heads=[0, 7],
             attn_steps={0, 64, 128, 255})


@pytest.mark.parametrize("bits", [2, 4, 8, 16])
def test_llama8b_layer_full(bits):
    """One layer, 8 sequences x 4096 tokens, uniform K = V bits, 64 steps."""
    w = workloads.llama8b_layer(bits)
    _sampled(w, 64, layers=[0], seqs=[0, 7], heads=[0, 3, 7], attn_steps={0, 31, 63},
             fused=False)

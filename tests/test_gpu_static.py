"""Static-artifact mode on the GPU against the oracle: the percentile select
(bit-exact thresholds), clipped quantization through append, fused step and
canary (bit-exact pages, attention and readings within tolerance), the
calibration (scores, choices, AutoK) and decode with a loaded artifact."""
import math

import numpy as np
import pytest
import torch

from mixed_precision_quantized_gb300 import artifacts as product
from mixed_precision_quantized_gb300 import build, ekv, workloads
from oracle import artifacts

from gpu_harness import KL_TOL, Run

pytestmark = pytest.mark.gpu

F16, F32 = np.float16, np.float32


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ekv.lib()


def _data(shape, seed):
    """fp16 draws with ties (integers), signed zeros and a few large outliers."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape) * 2
    m = rng.random(shape)
    x = np.where(m < 0.2, np.round(x), x)
    x = np.where(m > 0.995, x * 300, x)
    x = np.where((m > 0.4) & (m < 0.41), -0.0, x)
    return x.astype(F16)


QS = (0.0, 0.3, 0.5, 0.9, 0.99, 0.999, 1.0)


@pytest.mark.parametrize("T,H,d", [(1, 2, 64), (37, 3, 64), (1000, 8, 128), (5003, 1, 128)])
def test_percentile_thresholds_bit_exact(T, H, d):
    x = _data((T, H, d), T * 7 + H)
    xg = torch.from_numpy(x).cuda()
    for q in QS:
        assert np.array_equal(ekv.k_thresholds(xg, q).cpu().numpy(), artifacts.k_thresholds(x, q))
        assert np.array_equal(ekv.v_thresholds(xg, q).cpu().numpy(), artifacts.v_thresholds(x, q))


def test_percentile_ragged_and_strided_groups():
    x = _data((301, 90), 5)
    xg = torch.from_numpy(x).cuda()
    for q in QS:
        # 45 column groups (a ragged tile of 13), every other column
        got = ekv.abs_percentile(xg, q, 301, 90, 45, 2, 1).cpu().numpy()
        want = [artifacts.abs_percentile(x[:, 2 * g], q) for g in range(45)]
        assert np.array_equal(got, np.array(want, F32))
        # 9 segment groups of width 7 (not a multiple of the warp)
        got = ekv.abs_percentile(xg, q, 301, 90, 9, 10, 7).cpu().numpy()
        want = [artifacts.abs_percentile(x[:, 10 * g:10 * g + 7], q) for g in range(9)]
        assert np.array_equal(got, np.array(want, F32))


def test_percentile_invalid_arguments():
    x = torch.zeros(4, 8, dtype=torch.float16, device="cuda")
    for args in ((4, 8, 8, 1, 1, 1.5), (4, 8, 8, 1, 1, -0.1), (0, 8, 8, 1, 1, 0.5),
                 (4, 8, 0, 1, 1, 0.5), (4, 8, 8, 1, 0, 0.5)):
        n_rows, rs, ng, gs, gw, q = args
        with pytest.raises(ekv.EkvError) as ei:
            ekv.abs_percentile(x, q, n_rows, rs, ng, gs, gw,
                               out=torch.empty(8, dtype=torch.float32, device="cuda"))
        assert ei.value.code == 1


def test_clip_set_get_round_trip_and_invalid():
    cache = ekv.Cache(2, 1, 4, 2, 64, 64, {(4, 4): 16}, [4, 4], [4, 4])
    try:
        k, v = cache.get_clip(1)
        assert torch.isinf(k).all() and torch.isinf(v).all()
        kc = torch.rand(2, 64) + 0.5
        kc[1, 3] = math.inf
        cache.set_clip(1, kc, [2.0, math.inf])
        k, v = cache.get_clip(1)
        assert torch.equal(k, kc) and v.tolist() == [2.0, math.inf]
        assert torch.isinf(cache.get_clip(0)[0]).all()
        for bad in (0.0, -1.0, math.nan):
            with pytest.raises(ekv.EkvError) as ei:
                cache.set_clip(1, None, [bad, 1.0])
            assert ei.value.code == 1
        assert cache.get_clip(1)[1].tolist() == [2.0, math.inf]   # unchanged
        cache.set_clip(1, None, None)
        k, v = cache.get_clip(1)
        assert torch.isinf(k).all() and torch.isinf(v).all()
        with pytest.raises(ekv.EkvError):
            cache.set_clip(2, None, None)
    finally:
        cache.close()


def _clips_from_prefill(w, qk, qv):
    """Thresholds from the workload's own prefill (aggressive percentiles, so
    most groups are clipped), with a few channels and one head left unclipped."""
    clips = {}
    for l in range(w.num_layers):
        ks, vs = [], []
        for s in range(w.batch):
            k, v = w.prefill_kv(l, [s], n_tok=w.prefill[s])
            ks.append(k[0].numpy())
            vs.append(v[0].numpy())
        kc = artifacts.k_thresholds(np.concatenate(ks), qk)
        vc = artifacts.v_thresholds(np.concatenate(vs), qv)
        kc[0, ::7] = np.inf
        vc[-1] = np.inf
        clips[l] = (kc, vc)
    return clips


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_clipped_decode_matches_oracle(bits, fused):
    w = workloads.Workload(f"clip_b{bits}", 31, 2, 2, 8, 2, 128, [45, 70], 40, [bits, bits],
                           [bits, 4], canary_period=8, alpha=0.25, tau=0.05,
                           outlier_fixed=(5, 77), outlier_gain=8.0)
    run = Run(w, w.steps, gen_device="cpu", fused=fused, clips=_clips_from_prefill(w, 0.8, 0.9))
    try:
        for _ in range(w.steps):
            run.step()
        run.check_all_pages()
    finally:
        run.close()


CAL = dict(candidates=(1.0, 0.99, 0.9), frac=0.5, low=4, high=8)


def _cal_workload():
    return workloads.Workload("calib", 21, 3, 2, 4, 2, 64, [40, 70], 1, [4, 4, 4], [4, 8, 16],
                              outlier_fixed=(3, 17), outlier_gain=10.0)


def _ambiguous(scores, a, b, tol):
    return abs(float(scores[a]) - float(scores[b])) <= 2 * tol


def test_calibration_matches_oracle(tmp_path):
    w = _cal_workload()
    art, got = product.calibrate(w, **CAL)
    ref = artifacts.calibrate(w, CAL["candidates"], CAL["frac"], CAL["low"], CAL["high"])
    VTOL = 2.0 ** -9          # on sqrt(score): fp16 rounding of both attention outputs
    for l in range(w.num_layers):
        ks, kr = np.array(got["k_score"][l]), np.array(ref["k_score"][l])
        assert np.all(np.abs(ks - kr) <= KL_TOL), (l, ks, kr)
        vs, vr = np.array(got["v_score"][l]), np.array(ref["v_score"][l])
        assert np.all(np.abs(np.sqrt(vs) - np.sqrt(vr)) <= VTOL), (l, vs, vr)
        i, ir = got["k_choice"][l], ref["k_choice"][l]
        assert i == ir or _ambiguous(kr, i, ir, KL_TOL)
        if i == ir:
            assert np.array_equal(art.k_clip[l], ref["k_clip"][l])
        j, jr = got["v_choice"][l], ref["v_choice"][l]
        assert j == jr or abs(math.sqrt(vr[j]) - math.sqrt(vr[jr])) <= 2 * VTOL
        if j == jr:
            assert np.array_equal(art.v_clip[l], ref["v_clip"][l])
        assert abs(art.sensitivity[l] - ref["sensitivity"][l]) <= KL_TOL
    # AutoK of the library on the GPU's sensitivities is the oracle's, exactly
    k, order = ekv.autok(art.sensitivity, CAL["frac"])
    assert k == artifacts.autok(art.sensitivity, CAL["frac"]) == got["n_protected"]
    assert order == artifacts.sensitivity_order(art.sensitivity)
    assert art.k_bits == artifacts.allocate(art.sensitivity, k, CAL["low"], CAL["high"])
    if art.k_bits != ref["k_bits"]:     # only through sensitivities within the tolerance
        s = ref["sensitivity"]
        assert any(abs(s[a] - s[b]) <= 2 * KL_TOL for a in range(len(s)) for b in range(a))
    # the artifact survives a save and a read-only load
    p = tmp_path / "art.npz"
    art.save(p)
    back = product.Artifact.load(p)
    assert back.k_bits == art.k_bits and np.array_equal(back.k_clip, art.k_clip)
    assert not back.k_clip.flags.writeable


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
def test_static_mode_decode_matches_oracle(fused):
    w = _cal_workload()
    art, _ = product.calibrate(w, **CAL)
    ws = art.workload(w.scaled(steps=24))
    clips = {l: (art.k_clip[l], art.v_clip[l]) for l in range(w.num_layers)}
    run = Run(ws, ws.steps, gen_device="cpu", fused=fused, clips=clips)
    try:
        assert run.cache.state()["tiers"] == art.k_bits
        for _ in range(ws.steps):
            run.step()
        run.check_all_pages()
        assert run.cache.state()["tiers"] == art.k_bits      # read-only: never fired
    finally:
        run.close()


def test_output_error_sums_match_fp64():
    """ekv_output_error: sum (a - b)^2 and sum b^2 of two fp16 tensors, fp64 on the
    GPU, against numpy's fp64 sums (rounding order aside); empty input gives 0."""
    g = torch.Generator().manual_seed(7)
    for n in (1, 31, 1000, 70001):
        a = torch.randn(n, generator=g).half()
        b = (a.float() + 0.01 * torch.randn(n, generator=g)).half()
        num, den = ekv.output_error(a.cuda(), b.cuda())
        a64, b64 = a.double().numpy(), b.double().numpy()
        assert num == pytest.approx(float(((a64 - b64) ** 2).sum()), rel=1e-12)
        assert den == pytest.approx(float((b64 ** 2).sum()), rel=1e-12)
    z = torch.zeros(0, dtype=torch.float16, device="cuda")
    assert ekv.output_error(z, z) == (0.0, 0.0)

"""Pins of the static-artifact oracle: the clipped quantizer, nearest-rank
percentile thresholds, the AutoK allocator, candidate choice, the Value score
and the calibration's structure.

Independent checks: hand-worked clipped quantization with an exact scale;
numpy's inverted-CDF percentile (a library routine with its own definition);
brute force over every subset for AutoK; closed forms for the Value score.
"""
import itertools
import math

import numpy as np
import pytest

from mixed_precision_quantized_gb300 import workloads
from oracle import artifacts, canary, quant

F16, F32 = np.float16, np.float32


def test_clipped_quantizer_hand_worked():
    # c = 0.875 with b = 4: s = 0.875 / 7 = 0.125 exactly (absmax 5 is clipped away).
    x = np.array([0.1, 0.5, 3.0, -5.0, 0.0625, -0.1875], dtype=F16)
    q, s = quant.quantize(x, 4, axis=0, clip=F32(0.875))
    assert float(s) == 0.125
    # 0.1 (fp16 0.0999756) / 0.125 = 0.7998 -> 1; 0.5 -> 4; 3 and -5 saturate;
    # 0.0625 / 0.125 = 0.5 -> 0 (tie to even); -0.1875 / 0.125 = -1.5 -> -2 (tie to even)
    assert q.tolist() == [1, 4, 7, -7, 0, -2]


def test_clip_above_absmax_or_infinite_is_the_plain_quantizer():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((16, 64)) * 3).astype(F16)
    for b in (2, 4, 8):
        q0, s0 = quant.quantize(x, b, axis=0)
        for c in (np.full(64, np.inf, F32), np.abs(x).max(0).astype(F32),
                  np.abs(x).max(0).astype(F32) * 2):
            q1, s1 = quant.quantize(x, b, axis=0, clip=c)
            assert np.array_equal(q0, q1) and np.array_equal(s0.view(np.uint16), s1.view(np.uint16))


def test_clipped_values_saturate_and_inside_error_is_half_step():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((40, 32)) * 2).astype(F16)
    c = np.full(40, 1.5, F32)                       # one threshold per token (axis 1 groups)
    for b in (4, 8):
        qm = (1 << (b - 1)) - 1
        q, s = quant.quantize(x, b, axis=1, clip=c)
        xf = x.astype(np.float64)
        big = np.abs(xf) >= 1.5 + 1e-9
        assert np.all(np.abs(q[big]) == qm) and np.all(np.sign(q[big]) == np.sign(xf[big]))
        xh = quant.dequantize(q, s, axis=1).astype(np.float64)
        sf = s.astype(np.float64)[:, None]
        inside = np.abs(xf) <= (qm * sf)
        assert np.all(np.abs(xh - xf)[inside] <= (sf / 2 + 1e-6 * sf).repeat(32, 1)[inside])


def test_nonpositive_or_nan_threshold_rejected():
    x = np.ones(4, dtype=F16)
    for c in (0.0, -1.0, np.nan):
        with pytest.raises(ValueError):
            quant.quantize(x, 4, axis=0, clip=F32(c))


@pytest.mark.parametrize("n", [1, 2, 7, 16, 100, 1001])
def test_percentile_matches_numpy_inverted_cdf(n):
    rng = np.random.default_rng(n)
    x = (rng.standard_normal(n) * 4).astype(F16)
    a = np.abs(x.astype(np.float64))
    for q in (0.0, 0.01, 0.25, 0.5, 0.9, 0.99, 0.999, 1.0):
        want = np.percentile(a, q * 100, method="inverted_cdf") if q > 0 else a.min()
        assert float(artifacts.abs_percentile(x, q)) == float(want), q


def test_percentile_brute_force_definition():
    # the smallest data magnitude v with #{|x| <= v} >= q n (and at least one value)
    rng = np.random.default_rng(9)
    for _ in range(50):
        n = int(rng.integers(1, 12))
        x = rng.integers(-6, 7, n).astype(F16)
        q = float(rng.choice([0.0, 0.1, 1 / 3, 0.5, 0.75, 0.9, 1.0]))
        a = sorted(abs(float(v)) for v in x)
        want = min(v for v in a if sum(u <= v for u in a) >= max(1, q * n))
        assert float(artifacts.abs_percentile(x, q)) == want


def test_thresholds_per_channel_and_per_head():
    rng = np.random.default_rng(11)
    k = (rng.standard_normal((50, 3, 8)) * np.arange(1, 9)).astype(F16)   # channel scales differ
    kt = artifacts.k_thresholds(k, 0.9)
    a = np.abs(k.astype(np.float64))
    want = np.percentile(a, 90, axis=0, method="inverted_cdf")          # [3, 8]
    assert kt.shape == (3, 8) and np.array_equal(kt.astype(np.float64), want)
    vt = artifacts.v_thresholds(k, 0.9)
    want_v = [np.percentile(a[:, h, :].ravel(), 90, method="inverted_cdf") for h in range(3)]
    assert np.array_equal(vt.astype(np.float64), np.array(want_v))


def _min_protected_brute(s, frac):
    tot = math.fsum(s)
    for k in range(len(s) + 1):
        for sub in itertools.combinations(range(len(s)), k):
            if math.fsum(s[i] for i in sub) >= frac * tot - 1e-12 * tot:
                return k
    raise AssertionError


def test_autok_hand_example():
    s = [1.0, 8.0, 4.0, 3.0]                         # order 1, 2, 3, 0; prefix 8, 12, 15, 16
    assert artifacts.sensitivity_order(s) == [1, 2, 3, 0]
    assert artifacts.autok(s, 0.75) == 2               # 12 >= 12
    assert artifacts.autok(s, 0.76) == 3               # 12 < 12.16 <= 15
    assert artifacts.autok(s, 0.5) == 1
    assert artifacts.autok(s, 1.0) == 4
    assert artifacts.autok(s, 0.0) == 0
    assert artifacts.allocate(s, 2, 2, 8) == [2, 8, 8, 2]


def test_autok_brute_force_and_edges():
    rng = np.random.default_rng(5)
    for _ in range(200):
        L = int(rng.integers(1, 9))
        s = [float(v) for v in rng.integers(0, 20, L) / 8.0]     # dyadic: sums exact
        frac = float(rng.choice([0.0, 0.125, 0.25, 0.5, 0.625, 0.75, 0.875, 1.0]))
        k = artifacts.autok(s, frac)
        assert k == _min_protected_brute(s, frac)
        top = artifacts.sensitivity_order(s)[:k]
        assert math.fsum(s[i] for i in top) >= frac * math.fsum(s)
    assert artifacts.autok([0.0, 0.0, 0.0], 0.9) == 0
    assert artifacts.autok([0.0, 2.0, 0.0, 1.0], 1.0) == 2        # only positive layers count
    assert artifacts.autok([1.0] * 10, 0.35) == 4                # uniform: ceil(frac L)
    assert artifacts.sensitivity_order([2.0, 5.0, 2.0, 5.0]) == [1, 3, 0, 2]
    for bad in ([-1.0, 2.0], [float("nan")]):
        with pytest.raises(ValueError):
            artifacts.autok(bad, 0.5)
    with pytest.raises(ValueError):
        artifacts.autok([1.0], 1.5)


def test_choose_lowest_then_larger_percentile():
    assert artifacts.choose([1.0, 0.99, 0.9], [0.3, 0.1, 0.2]) == 1
    assert artifacts.choose([0.9, 1.0, 0.99], [0.1, 0.1, 0.2]) == 1
    assert artifacts.choose([0.99, 0.999], [0.0, 0.0]) == 1


def test_value_score_closed_forms():
    rng = np.random.default_rng(2)
    T, H, d, G = 20, 2, 16, 2
    ks = [(rng.standard_normal((T, H, d))).astype(F16)]
    Q = (rng.standard_normal((1, H * G, d))).astype(F16)
    row = np.concatenate([np.arange(-127, 128, 17), [127]])[:d].astype(F16)   # integers, absmax 127
    vs = [np.broadcast_to(row, (T, H, d)).astype(F16)]
    inf = np.full(H, np.inf, F32)
    # 8-bit with s = 1: every integer row is exact, so the output does not move
    assert artifacts.v_perturbation(Q, ks, vs, 8, inf) == 0.0
    assert artifacts.v_perturbation(Q, ks, vs, 16, np.full(H, 1.0, F32)) == 0.0
    # clip at 63.5: s = 0.5, every token's row becomes clip(row, +-63.5) exactly,
    # so o moves from row to the clipped row whatever the attention weights
    got = artifacts.v_perturbation(Q, ks, vs, 8, np.full(H, 63.5, F32))
    r = row.astype(np.float64)
    want = ((np.clip(r, -63.5, 63.5) - r) ** 2).sum() / (r ** 2).sum()
    assert got == pytest.approx(want, rel=1e-12)


def test_calibration_structure_on_a_tiny_workload():
    w = workloads.Workload("calib", 21, 3, 2, 4, 2, 64, [40, 70], 1, [4, 4, 4], [4, 8, 16],
                           outlier_fixed=(3, 17), outlier_gain=10.0)
    cands = (1.0, 0.99, 0.9)
    out = artifacts.calibrate(w, cands, frac=0.5, low=4, high=8)
    L, Hkv, d = w.num_layers, w.num_kv_heads, w.head_dim
    assert out["k_clip"].shape == (L, Hkv, d) and out["v_clip"].shape == (L, Hkv)
    for l in range(L):
        ks, vs, Q = artifacts.calibration_data(w, l)
        K = np.concatenate(ks)
        i, j = out["k_choice"][l], out["v_choice"][l]
        assert np.array_equal(out["k_clip"][l], artifacts.k_thresholds(K, cands[i]))
        assert out["sensitivity"][l] == out["k_score"][l][i]
        assert out["k_score"][l][i] == min(out["k_score"][l])
        # q = 1 thresholds are the absmax of all calibration keys: no clipping,
        # so the score is the plain canary's 4-bit reading
        wins = [k[-64:].transpose(1, 0, 2) for k in ks]
        assert out["k_score"][l][0] == canary.layer_delta(Q, wins)[1]
    k = out["n_protected"]
    assert k == artifacts.autok(out["sensitivity"], 0.5)
    assert sorted(out["k_bits"]).count(8) == k and set(out["k_bits"]) <= {4, 8}
    assert out["v_bits"] == list(w.v_bits)

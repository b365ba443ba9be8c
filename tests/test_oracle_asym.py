"""Pins of the oracle's KIVI-style asymmetric quantizer, its page bytes and
its canary, independent of its own code: hand-worked cases with exact scales,
a brute-force characterisation (u is the nearest code in [0, 2^b - 1] to
(x - z) / s, ties to even; s is the fp16 rounding of the fp32 rounding of
(hi - lo) / (2^b - 1), computed through Python's struct module), the error
bound, the exact group minimum, packing by hand, and a window the quantizer
represents exactly (KL exactly 0)."""
import struct

import numpy as np
import pytest

from oracle import canary, pages, quant

F16, F32 = np.float16, np.float32


def h(*xs):
    return np.array(xs, dtype=F16)


def test_hand_worked_b2_b4():
    u, s, z = quant.quantize_asym(h(0, 1, 2, 3), 2, axis=0)
    assert (u.tolist(), float(s), float(z)) == ([0, 1, 2, 3], 1.0, 0.0)
    # lo -1, hi 2: s = 3 / 3 = 1; x - lo = 0, 1.5, 3 -> 0, 2 (tie to even), 3
    u, s, z = quant.quantize_asym(h(-1, 0.5, 2), 2, axis=0)
    assert (u.tolist(), float(s), float(z)) == ([0, 2, 3], 1.0, -1.0)
    # lo -2, hi 13: s = 15 / 15 = 1; x - lo = 0, 0.5, 2.5, 15 -> 0, 0, 2, 15 (ties to even)
    u, s, z = quant.quantize_asym(h(-2, -1.5, 0.5, 13), 4, axis=0)
    assert (u.tolist(), float(s), float(z)) == ([0, 0, 2, 15], 1.0, -2.0)
    # b = 8: lo 10, hi 265 -> s = 255 / 255 = 1
    u, s, z = quant.quantize_asym(h(10, 137.5, 265, 11), 8, axis=0)
    assert (u.tolist(), float(s), float(z)) == ([0, 128, 255, 1], 1.0, 10.0)


def test_constant_group_has_zero_scale_and_exact_values():
    x = h(3.25, 3.25, 3.25)
    for b in (2, 4, 8):
        u, s, z = quant.quantize_asym(x, b, axis=0)
        assert float(s) == 0.0 and u.tolist() == [0, 0, 0] and float(z) == 3.25
        assert quant.dequantize_asym(u, s, z, axis=0).tolist() == [3.25] * 3


def _f32(v):
    return struct.unpack("f", struct.pack("f", v))[0]


def _f16(v):
    return struct.unpack("e", struct.pack("e", v))[0]


def test_brute_force_characterisation():
    rng = np.random.default_rng(6)
    for _ in range(300):
        b = int(rng.choice([2, 4, 8]))
        n = int(rng.integers(2, 20))
        x = (rng.standard_normal(n) * rng.choice([0.01, 1, 30])).astype(F16)
        u, s, z = quant.quantize_asym(x, b, axis=0)
        xs = [float(v) for v in x]
        lo, hi = min(xs), max(xs)
        L = (1 << b) - 1
        s_ref = _f16(_f32(_f32(hi - lo) / L))
        assert float(s) == s_ref and float(z) == lo
        for xi, ui in zip(xs, u.tolist()):
            if s_ref == 0:
                assert ui == 0
                continue
            r = _f32(_f32(xi - lo) / s_ref)
            best = min(range(L + 1), key=lambda c: (abs(c - r), c % 2))
            assert ui == best, (xi, r, ui, best)


def test_error_bound_and_exact_minimum():
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((16, 64)) * 3 + 1).astype(F16)
    for b in (2, 4, 8):
        u, s, z = quant.quantize_asym(x, b, axis=0)
        xh = quant.dequantize_asym(u, s, z, axis=0).astype(np.float64)
        xf = x.astype(np.float64)
        sf = s.astype(np.float64)
        # the group minimum is reproduced exactly; every value within half a step
        # (plus the fp32 roundings of the difference, the division and the sum)
        assert np.array_equal(xh[np.argmin(xf, 0), np.arange(64)], xf.min(0))
        assert np.all(np.abs(xh - xf) <= sf / 2 * (1 + 1e-3) + 1e-6 * np.abs(xf))


def test_unsigned_packing_by_hand():
    # 4-bit: channel c in byte c // 2, low nibble first
    assert quant.pack_unsigned(np.array([[1, 15, 0, 7]]), 4).tolist() == [[0xF1, 0x70]]
    # 2-bit: four channels per byte, LSB first
    assert quant.pack_unsigned(np.array([[3, 0, 1, 2]]), 2).tolist() == [[0b10010011]]


def test_asym_page_regions_and_bytes():
    d = 64
    r = pages.regions(4, 4, d, asym=True)
    assert r["k_zeros"] == (16 * d // 2 + 2 * d, 2 * d, 1)
    vo = pages.k_part_bytes(4, d, asym=True)
    assert vo == 16 * d // 2 + 4 * d
    assert r["v_zeros"] == (vo + 16 * d // 2 + 32, 2, 16)
    assert pages.page_bytes(4, 4, d, asym=True) == pages.page_bytes(4, 4, d) + 2 * d + 32
    assert pages.page_bytes(16, 16, d, asym=True) == pages.page_bytes(16, 16, d)
    k16 = (np.arange(16 * d).reshape(16, d) % 11 - 3).astype(F16)
    got = pages.sealed_k_bytes(4, k16, asym=True)
    # every channel holds -3 .. 7 over the block: s = 10 / 15 rounded, z = -3
    z = got["k_zeros"].view(F16)
    assert np.all(z == F16(-3)) and got["k_zeros"].shape == (1, 2 * d)
    with pytest.raises(ValueError):
        pages.sealed_k_bytes(4, k16, clip=np.ones(d, F32), asym=True)


def test_canary_exact_window_gives_zero_kl():
    # every channel's 16-row group holds integers 0..3 with both ends present:
    # lo 0, hi 3, s = 1, codes exact -> the quantized window equals the window
    rng = np.random.default_rng(1)
    w = rng.integers(0, 4, (32, 16)).astype(F16)
    w[0], w[1], w[16], w[17] = 0, 3, 0, 3
    q = rng.standard_normal((4, 16)).astype(F16)
    for b in (2, 4, 8):
        assert canary.window_dequant(w, 2, asym=True).tolist() == w.astype(F32).tolist()
        assert np.all(canary.kl_per_query(q, w, 2, asym=True) == 0.0)
    # and a symmetric quantizer does not represent it: 3 / 1 = 3 > qmax at 2 bits
    assert np.any(canary.kl_per_query(q, w, 2) > 0)

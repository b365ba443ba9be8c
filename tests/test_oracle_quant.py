"""Pins of the oracle's quantizer and code packing, independent of its own code.

Each case is worked by hand from the quantizer's definition (the workloads'
formula q = clamp(round_half_even(x/s), -qmax, qmax), s = absmax/qmax stored
as fp16), or checked against a brute-force characterisation: q is the
candidate in [-qmax, qmax] nearest to x/s, ties to even; s is the fp16
rounding of the fp32 rounding of absmax/qmax, computed through Python's
struct module (a separate rounding implementation).
"""
import struct

import numpy as np
import pytest
import torch

from mixed_precision_quantized_gb300 import synth
from oracle import quant

F16 = np.float16


def h(*xs):
    return np.array(xs, dtype=F16)


def test_rne_ties_b4():
    # absmax 7 -> s = 7/7 = 1 exactly; x/s = x; ties go to the even integer.
    q, s = quant.quantize(h(7, 3.5, -3.5, 0.5, -0.5, 1.5, 2.5, -2.5), 4, axis=0)
    assert float(s) == 1.0
    assert q.tolist() == [7, 4, -4, 0, 0, 2, 2, -2]


def test_rne_ties_b2_b8():
    q, s = quant.quantize(h(1, 0.5, -0.5, -1, 0.75), 2, axis=0)
    assert float(s) == 1.0 and q.tolist() == [1, 0, 0, -1, 1]
    q, s = quant.quantize(h(127, 63.5, 64.5, -0.5, -126.5), 8, axis=0)
    assert float(s) == 1.0 and q.tolist() == [127, 64, 64, 0, -126]


def test_scale_rounding_one_seventh():
    # 1/7 = 1.142857 * 2^-3; mantissa 0.142857*1024 = 146.29 -> 146 -> fp16 bits 0x3092
    # = 0.142822265625.  1/0.142822265625 = 7.0017 -> 7.  dequant = 7*0.142822265625.
    q, s = quant.quantize(h(1.0, -0.5), 4, axis=0)
    assert np.asarray(s, dtype=F16).view(np.uint16) == 0x3092
    assert q.tolist() == [7, -4]   # -0.5/0.1428 = -3.5009 -> -4
    xh = quant.dequantize(q, s, axis=0)
    assert xh.tolist() == [np.float32(7 * 0.142822265625), np.float32(-4 * 0.142822265625)]


def test_clamp_with_subnormal_scale():
    # fp16(1e-4) = (1 + 654/1024) * 2^-14; /127 = 7.875e-7 = 13.21 * 2^-24 -> s = 13 * 2^-24
    # (subnormal, rounded down by 1.6%) so x/s = 129.08 -> 129 -> clamped to 127.
    q, s = quant.quantize(h(1e-4), 8, axis=0)
    assert np.asarray(s, dtype=F16).view(np.uint16) == 13
    assert q.tolist() == [127]


def test_zero_and_underflow_groups():
    q, s = quant.quantize(h(0, 0, -0.0), 4, axis=0)
    assert float(s) == 0.0 and q.tolist() == [0, 0, 0]
    # absmax 2^-24 (smallest subnormal): 2^-24/127 rounds to fp16 zero -> all codes 0
    tiny = np.array([1], dtype=np.uint16).view(F16)
    q, s = quant.quantize(np.concatenate([tiny, -tiny]), 8, axis=0)
    assert float(s) == 0.0 and q.tolist() == [0, 0]


def _struct_scale(m: float, b: int) -> float:
    qm = (1 << (b - 1)) - 1
    s32 = struct.unpack("<f", struct.pack("<f", m / qm))[0]
    return struct.unpack("<e", struct.pack("<e", s32))[0]


def _brute_q(x: float, s: float, b: int) -> int:
    qm = (1 << (b - 1)) - 1
    if s == 0.0:
        return 0
    best = None
    for c in range(-qm, qm + 1):
        e = abs(x - c * s)
        if best is None or e < best[0] or (e == best[0] and c % 2 == 0):
            best = (e, c)
    return best[1]


@pytest.mark.parametrize("b", [2, 4, 8])
def test_brute_force_against_definition(b):
    # groups of 16 fp16 values: N(0,1), an x10 outlier, tiny magnitudes (subnormal scales)
    z = synth.draw16(7, 99, synth.T_K, b, [0], [0], 60, 1, 16)[0, :, 0].numpy()
    groups = [z[i] for i in range(40)]
    groups += [(z[i].astype(np.float32) * 10).astype(F16) for i in range(40, 50)]
    groups += [(z[i].astype(np.float32) * 2e-5).astype(F16) for i in range(50, 60)]
    for g in groups:
        q, s = quant.quantize(g, b, axis=0)
        m = float(np.max(np.abs(g.astype(np.float64))))
        assert float(s) == _struct_scale(m, b)
        for xi, qi in zip(g.astype(np.float64), q.tolist()):
            assert qi == _brute_q(xi, float(s), b)


@pytest.mark.parametrize("b", [2, 4, 8])
def test_round_trip_bound(b):
    # |x - q s| <= s/2 where not clamped; with clamping, <= s/2 + |absmax - qmax s|
    z = synth.draw16(3, 98, synth.T_V, 0, [0], [0], 200, 1, 64)[0, :, 0].numpy()
    q, s = quant.quantize(z, b, axis=1)
    xh = quant.dequantize(q, s, axis=1).astype(np.float64)
    x = z.astype(np.float64)
    sf = s.astype(np.float64)[:, None]
    m = np.abs(x).max(axis=1, keepdims=True)
    bound = sf / 2 + np.abs(m - ((1 << (b - 1)) - 1) * sf)
    assert np.all(np.abs(x - xh) <= bound + 1e-12)
    assert np.all(np.abs(q) <= (1 << (b - 1)) - 1)


def test_pack_hand_bytes():
    # INT4: q [-7, 7, 0, 1] -> u [1, 15, 8, 9] -> bytes 0xF1, 0x98 (LSB first)
    assert quant.pack(np.array([-7, 7, 0, 1]), 4).tolist() == [0xF1, 0x98]
    # INT2: q [-1, 0, 1, 0] -> u [1, 2, 3, 2] -> 1 | 2<<2 | 3<<4 | 2<<6 = 0xB9
    assert quant.pack(np.array([-1, 0, 1, 0]), 2).tolist() == [0xB9]
    # INT8: offset binary 128
    assert quant.pack(np.array([-127, 0, 127, -1]), 8).tolist() == [0x01, 0x80, 0xFF, 0x7F]


@pytest.mark.parametrize("b", [2, 4, 8])
def test_pack_round_trip(b):
    rng = np.random.default_rng(b)
    qm = (1 << (b - 1)) - 1
    q = rng.integers(-qm, qm + 1, size=(5, 3, 128))
    assert np.array_equal(quant.unpack(quant.pack(q, b), b, 128), q)


def test_generator_cpu_batched_matches_single():
    a = synth.draw16(0, 1, synth.T_K, 3, [0, 5], [10, 20], 7, 2, 64)
    b0 = synth.draw16(0, 1, synth.T_K, 3, [0], [10], 7, 2, 64)
    b1 = synth.draw16(0, 1, synth.T_K, 3, [5], [23], 4, 2, 64)
    assert torch.equal(a[0], b0[0])
    assert torch.equal(a[1, 3:], b1[0])

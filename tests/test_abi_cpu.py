"""The C-ABI library builds for sm_103a, loads, and exports every symbol
include/ekv.h declares; host-only entry points agree with the oracle's byte
accounting.  No GPU needed (no compute call is made)."""
import os
import re
import shutil

import pytest

from conftest import ROOT
from oracle import pages

HEADER = os.path.join(ROOT, "include", "ekv.h")


def declared_symbols():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"EKV_API\s+[\w\s\*]+?\b(ekv_\w+)\s*\(", txt)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("no CUDA toolkit on this host")
    from mixed_precision_quantized_gb300 import build, ekv
    build.build()
    return ekv.lib()


def test_header_declares_the_hot_path():
    syms = declared_symbols()
    for s in ("ekv_append", "ekv_decode_attn", "ekv_canary_kl", "ekv_tier_update",
              "ekv_block_table", "ekv_create", "ekv_destroy", "ekv_sync"):
        assert s in syms


def test_every_declared_symbol_is_exported(lib):
    from mixed_precision_quantized_gb300 import ekv
    for s in declared_symbols():
        assert hasattr(lib, s), s
    assert sorted(ekv.EXPORTS) == declared_symbols()


def test_page_bytes_matches_oracle_layout(lib):
    for kb in (2, 4, 8, 16):
        for vb in (2, 4, 8, 16):
            for d in (64, 128):
                assert lib.ekv_page_bytes(kb, vb, d) == pages.page_bytes(kb, vb, d)
    assert lib.ekv_page_bytes(3, 4, 128) == -1
    assert lib.ekv_page_bytes(4, 4, 96) == -1
    for kb in (2, 4, 8, 16):
        for vb in (2, 4, 8, 16):
            for d in (64, 128):
                assert lib.ekv_page_bytes_q(kb, vb, d, 1) == pages.page_bytes(kb, vb, d, asym=True)
                assert lib.ekv_page_bytes_q(kb, vb, d, 0) == pages.page_bytes(kb, vb, d)
    assert lib.ekv_page_bytes_q(4, 4, 128, 2) == -1


def test_status_strings(lib):
    for code in range(7):
        assert lib.ekv_status_string(code)
    assert lib.ekv_status_string(99) == b"unknown status"


def test_create_rejects_bad_config_without_gpu(lib):
    import ctypes
    from mixed_precision_quantized_gb300 import ekv
    cfg = ekv.EkvConfig()
    cfg.num_layers = 0
    h = ctypes.c_void_p()
    kb = (ctypes.c_uint8 * 1)(4)
    assert lib.ekv_create(ctypes.byref(cfg), kb, kb, ctypes.byref(h)) == 1   # EINVAL
    assert lib.ekv_create(None, kb, kb, ctypes.byref(h)) == 1


def test_autok_host_allocator_matches_oracle(lib):
    """AutoK runs on the host: the library's order and count equal the oracle's."""
    import numpy as np
    from mixed_precision_quantized_gb300 import ekv
    from oracle import artifacts
    rng = np.random.default_rng(17)
    for _ in range(300):
        L = int(rng.integers(0, 40))
        s = rng.random(L) ** 3
        s[rng.random(L) < 0.2] = 0.0
        s[rng.random(L) < 0.2] = s[0] if L else 0.0          # equal values: order by layer
        frac = float(rng.choice([0.0, 0.3, 0.5, 0.9, 0.99, 1.0, rng.random()]))
        k, order = ekv.autok(s.tolist(), frac)
        assert order == artifacts.sensitivity_order(s)
        assert k == artifacts.autok(s, frac)
    for bad_s, bad_f in (([1.0, -1.0], 0.5), ([float("nan")], 0.5), ([float("inf")], 0.5),
                         ([1.0], 1.01), ([1.0], -0.5)):
        with pytest.raises(ekv.EkvError):
            ekv.autok(bad_s, bad_f)


def test_artifact_save_load_round_trip(tmp_path):
    """The static-artifact bundle survives a save and comes back read-only."""
    import numpy as np
    from mixed_precision_quantized_gb300 import artifacts as product
    a = product.Artifact([4, 8, 4], [4, 8, 16], np.arange(3 * 2 * 64, dtype=np.float32).reshape(3, 2, 64) + 1,
                         np.array([[1, np.inf], [2, 3], [4, 5]], np.float32), [1.0, 0.99, 0.9],
                         [1.0, 1.0, 0.99], [0.1, 0.3, 0.2], 0.5, 4, 8)
    p = tmp_path / "a.npz"
    a.save(p)
    b = product.Artifact.load(p)
    assert (b.k_bits, b.v_bits, b.k_percentile, b.v_percentile, b.sensitivity, b.frac, b.low,
            b.high) == (a.k_bits, a.v_bits, a.k_percentile, a.v_percentile, a.sensitivity,
                        a.frac, a.low, a.high)
    assert np.array_equal(b.k_clip, a.k_clip) and np.array_equal(b.v_clip, a.v_clip)
    assert not b.v_clip.flags.writeable

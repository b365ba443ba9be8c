"""bench.py's host-side pieces that run without a GPU: the reference arm (the
oracle timed on the host cores, printing the same JSON line as the GPU arm)
and the canary amortization of a timed region."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "1"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600, env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["steps"] == 2 and d["warmup"] == 1
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert "2 of 2 layers" in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


@pytest.mark.parametrize("fired, steps, period, want", [
    (1, 64, 64, 1.0),      # one firing held, one firing's share: unchanged
    (0, 64, 64, 1.1),      # none held: one firing added
    (1, 8, 64, 0.9125),    # one held in 8 steps: 1/8 of a firing kept
    (2, 128, 64, 1.0),
    (1, 64, 0, 1.0),       # no canary: unchanged
])
def test_amortized_region(fired, steps, period, want):
    assert bench.amortized_region(1.0, fired, 0.1, steps, period) == pytest.approx(want)


def test_reference_arm_under_torchrun_prints_once():
    """Launched as two ranks (gloo on the host), rank 0 alone times the oracle and
    prints the line; the other rank exits 0 without work."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                        "--master-port", str(port), "bench.py", "--impl", "reference",
                        "--gpus", "2", "--workload", "tiny", "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0


def test_traffic_field_only_for_the_captured_kernel_and_step(monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_SOURCE_SHA", bench.attn_source_sha())
    assert bench.traffic_field("llama70b_128k", True, True, False, False)[0] == bench.TRAFFIC_BYTES
    for args in (("qwen14b_32k", True, True, False, False),
                 ("llama70b_128k", False, True, False, False),   # --layers
                 ("llama70b_128k", True, False, False, False),   # separate calls
                 ("llama70b_128k", True, True, True, False),     # asymmetric pages
                 ("llama70b_128k", True, True, False, True)):    # static artifact
        value, note = bench.traffic_field(*args)
        assert value is None and note
    monkeypatch.setattr(bench, "TRAFFIC_SOURCE_SHA", "0" * 16)
    value, note = bench.traffic_field("llama70b_128k", True, True, False, False)
    assert value is None and "0" * 16 in note and bench.attn_source_sha() in note

"""Decode-step benchmark of the mixed-precision quantized KV-cache path on GB300.

One step = one decode token for every sequence through every layer: per layer
append (ring write, V quantization, K staging/seal, page admission at the
layer's tier) and decode attention over the whole cache, as one fused launch
(`--separate`: two launches); on every 64th step the canary runs for every
layer and the controller updates the tiers.

Default workload: Llama-3.1-70B shape, 80 layers, batch 1, 64 q / 8 kv heads,
head_dim 128, 131072 cached tokens, K starting at INT4 with the canary every 64
steps (tau 0.05, alpha 0.25), V INT4; synthetic N(0,1) inputs with one K
outlier channel (x10) per head and K gain 1 + 0.05 * layer.  A step reads
~12.3 GB of pages, far above the 129 MB L2, so no L2 flush is needed.

Timed regions (all on one stream, CUDA events, synchronize + barrier on both
sides, max over ranks):
  A  K steps replayed as one CUDA graph                  -> value, ms_per_step
  B  the next K steps, each attention launch (fused: append + attention)
     bracketed by timing events inside the graph         -> roofline (attention)
  E  the next K steps with a pinned-host -> device copy of the step's inputs
     and a device -> pinned-host copy of every layer's output per step -> e2e
The canary cost is timed separately (every layer's canary in one launch + one
controller update, replayed as a graph) -> canary_us_per_firing.

`--impl reference` times the CPU oracle on the same workload on a bounded
sample (a few layers of one decode step), on rank 0 only.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized-KV decode attn HBM GB/s (% of peak), tokens/s; canary µs/firing"
L2_BYTES = 129 * 2 ** 20        # GB300 L2

# DRAM bytes (read + write) per decode-attention launch from one ncu capture of
# the 2-layer case of the 70B workload (the same per-launch work as one layer of
# the full workload), valid only for the kernel source it was taken on: any
# change to that source reports null until re-captured.
TRAFFIC_BYTES = 157.13e6
TRAFFIC_SOURCE_SHA = "f1986ffba0a2f29a"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=64)
    p.add_argument("--warmup", type=int, default=4)
    p.add_argument("--impl", default="ekv", choices=["ekv", "reference"])
    p.add_argument("--workload", default="llama70b_128k")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-sample-layers", type=int, default=2)
    p.add_argument("--layers", type=int, default=0,
                   help="run only the first N layers of the workload (profiling cases)")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    p.add_argument("--rotate", type=int, default=1,
                   help="rotate steps over N caches of the workload, so that a workload whose "
                        "pages fit in L2 is still read from HBM")
    p.add_argument("--no-overlap-check", action="store_true",
                   help="skip timing the fused step without the overlap of consecutive layers")
    p.add_argument("--static", action="store_true",
                   help="static-artifact mode: calibrate thresholds and per-layer K bits on "
                        "the workload's first --calib-tokens prefill tokens, load them, and "
                        "time the same step with the canary off")
    p.add_argument("--calib-tokens", type=int, default=8192)
    p.add_argument("--tau-ctx0", type=int, default=0,
                   help="controller budget tau * sqrt(L / tau_ctx0) (0: plain tau)")
    p.add_argument("--hysteresis", type=float, default=0.0, help="controller demotion margin")
    p.add_argument("--vote", type=int, default=1, help="consecutive firings a tier change needs")
    p.add_argument("--asym", action="store_true",
                   help="KIVI-style asymmetric quantizer for the pages and the canary")
    p.add_argument("--separate", action="store_true",
                   help="append and attention as two launches per layer (default: one fused launch)")
    p.add_argument("--split", default="batch", choices=["batch", "heads"],
                   help="several GPUs: each holds its own sequences (batch, weak scaling) or "
                        "a share of every sequence's KV heads (heads, strong scaling)")
    p.add_argument("--overlap", default="dependent", choices=["dependent", "independent", "none"],
                   help="how each timed step's fused launches overlap (region A): starting while "
                        "the previous launch ends and reading q, k, v after it (dependent, as in "
                        "a model), reading them before it too (independent), or not at all")
    p.add_argument("--no-short", action="store_true",
                   help="skip the extra 32K-context figure (Qwen2.5-14B shape) of the default run")
    p.add_argument("--context", type=int, default=0,
                   help="cached tokens per sequence before the timed steps (0: the workload's)")
    p.add_argument("--force-kbits", type=int, default=0,
                   help="create the cache with every layer at this K width and keep the canary "
                        "off (per-width measurement at the workload's context)")
    return p.parse_args()


def attn_source_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ("ekv_attn.cu", "ekv_attn_body.cuh", "ekv_internal.h", "ekv_quant.cuh"):
        with open(os.path.join(ROOT, "mixed_precision_quantized_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class Clocks:
    """nvidia-smi sampling during a timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        time.sleep(1.0)
        return self

    def __exit__(self, *a):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()

    def summary(self):
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def hold_gpu(us: float = 200.0) -> None:
    """Queue a short device-side sleep on the current stream right before a timed
    region's start event, so the region's work is already submitted when the
    event fires and host submission latency stays out of the device timing."""
    import torch
    torch.cuda._sleep(int(us * 2e3))  # ~2 GHz SM clock: cycles for `us` microseconds


def graph_upload(g, stream) -> bool:
    """Upload a captured graph to the device before it is timed (cuGraphUpload),
    so its first replay does not pay the upload; False when this torch does not
    expose the executable graph."""
    import ctypes
    get = getattr(g, "raw_cuda_graph_exec", None)
    if get is None:
        return False
    try:
        handle = get()
        cu = ctypes.CDLL("libcuda.so.1")
        cu.cuGraphUpload.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        ok = cu.cuGraphUpload(ctypes.c_void_p(int(handle)), ctypes.c_void_p(stream.cuda_stream)) == 0
        stream.synchronize()
        return ok
    except Exception:  # noqa: BLE001
        return False


def attn_bytes_per_layer(cache, w, layer: int) -> float:
    """Algorithmic bytes one decode-attention launch reads and writes for a layer."""
    from mixed_precision_quantized_gb300 import ekv
    d, Hkv, Hq = w.head_dim, w.num_kv_heads, w.num_q_heads
    vb = w.v_bits[layer]
    total = 0.0
    for s in range(w.batch):
        T = cache.seq_len(layer, s)
        nopen = T % 16
        for h in range(Hkv):
            bt = cache.block_table(layer, s, h)
            for j, e in enumerate(bt):
                fmt = (e >> 28) & 15
                kb = 2 << (fmt >> 2)
                if nopen and j == len(bt) - 1:
                    vrow = d * 2 if vb == 16 else d * vb // 8 + (4 if w.asym else 2)
                    total += nopen * (2 * d + vrow)       # open rows: fp16 K + V row
                else:
                    total += ekv.page_bytes(kb, vb, d, w.asym)
                total += 4                                  # page-table entry
        total += 2 * Hq * d * 2                             # Q in, O out
    return total


def cpu_baseline(w, sample_layers: int, device, steps: int = 1, warmup: int = 1):
    """Time the oracle (as it stands) on a bounded sample of the decode steps:
    `warmup` untimed then `steps` timed steps over the first `sample_layers`
    layers (append + attention of every sequence and head), scaled to all
    layers."""
    import numpy as np  # noqa: F401
    from oracle import decoder
    layers = list(range(min(sample_layers, w.num_layers)))
    if warmup + steps > w.steps:
        raise SystemExit(f"workload holds {w.steps} decode steps; asked for {warmup + steps}")
    tr = decoder.Trace()
    tr.tiers = [list(w.k_bits_init)] * (w.steps + 1)
    ref = decoder.ReferenceRun(w, tr, layers=layers, device=device)
    ref.prefill()

    def step():
        ref.advance()
        for l in layers:
            for s in ref.seqs:
                ref.attend(l, s)

    for _ in range(max(1, warmup)):    # untimed (the first fills the sealed-block memo)
        step()
    c0, t0 = time.process_time(), time.perf_counter()
    for _ in range(steps):
        step()
    wall = time.perf_counter() - t0
    cpu = time.process_time() - c0
    per_step = wall / steps * w.num_layers / len(layers)
    return {"value": w.batch / per_step, "unit": "tokens/s",
            "cores": round(max(1.0, cpu / wall), 1), "kind": "oracle",
            "sample": f"{len(layers)} of {w.num_layers} layers of {steps} decode step(s) at the "
                      f"full context after {max(1, warmup)} untimed, all {w.batch} sequence(s) "
                      f"and heads; per-step time scaled by {w.num_layers / len(layers):g}; "
                      f"wall {wall:.2f} s",
            "ms_per_step": 1e3 * per_step, "steps": steps, "warmup": max(1, warmup),
            "host": os.uname().machine, "nproc": os.cpu_count()}


def traffic_field(workload_name: str, full_size: bool, fused: bool, asym: bool,
                  static: bool) -> tuple:
    """(DRAM bytes per launch, note): the captured figure when this run is the
    captured configuration on the captured kernel source, else None and why."""
    if not (workload_name == "llama70b_128k" and full_size and fused and not asym
            and not static):
        return None, "captured for the default 70B/128K fused step only"
    if attn_source_sha() != TRAFFIC_SOURCE_SHA:
        return None, (f"the last capture ({TRAFFIC_BYTES / 1e6:.1f} MB per launch) was taken "
                      f"on kernel source {TRAFFIC_SOURCE_SHA}, not on this one "
                      f"({attn_source_sha()})")
    return TRAFFIC_BYTES, "dram__bytes_read.sum + dram__bytes_write.sum of one ncu capture"


def amortized_region(t_region: float, fired: int, canary_s: float, steps: int,
                     period: int) -> float:
    """A timed region's time with the canary at its 1-in-`period` share: the
    firings it happened to hold replaced by steps / period firings."""
    if not period:
        return t_region
    return t_region - fired * canary_s + steps / period * canary_s


def short_context_figure(dev, K: int = 16, W: int = 3) -> dict:
    """The fused decode step at 32K context (Qwen2.5-14B shape: 48 layers, 40 q /
    8 kv heads, K 2/4/8 mixed, V4): per-launch time and HBM fraction with and
    without the overlap of consecutive layers, CUDA-graph replay, events on the
    launching stream."""
    import torch
    from mixed_precision_quantized_gb300 import ekv, runner, workloads
    w = workloads.qwen14b_32k()
    L = w.num_layers
    slots = torch.arange(w.batch, dtype=torch.int32, device=dev)
    cache = ekv.cache_for(w, device=dev)
    runner.prefill(cache, w, slots, device=dev)
    inp = runner.Inputs(w, 0, W + 2 * K, device=dev)
    outs = [torch.empty(w.batch, w.num_q_heads, w.head_dim, dtype=torch.float16, device=dev)
            for _ in range(L)]
    for i in range(W):
        runner.decode_step(cache, w, slots, inp, i, outs, False, fused=True)
    cache.sync()
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    res = {}
    for name, first, overlap in (("overlap", W, "dependent"), ("no_overlap", W + K, False)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(first, first + K):
                runner.decode_step(cache, w, slots, inp, i, outs, False, fused=True,
                                   overlap=overlap)
        graph_upload(g, stream)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            hold_gpu()
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        cache.sync()
        res[name] = e0.elapsed_time(e1) / 1e3
        del g
    nbytes = sum(attn_bytes_per_layer(cache, w, l) for l in range(L)) / L
    peak, _ = peaks()
    cache.close()
    out = {"workload": f"{w.name}: {L} layers, batch 1, {w.num_q_heads} q / {w.num_kv_heads} kv "
                       f"heads, d {w.head_dim}, {w.prefill[0]} cached tokens, K 2/4/8 mixed "
                       f"per layer, V INT4, fused step, {K} steps",
           "bytes_per_launch": nbytes}
    for name, t in res.items():
        us = t / (K * L) * 1e6
        out[name] = {"tokens_s": K * w.batch / t, "avg_launch_us": us,
                     "achieved_gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak}
    return out


def main():
    a = parse()
    import torch
    import torch.distributed as dist

    from mixed_precision_quantized_gb300 import replicas, workloads

    R = replicas.from_env()
    world, rank, local = R.world, R.rank, R.local
    if world > 1:
        dist.init_process_group("nccl" if a.impl == "ekv" else "gloo")

    heads = a.split == "heads" and world > 1
    w = (replicas.head_shard(workloads.by_name(a.workload), rank, world) if heads
         else replicas.shard(workloads.by_name(a.workload), rank))
    # tokens/s over the job: every rank's own sequences (batch split), or the
    # same sequences' tokens once (head split: the ranks share each token)
    rate = (lambda units, t: units / t) if heads else (
        lambda units, t: replicas.whole_job_rate(R, units, t))
    if a.layers:
        w = w.scaled(num_layers=a.layers)
    if a.force_kbits:
        w = w.scaled(k_bits_init=[a.force_kbits] * w.num_layers, canary_period=0,
                     name=f"{w.name}_k{a.force_kbits}")
    if a.context:
        w = w.scaled(prefill=[a.context] * w.batch, name=f"{w.name}_ctx{a.context}")
    if a.asym:
        if a.static:
            raise SystemExit("the static artifact's thresholds cap the symmetric quantizer")
        w = w.scaled(asym=True)

    if a.impl == "reference":
        if rank != 0:
            return
        dev = "cuda:0" if torch.cuda.is_available() else "cpu"
        cb = cpu_baseline(w, a.cpu_sample_layers, dev, steps=a.steps, warmup=a.warmup)
        line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "tokens/s",
                "n_gpus": 0, "steps": cb["steps"], "warmup": cb["warmup"],
                "ms_per_step": cb["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic",
                "config": {"workload": w.name}, "cpu_baseline": cb,
                "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    from mixed_precision_quantized_gb300 import build, ekv, runner

    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    K, W = a.steps, a.warmup
    fused = not a.separate
    if W < 3:
        raise SystemExit("at least 3 warm-up steps")
    n_steps_total = W + (3 if not a.no_e2e else 2) * K + (2 * K if not a.no_overlap_check else 0)
    if n_steps_total > w.steps:
        raise SystemExit(f"workload holds {w.steps} decode steps; asked for {n_steps_total}")
    # Region F: `period` steps that hold exactly one canary firing (the first
    # firing step after the other regions), timed like region A.
    P = w.canary_period
    sF = -(-n_steps_total // P) * P if P else None
    if sF is not None and sF + P > w.steps:
        sF = None

    static = None
    if a.static:
        from mixed_precision_quantized_gb300 import artifacts
        wc = w.scaled(prefill=[min(t, a.calib_tokens) for t in w.prefill])
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        # one model-level artifact: rank 0 calibrates, every rank loads its copy
        art = artifacts.calibrate(wc, device=dev)[0] if rank == 0 else None
        torch.cuda.synchronize()
        cal_s = time.perf_counter() - t0
        art = replicas.share_artifact(R, art)
        # the percentile select on one layer's full prefill keys and values
        kf, vf = w.prefill_kv(0, list(range(w.batch)), device=dev)
        kf, vf = kf.flatten(0, 1).contiguous(), vf.flatten(0, 1).contiguous()
        sel = {}
        for name, fn, x in (("k", ekv.k_thresholds, kf), ("v", ekv.v_thresholds, vf)):
            fn(x, 0.999)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(5):
                fn(x, 0.999)
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / 5
            sel[name] = {"us": us, "bytes_read": 2 * x.numel() * 2,
                         "gbs": 2 * x.numel() * 2 / (us * 1e-6) / 1e9}
        del kf, vf
        bits = {str(b): art.k_bits.count(b) for b in sorted(set(art.k_bits))}
        static = {"calibration_s": cal_s, "calibration_tokens_per_seq": wc.prefill[0],
                  "k_bits_layers": bits, "frac": art.frac, "low": art.low, "high": art.high,
                  "k_percentiles": sorted(set(art.k_percentile)),
                  "v_percentiles": sorted(set(art.v_percentile)),
                  "percentile_select": {**sel, "note": "two passes over the data (radix "
                                        "select): bytes_read counts both; one layer's "
                                        "full prefill"}}
        w = art.workload(w)

    NR = max(1, a.rotate)
    if K % NR:
        raise SystemExit("--steps must be a multiple of --rotate")
    if W < NR:
        raise SystemExit("--warmup must cover every rotated cache (>= --rotate)")
    # Timed steps must read from HBM: the caches the steps rotate over must hold
    # well over L2's worth of pages (estimate at the initial tiers).
    est = sum(-(-t // 16) * w.num_kv_heads * ekv.page_bytes(w.k_bits_init[l], w.v_bits[l],
                                                             w.head_dim, w.asym)
              for l in range(w.num_layers) for t in w.prefill)
    if NR * est < 1.5 * L2_BYTES:
        need = int(-(-1.5 * L2_BYTES // est))
        raise SystemExit(f"{NR} cache(s) of {est / 1e6:.1f} MB of pages are under 1.5 times "
                         f"the {L2_BYTES / 1e6:.0f} MB L2: use --rotate >= {need}")
    slots = torch.arange(w.batch, dtype=torch.int32, device=dev)
    caches = []
    t0 = time.perf_counter()
    for _ in range(NR):
        caches.append(ekv.cache_for(w, device=dev, tau_ctx0=a.tau_ctx0,
                                    hysteresis=a.hysteresis, vote=a.vote))
        if static is not None:
            art.apply(caches[-1])
        runner.prefill(caches[-1], w, slots, device=dev)
        caches[-1].sync()
    prefill_s = (time.perf_counter() - t0) / NR
    cache = caches[0]
    # Decode steps list the slots longest sequence first (a scheduler knows its
    # sequences' lengths): the kernel starts the CTAs of the listed sequences in
    # that order, so a ragged batch's long sequences do not end up in its last
    # wave.  Slot s holds sequence s; batch position i holds sequence order[i].
    order = sorted(range(w.batch), key=lambda s: (-w.prefill[s], s))
    slots = torch.tensor(order, dtype=torch.int32, device=dev)

    def C(i):  # the cache decode step i runs on
        return caches[i % NR]
    inp = runner.Inputs(w, 0, W + 2 * K, device=dev, order=order)
    L, B = w.num_layers, w.batch
    out = torch.empty(L, B, w.num_q_heads, w.head_dim, dtype=torch.float16, device=dev)
    outs = [out[l] for l in range(L)]

    # Several GPUs: each holds a shard of the batch; at a canary firing the ranks
    # combine their readings (all-reduce) before the identical tier update.
    combine, delta_buf = None, None
    if world > 1:
        import functools
        nq = B * w.num_q_heads
        delta_buf = torch.zeros(L, 3, dtype=torch.float32, device=dev)
        combine = functools.partial(replicas.combine_readings, R, n_queries=nq,
                                    total=replicas.total_queries(R, nq, dev))

    def canary(c, q_layers):  # every layer's canary in one launch; q_layers [L, B, Hq, d]
        c.canary_kl_layers(0, slots, q_layers, delta_buf)

    def fire_end(c, freeze=False):
        if combine is None:
            c.tier_update(freeze=freeze)
        else:
            combine(delta_buf)
            c.tier_update(delta_buf, freeze=freeze)

    ovA = {"dependent": "dependent", "independent": "independent", "none": False}[a.overlap]
    # warm-up (eager)
    for i in range(W):
        runner.decode_step(C(i), w, slots, inp, i, outs, w.fires(i), delta_out=delta_buf,
                           fused=fused, combine=combine, overlap=ovA)
    for c in caches:
        c.sync()

    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())

    uploaded = []

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        uploaded.append(graph_upload(g, stream))
        return g

    # ---- A: K steps as one graph -------------------------------------------------
    gA = capture(lambda: [runner.decode_step(C(i), w, slots, inp, i, outs, w.fires(i),
                                             delta_out=delta_buf, fused=fused, combine=combine,
                                             overlap=ovA)
                          for i in range(W, W + K)])
    per_layer = 1 if fused else 2
    launches = sum(per_layer * L + (2 if w.fires(i) else 0) for i in range(W, W + K))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    clk = Clocks(local).__enter__()
    replicas.barrier(R)
    with torch.cuda.stream(stream):
        hold_gpu()  # the GPU is busy while the host submits what follows
        ev0.record(stream)
        gA.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    replicas.barrier(R)
    tA = ev0.elapsed_time(ev1) / 1e3
    for c in caches:
        c.sync()
    fired_A = sum(1 for i in range(W, W + K) if w.fires(i))

    # ---- A', A'': the same steps without any overlap of consecutive launches, and
    # with each layer reading its inputs before the previous launch ends (valid
    # only for this workload's fresh-draw inputs)
    tA2 = tA3 = None
    if fused and not a.no_overlap_check:
        for which in ("none", "independent"):
            s2 = W + 2 * K + (0 if a.no_e2e else K) + (K if which == "independent" else 0)
            inpA2 = runner.Inputs(w, s2, K, device=dev, order=order)
            ov = False if which == "none" else "independent"
            gA2 = capture(lambda: [runner.decode_step(C(i), w, slots, inpA2, i - s2, outs,
                                                      w.fires(i), delta_out=delta_buf,
                                                      fused=True, combine=combine, overlap=ov)
                                   for i in range(s2, s2 + K)])
            torch.cuda.synchronize()
            replicas.barrier(R)
            with torch.cuda.stream(stream):
                f0, f1 = (torch.cuda.Event(enable_timing=True),
                          torch.cuda.Event(enable_timing=True))
                hold_gpu()  # the GPU is busy while the host submits what follows
                f0.record(stream)
                gA2.replay()
                f1.record(stream)
            torch.cuda.synchronize()
            replicas.barrier(R)
            t = replicas.max_over_ranks(R, f0.elapsed_time(f1) / 1e3, dev)
            if which == "none":
                tA2 = t
            else:
                tA3 = t
            for c in caches:
                c.sync()
            del gA2, inpA2

    # ---- B: next K steps, attention launches bracketed by timing events --------
    try:
        pairs = [(torch.cuda.Event(enable_timing=True, external=True),
                  torch.cuda.Event(enable_timing=True, external=True)) for _ in range(K * L)]
        external_ok = True
    except TypeError:
        pairs, external_ok = [], False

    def steps_with_events():
        for n, i in enumerate(range(W + K, W + 2 * K)):
            c = C(i)
            for l in range(L):
                q, k, v = inp.layer(l, i)
                if not fused:
                    c.append(l, slots, k, v)
                if external_ok:
                    pairs[n * L + l][0].record(stream)
                if fused:
                    c.append_decode_attn(l, slots, k, v, q, outs[l])
                else:
                    c.decode_attn(l, slots, q, outs[l])
                if external_ok:
                    pairs[n * L + l][1].record(stream)
            if w.fires(i):
                canary(c, inp.step_q(i))
                fire_end(c)

    gB = capture(steps_with_events)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        gB.replay()
    torch.cuda.synchronize()
    for c in caches:
        c.sync()
    attn_ms = [p[0].elapsed_time(p[1]) for p in pairs] if external_ok else []
    # algorithmic bytes per attention launch, at the state of region B's middle
    layer_bytes = [attn_bytes_per_layer(cache, w, l) for l in range(L)]
    bytes_per_launch = sum(layer_bytes) / L
    attn_avg_s = (sum(attn_ms) / len(attn_ms) / 1e3) if attn_ms else None

    # ---- canary: all layers + one controller update ----------------------------
    q_last = inp.step_q(W + 2 * K - 1)

    def firing():
        canary(cache, q_last)
        fire_end(cache, freeze=True)

    gC = capture(firing)
    reps = 20
    with torch.cuda.stream(stream):
        gC.replay()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_gpu()  # the GPU is busy while the host submits what follows
        c0.record(stream)
        for _ in range(reps):
            gC.replay()
        c1.record(stream)
    torch.cuda.synchronize()
    canary_us = c0.elapsed_time(c1) * 1e3 / reps
    # With the fused step, region A holds nothing but the L fused launches of each
    # step and its canary firings: their time, less the firings (timed just
    # above), over the K * L launches is the launch duration inside the step
    # (inter-launch gaps included).  Events around each launch (region B) add
    # their own gaps; that figure is kept beside it.
    bracketed_s = attn_avg_s
    if fused:
        attn_avg_s = (tA - fired_A * canary_us * 1e-6) / (K * L)

    # ---- attention alone, all layers back to back (read-only, replayable) ------
    def attn_only():
        for c in caches:
            for l in range(L):
                c.decode_attn(l, slots, q_last[l], outs[l])

    gD = capture(attn_only)
    with torch.cuda.stream(stream):
        gD.replay()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_gpu()  # the GPU is busy while the host submits what follows
        d0.record(stream)
        for _ in range(5):
            gD.replay()
        d1.record(stream)
    torch.cuda.synchronize()
    attn_only_us = d0.elapsed_time(d1) * 1e3 / (5 * L * NR)
    if attn_avg_s is None:
        attn_avg_s = attn_only_us * 1e-6

    # ---- E: end to end with host buffers ------------------------------------------
    e2e = None
    if not a.no_e2e:
        s0 = W + 2 * K
        inpE = runner.Inputs(w, s0, K, device=dev, order=order)
        per_step = [torch.cat([inpE.q[l][i].reshape(-1) for l in range(L)] +
                              [inpE.k[l][i].reshape(-1) for l in range(L)] +
                              [inpE.v[l][i].reshape(-1) for l in range(L)]) for i in range(K)]
        host_in = torch.stack(per_step).cpu().pin_memory()
        del per_step, inpE
        nq, nkv = B * w.num_q_heads * w.head_dim, B * w.num_kv_heads * w.head_dim
        # Double-buffered: step n+1's inputs are uploaded and step n's outputs
        # read back on a copy stream while step n computes; every step still
        # pays its own host copies.
        def views(buf):
            qa = buf[:L * nq].view(L, B, w.num_q_heads, w.head_dim)
            ks = [buf[L * nq + l * nkv:L * nq + (l + 1) * nkv]
                  .view(B, 1, w.num_kv_heads, w.head_dim) for l in range(L)]
            vs = [buf[L * (nq + nkv) + l * nkv:L * (nq + nkv) + (l + 1) * nkv]
                  .view(B, 1, w.num_kv_heads, w.head_dim) for l in range(L)]
            return qa, ks, vs

        dbufs = [torch.empty(host_in.shape[1], dtype=torch.float16, device=dev) for _ in range(2)]
        dviews = [views(b) for b in dbufs]
        obufs = [torch.empty_like(out) for _ in range(2)]
        host_out = torch.empty(K, *out.shape, dtype=torch.float16).pin_memory()
        cs = torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(K)]
        ev_done = [torch.cuda.Event() for _ in range(K)]
        ev_out = [torch.cuda.Event() for _ in range(K)]

        def e2e_steps():
            cs.wait_stream(stream)
            with torch.cuda.stream(cs):
                dbufs[0].copy_(host_in[0], non_blocking=True)
                ev_in[0].record(cs)
            for n in range(K):
                i, b = s0 + n, n % 2
                c = C(i)
                qa, ks, vs = dviews[b]
                stream.wait_event(ev_in[n])
                if n >= 2:
                    stream.wait_event(ev_out[n - 2])      # obufs[b] read back
                for l in range(L):
                    if fused:
                        # (a one-layer step's previous launch appends to this layer)
                        c.append_decode_attn(l, slots, ks[l], vs[l], qa[l], obufs[b][l],
                                             after_producer=ovA == "dependent" and L > 1,
                                             after_other_layer=ovA == "independent" and l > 0)
                    else:
                        c.append(l, slots, ks[l], vs[l])
                        c.decode_attn(l, slots, qa[l], obufs[b][l])
                if w.fires(i):
                    canary(c, qa)
                    fire_end(c)
                ev_done[n].record(stream)
                with torch.cuda.stream(cs):
                    if n + 1 < K:
                        if n >= 1:
                            cs.wait_event(ev_done[n - 1])  # dbufs[1 - b] consumed
                        dbufs[1 - b].copy_(host_in[n + 1], non_blocking=True)
                        ev_in[n + 1].record(cs)
                    cs.wait_event(ev_done[n])
                    host_out[n].copy_(obufs[b], non_blocking=True)
                    ev_out[n].record(cs)
            stream.wait_stream(cs)

        gE = capture(e2e_steps)
        torch.cuda.synchronize()
        replicas.barrier(R)
        with torch.cuda.stream(stream):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            hold_gpu()  # the GPU is busy while the host submits what follows
            e0.record(stream)
            gE.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        replicas.barrier(R)
        tE = e0.elapsed_time(e1) / 1e3
        for c in caches:
            c.sync()
        tE = replicas.max_over_ranks(R, tE, dev)
        e2e = {"value": rate(B * K, tE), "unit": "tokens/s",
               "h2d_bytes_per_step": int(host_in.shape[1] * 2),
               "d2h_bytes_per_step": int(out.numel() * 2)}

    # ---- F: one period of steps holding one canary firing ------------------------
    canary_in_loop = None
    if sF is not None:
        inpF = runner.Inputs(w, sF, P, device=dev, order=order)
        gF = capture(lambda: [runner.decode_step(C(i), w, slots, inpF, i - sF, outs, w.fires(i),
                                                 delta_out=delta_buf, fused=fused,
                                                 combine=combine, overlap=ovA)
                              for i in range(sF, sF + P)])
        torch.cuda.synchronize()
        replicas.barrier(R)
        with torch.cuda.stream(stream):
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            hold_gpu()  # the GPU is busy while the host submits what follows
            g0.record(stream)
            gF.replay()
            g1.record(stream)
        torch.cuda.synchronize()
        replicas.barrier(R)
        tF = replicas.max_over_ranks(R, g0.elapsed_time(g1) / 1e3, dev)
        for c in caches:
            c.sync()
        del gF, inpF
        fired_F = sum(1 for i in range(sF, sF + P) if w.fires(i))
        t_step_nofire = (tA - fired_A * canary_us * 1e-6) / K   # region A's steps, firings out
        canary_in_loop = {
            "steps": P, "first_step": sF, "firings": fired_F, "ms": 1e3 * tF,
            "ms_per_step": 1e3 * tF / P,
            "overhead_frac_measured": (tF - P * t_step_nofire) / (P * t_step_nofire),
            "overhead_frac_derived": canary_us * 1e-6 / P / t_step_nofire,
            "note": "region F (one period of steps with its one firing) against region A's "
                    "steps without firings; derived = standalone firing time / period / step"}

    precision = None
    try:
        st_ = cache.stats()
        precision = {"k_bits_per_element": st_["k_bits"], "v_bits_per_element": st_["v_bits"],
                     "avg_bits_per_element": (st_["k_bits"] + st_["v_bits"]) / 2,
                     "memory_saved_vs_fp16": st_["saved_vs_fp16"],
                     "code_bits_vs_c0": st_["cost_vs_c0"],
                     "page_bytes": st_["page_bytes"], "fp16_bytes": st_["fp16_bytes"],
                     "pages_by_k_bits": {str(2 << kc): sum(st_["sealed_pages"][kc * 4 + vc] +
                                                           st_["open_pages"][kc * 4 + vc]
                                                           for vc in range(4))
                                         for kc in range(4)
                                         if any(st_["sealed_pages"][kc * 4 + vc] +
                                                st_["open_pages"][kc * 4 + vc]
                                                for vc in range(4))},
                     "source": "ekv_stats over every layer of the first cache after the timed "
                               "regions"}
    except Exception as ex:  # noqa: BLE001
        precision = {"error": repr(ex)}

    clk.__exit__(None, None, None)
    tA_raw = replicas.max_over_ranks(R, tA, dev)
    # `value` carries the canary at its 1-in-period share whatever firings the
    # timed window happened to hold.
    tA = amortized_region(tA_raw, fired_A, canary_us * 1e-6, K, P)

    peak, peak_kind = peaks()
    achieved = bytes_per_launch / attn_avg_s / 1e9 if attn_avg_s else None
    step_bytes = sum(layer_bytes)
    traffic = traffic_field(w.name, not a.layers, fused, a.asym, bool(a.static))
    line = {
        "metric": METRIC,
        "value": rate(B * K, tA),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": 1e3 * tA / K,
        "higher_is_better": True,
        "scaling": "strong" if heads else "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.num_layers} layers, batch {B}, "
                               f"{w.num_q_heads} q / {w.num_kv_heads} kv heads, d {w.head_dim}, "
                               f"{w.prefill[0] if len(set(w.prefill)) == 1 else 'ragged'} cached "
                               + (f"tokens, K fixed at INT{a.force_kbits} (canary off), "
                                  if a.force_kbits else
                                  f"tokens, K tier by canary every {w.canary_period} steps "
                                  f"(tau {w.tau}), " if static is None else
                                  "tokens, K bits per layer from the static artifact, ")
                               + f"V INT{w.v_bits[0]}"
                               + (", KIVI-style asymmetric quantizer" if w.asym else ""),
                   "l2": (f"inputs larger than L2: {step_bytes / 1e9:.2f} GB of pages read per step"
                          if NR == 1 else
                          f"steps rotate over {NR} caches of {step_bytes / 1e9:.3f} GB of pages "
                          f"each ({NR * step_bytes / 1e6:.0f} MB, over 1.5 times the "
                          f"{L2_BYTES / 1e6:.0f} MB L2)"),
                   "parallelism": (f"KV heads split over {world} GPUs ({w.num_kv_heads} each)"
                                   if heads else
                                   f"replicas x{world} (one sequence set per GPU)"),
                   "graph": ("CUDA graph of the timed steps, uploaded before timing"
                             if uploaded and all(uploaded) else
                             "CUDA graph of the timed steps (first replay includes its upload)"),
                   "canary_fires_in_timed": fired_A,
                   "controller": {"tau_ctx0": a.tau_ctx0, "hysteresis": a.hysteresis,
                                  "vote": a.vote},
                   "step": ("one fused append + attention launch per layer" +
                            {"dependent": ", each starting while the previous launch ends and "
                                          "reading its q, k, v only after it (valid when they "
                                          "come from the previous layer's output, as in a "
                                          "model)",
                             "independent": ", each starting while the previous launch ends "
                                            "and reading its q, k, v before it (valid only for "
                                            "inputs independent of the previous layer)",
                             "none": ", each after the previous one"}[a.overlap] if fused
                            else "append and attention launches per layer")
                           + ("; static artifact: calibrated per-layer K bits and clipping "
                              "thresholds loaded, canary off" if static else "")},
        "static": static,
        "attn_hbm_gbs": achieved,
        "attn_frac_of_8tbs": achieved / NOMINAL_HBM_GBS if achieved else None,
        "step_hbm_gbs": step_bytes / (tA / K) / 1e9,
        "canary_us_per_firing": canary_us,
        "canary_overhead_frac_at_1_in_64": canary_us * 1e-6 / 64 / (tA / K),
        "prefill_s": prefill_s,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak if achieved else None,
                     "traffic": traffic[0],
                     "traffic_note": traffic[1],
                     "traffic_unit": "bytes per launch",
                     "kernel": ("decode_attn_kernel (fused append + attention)" if fused
                                else "decode_attn_kernel"), "peak_kind": peak_kind,
                     "bytes_per_launch": bytes_per_launch,
                     "avg_launch_us": attn_avg_s * 1e6 if attn_avg_s else None,
                     "launches_timed": K * L if fused else len(attn_ms),
                     "bracketed_launch_us": bracketed_s * 1e6 if bracketed_s else None,
                     "timing": ("timed region A (CUDA events around the K steps) less its "
                                "canary firings, per fused launch") if fused else
                               "events around each launch inside timed region B" if attn_ms
                               else "attention-only graph (all layers back to back)",
                     "attn_only_avg_us": attn_only_us},
        "e2e": e2e,
        "no_overlap": (None if tA2 is None else
                       {"value": rate(B * K, amortized_region(tA2, fired_A, canary_us * 1e-6,
                                                              K, P)),
                        "unit": "tokens/s",
                        "avg_launch_us": (tA2 - fired_A * canary_us * 1e-6) / (K * L) * 1e6,
                        "roofline_frac": (bytes_per_launch /
                                          ((tA2 - fired_A * canary_us * 1e-6) / (K * L)) / 1e9
                                          / peak),
                        "note": "same steps, each layer's launch waiting for the previous "
                                "one (inputs that depend on the previous layer's output); "
                                "canary at its 1-in-period share"}),
        "independent_inputs": (None if tA3 is None else
                               {"value": rate(B * K, amortized_region(tA3, fired_A,
                                                                       canary_us * 1e-6, K, P)),
                                "unit": "tokens/s",
                                "avg_launch_us": (tA3 - fired_A * canary_us * 1e-6) / (K * L)
                                * 1e6,
                                "roofline_frac": (bytes_per_launch /
                                                  ((tA3 - fired_A * canary_us * 1e-6) / (K * L))
                                                  / 1e9 / peak),
                                "note": "each layer's launch also reads its q, k, v before the "
                                        "previous layer's launch ends: valid for this "
                                        "workload's fresh-draw inputs only, not for a model"}),
        "canary_amortized": {"firings_in_region_A": fired_A,
                             "firings_counted": K / P if P else 0,
                             "value_before_amortizing": rate(B * K, tA_raw),
                             "note": "value and ms_per_step carry K/period canary firings "
                                     "(timed standalone) in place of those region A held"},
        "canary_in_loop": canary_in_loop,
        "precision": precision,
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if (rank == 0 and world == 1 and not a.no_short and not a.layers and not a.static
            and not a.asym and not a.force_kbits and w.name == "llama70b_128k"):
        for c in caches:
            c.close()
        caches = []
        try:
            line["ctx32k"] = short_context_figure(dev)
        except Exception as ex:  # noqa: BLE001
            line["ctx32k"] = {"error": repr(ex)}
    if rank == 0 and world == 1 and not a.no_cpu:
        try:
            line["cpu_baseline"] = cpu_baseline(w, a.cpu_sample_layers, dev)
        except Exception as ex:  # noqa: BLE001
            line["cpu_baseline"] = {"value": None, "error": repr(ex)}
    for c in caches:
        c.close()
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

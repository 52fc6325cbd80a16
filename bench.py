"""Backward-pass throughput of the GB300 FlashAttention library.

One step = one full backward (fa_bwd: D preprocess, key/value-major dK/dV
kernel, dQ step) over the causal bf16 workload B=1, H=32, N=8192, d=128, with
inputs resident in HBM. Throughput is counted as 10*N^2*d FLOPs per head,
halved under the causal mask, per step. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--dq deterministic|recompute|atomic|ordered]

Under torchrun each rank runs the same workload on its own GPU (independent
replicas: heads shard with no exchange, so there is no data-path collective);
value = units of all ranks / max-over-ranks time. ``--impl reference`` times
the float64 CPU oracle on the host cores (rank 0 only): W warm-up and K timed
steps, each the oracle backward of one head of the same workload, within a
few minutes.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from flashattention_backward_fa_gb300.inputs import HEADLINE, WORKLOADS, make_inputs  # noqa: E402

METRIC = "attn bwd TFLOP/s and % of dense bf16 peak (causal, d=128, N=8192), 1 GB300"
# --dq choices -> the `deterministic` argument of the backward (fa.h FA_DQ_*):
# the library's deterministic default, the query-major recompute, atomic and
# ordered accumulation.
DQ_MODES = {"deterministic": 1, "recompute": 2, "atomic": 0, "ordered": 3}
DQ_ALGOS = ("recompute", "atomic", "ordered")


def accumulates(mode: int) -> bool:
    """True for the dQ modes whose key/value-major kernel also forms dQ (5 contractions a pair)."""
    return mode in (0, 3)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def counted_flops(w) -> float:
    """10*N^2*d per head, halved under causal; windowed: 10*d per allowed pair."""
    if w.window > 0:
        W = min(w.window, w.N)
        # causal: keys (i - W, i]; without the causal mask the window is one-sided,
        # keys (i - W, N)
        pairs = (W * (W + 1) // 2 + (w.N - W) * W) if w.causal else sum(
            w.N - max(0, i - w.window + 1) for i in range(w.N))
        return 10.0 * w.d * pairs * w.B * w.H
    per_head = 10.0 * w.N * w.N * w.d
    return w.B * w.H * (per_head / 2 if w.causal else per_head)


def causal_pairs(w) -> float:
    return counted_flops(w) / (10.0 * w.d)


def dkdv_traffic(w, deterministic: bool):
    """DRAM bytes per launch of the key/value-major kernel from the committed ncu capture,
    scaled to this workload's head count; None unless the kernel source still matches
    the capture, and for workloads the capture does not cover: the atomic variant, or
    another dtype, length, head dimension or mask than its bf16 causal N=8192 d=128."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dkdv_traffic.json")
    if not deterministic or not os.path.exists(path):
        return None
    if (w.dtype, w.N, w.d, w.causal, w.window, w.dropout_p) != ("bf16", 8192, 128, True, 0, 0.0):
        return None
    with open(path) as f:
        rec = json.load(f)
    csrc = os.path.join(ROOT, "flashattention_backward_fa_gb300", "csrc")
    src = b"".join(open(os.path.join(csrc, n), "rb").read()
                   for n in ("kernels_bwd_kv.cu", "device_common.cuh", "fa_internal.h"))
    if hashlib.sha256(src).hexdigest() != rec["source_sha256"]:
        return None
    return rec["dram_bytes_per_launch_capture"] * (w.B * w.H) / rec["heads_in_capture"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in self.rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def flush_l2(buf: torch.Tensor):
    buf.add_(1)


def _gpu_busy(stream, ms: float = 2.0):
    """Keep the stream busy for about ``ms`` (a spin kernel) so that the host
    work of the launches enqueued after it (argument checks, pointer lookups,
    tensor-map encoding) happens while the GPU is still busy and stays outside
    the event intervals that follow."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(ms * 1e-3 * 2.0e9))


def time_stages(fa, q, k, v, o, do, lse, dq, dk, dv, ws, kw, deterministic, stream, steps):
    """Device time of each of the three backward stages, launched back to back
    on one stream behind a spin kernel, with an event between consecutive
    launches: each interval holds one kernel's execution and no host work."""
    stage_ms = [0.0, 0.0, 0.0]
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for _ in range(steps):
        _gpu_busy(stream)
        evs[0].record(stream)
        for s in range(3):
            fa.fa_bwd_stage(s, q, k, v, o, do, lse, dq, dk, dv, ws, **kw, deterministic=deterministic,
                            stream=stream)
            evs[s + 1].record(stream)
        torch.cuda.synchronize()
        for s in range(3):
            stage_ms[s] += evs[s].elapsed_time(evs[s + 1]) / steps
    return stage_ms


def time_workload(fa, w, steps=5, warmup=3):
    """Backward ms and TFLOP/s of one workload in both dQ modes (the per-workload
    block of the JSON line), plus the forward's ms. Inputs resident in HBM."""
    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v, do = (t.to(dev) for t in make_inputs(w))
    kw = dict(scale=w.scale, causal=w.causal, window=w.window, dropout_p=w.dropout_p, seed=w.philox_seed,
              offset=w.philox_offset)
    o, lse = fa.attention_forward(q, k, v, **kw)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.current_stream()
    flops = counted_flops(w)
    out = {"B": w.B, "H": w.H, "N": w.N, "d": w.d, "dtype": w.dtype, "causal": w.causal, "window": w.window,
           "dropout_p": w.dropout_p}
    modes = ("recompute",) if w.dtype == "f32" else DQ_ALGOS
    for name in modes:
        det = DQ_MODES[name]
        ws = fa.alloc_workspace(q, det)
        for _ in range(warmup):
            fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, **kw, deterministic=det, stream=stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _gpu_busy(stream, 5.0)  # covers the host's enqueue of all steps: device time per step
        e0.record(stream)
        for _ in range(steps):
            fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, **kw, deterministic=det, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        out[name] = {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12}
        del ws
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    for _ in range(warmup):
        fa.fa_fwd(q, k, v, o2, lse2, **kw, stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _gpu_busy(stream, 5.0)
    e0.record(stream)
    for _ in range(steps):
        fa.fa_fwd(q, k, v, o2, lse2, **kw, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    fms = e0.elapsed_time(e1) / steps
    out["forward"] = {"ms": fms, "tflops": 0.4 * flops / (fms * 1e-3) / 1e12}
    status = fa.fa_get_device_status(clear=True)
    if status:
        raise RuntimeError(f"device status {status} after timing {w.name}")
    return out


def time_ours(w, steps, warmup, deterministic, world):
    import flashattention_backward_fa_gb300 as fa
    fa.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v, do = (t.to(dev) for t in make_inputs(w))
    kw = dict(scale=w.scale, causal=w.causal, window=w.window, dropout_p=w.dropout_p, seed=w.philox_seed,
              offset=w.philox_offset)
    o, lse = fa.attention_forward(q, k, v, **kw)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = fa.alloc_workspace(q, deterministic)
    stream = torch.cuda.current_stream()

    def step():
        fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, **kw, deterministic=deterministic, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    # Inputs (5 x 64 MiB at the headline size) exceed the 129 MB L2, so consecutive
    # steps do not hit in L2 on their inputs.
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = ev0.elapsed_time(ev1) / steps
    # Per-stage durations (same stream), for the roofline of the dominant kernel.
    stage_ms = time_stages(fa, q, k, v, o, do, lse, dq, dk, dv, ws, kw, deterministic, stream, steps)
    sampler.stop()
    status = fa.fa_get_device_status(clear=True)
    if status:
        raise RuntimeError(f"device status {status} after the timed region")
    # e2e: the host-buffer entry point fa_bwd_host on pinned host tensors: every step
    # uploads the step's inputs, runs the backward and downloads the gradients
    # (the library overlaps the three over groups of heads).
    host_in = [t.cpu().pin_memory() for t in (q, k, v, o, do, lse)]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq, dk, dv)]
    staging = torch.empty(fa.fa_bwd_host_buffer_size(w.B, w.H, w.N, w.d, q.dtype, deterministic),
                          dtype=torch.uint8, device=dev)
    e2e_steps = max(1, min(steps, 5))
    fa.fa_bwd_host(*host_in, *host_out, staging, **kw, deterministic=deterministic, stream=stream)  # warm-up
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        fa.fa_bwd_host(*host_in, *host_out, staging, **kw, deterministic=deterministic, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    # The forward that produced O and L (support for the backward; not in `value`),
    # for the forward / backward speed ratio.
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    for _ in range(2):
        fa.fa_fwd(q, k, v, o2, lse2, **kw, stream=stream)
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(e2e_steps):
        fa.fa_fwd(q, k, v, o2, lse2, **kw, stream=stream)
    f1.record(stream)
    torch.cuda.synchronize()
    fwd_ms = f0.elapsed_time(f1) / e2e_steps
    # Every dQ algorithm on the same inputs (each with its own workspace), timed
    # the same way, so that one line reports all of them.
    mode_ms = {}
    for name in DQ_ALGOS:
        m = DQ_MODES[name]
        ws_m = fa.alloc_workspace(q, m)
        for _ in range(max(3, warmup)):
            fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws_m, **kw, deterministic=m, stream=stream)
        torch.cuda.synchronize()
        v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        v0.record(stream)
        for _ in range(steps):
            fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws_m, **kw, deterministic=m, stream=stream)
        v1.record(stream)
        torch.cuda.synchronize()
        mode_ms[name] = v0.elapsed_time(v1) / steps
        del ws_m
    status = fa.fa_get_device_status(clear=True)
    if status:
        raise RuntimeError(f"device status {status} after timing the dQ modes")
    return dict(ms=ms, stage_ms=stage_ms, clocks=sampler.summary(), e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, fwd_ms=fwd_ms,
                mode_ms=mode_ms)


def run_reference_steps(w, steps, warmup, budget_s=150.0):
    """The reference arm: the float64 oracle's backward of one head per step.

    W untimed warm-up steps, then K timed steps, each the oracle backward of the
    same single-head sample of the workload. If one head is so slow that K + W
    steps would not fit in about budget_s seconds, fewer steps run (at least one
    warm-up and one timed step) and the sample text says how many.
    Returns (TFLOP/s, sample text, cores, seconds per head).
    """
    import numpy as np

    import oracle
    q, k, v, do = make_inputs(w.with_(B=1, H=1))
    q, k, v, do = (t.float().numpy() for t in (q, k, v, do))
    args = (w.scale, w.causal, w.window, w.dropout_p, w.philox_seed, w.philox_offset)
    O, L = oracle.forward(q, k, v, *args)

    def step():
        oracle.backward(q, k, v, O, do, L, *args)

    t0 = time.perf_counter()
    step()                                   # first warm-up step, also sizes the run
    t_head = time.perf_counter() - t0
    fit = max(2, int(budget_s / max(t_head, 1e-9)))
    w_rest = min(max(warmup - 1, 0), fit // 4)
    k_run = max(1, min(steps, fit - 1 - w_rest))
    for _ in range(w_rest):
        step()
    t0 = time.perf_counter()
    for _ in range(k_run):
        step()
    el = time.perf_counter() - t0
    flops = counted_flops(w.with_(B=1, H=1)) * k_run
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = (f"{k_run} timed step(s) after {1 + w_rest} warm-up step(s); each step is the float64 oracle "
              f"backward of one head (B=1,H=1,N={w.N},d={w.d}) of the workload, numpy/OpenBLAS")
    del np
    return flops / el / 1e12, sample, cores, el / k_run


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--dq", default="deterministic", choices=sorted(DQ_MODES))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the per-workload block")
    ap.add_argument("--shape", default=None, help="B,H,N override (smaller cases for profiler captures)")
    ap.add_argument("--profile", action="store_true",
                    help="forward, then --warmup + 1 backward steps, no timing (for ncu captures)")
    a = ap.parse_args()
    w = WORKLOADS[a.workload]
    if a.shape:
        B, H, N = (int(x) for x in a.shape.split(","))
        w = w.with_(B=B, H=H, N=N, name=f"{w.name}@B{B}H{H}N{N}")
    if a.profile:
        import flashattention_backward_fa_gb300 as fa
        q, k, v, do = (t.cuda() for t in make_inputs(w))
        kw = dict(scale=w.scale, causal=w.causal, window=w.window, dropout_p=w.dropout_p, seed=w.philox_seed,
                  offset=w.philox_offset)
        o, lse = fa.attention_forward(q, k, v, **kw)
        for _ in range(a.warmup + 1):
            fa.attention_backward(q, k, v, o, do, lse, **kw, deterministic=DQ_MODES[a.dq])
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": w.name, "status": fa.fa_get_device_status(clear=True)}))
        return
    world, rank, _ = dist_setup()
    peaks, peak_src = load_peaks()
    config = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
              "window": w.window, "dropout_p": w.dropout_p, "dq_mode": a.dq,
              "l2": "inputs larger than L2 (5 x 64 MiB at the headline size), no flush"}
    if a.impl == "reference":
        if rank != 0:
            return
        tf, sample, cores, sec_per_head = run_reference_steps(w, a.steps, a.warmup)
        # Each timed step is one head of the workload (the oracle needs about a
        # second per head at N = 8192): ms_per_step is that measured time, and
        # config says how much of the workload a step covers.
        ref_config = dict(config, reference_step=f"one head (B=1, H=1) of the {w.B * w.H} (batch, head) "
                                                 f"units of {w.name}")
        line = {"impl": "reference", "metric": METRIC, "value": tf, "unit": "TFLOP/s", "n_gpus": a.gpus,
                "steps": a.steps, "warmup": a.warmup, "ms_per_step": sec_per_head * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": ref_config,
                "cpu_baseline": {"kind": "oracle", "cores": cores, "sample": sample, "value": tf,
                                 "unit": "TFLOP/s"},
                "e2e": {"value": tf, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return
    mode = DQ_MODES[a.dq]
    r = time_ours(w, a.steps, a.warmup, mode, world)
    ms = max_over_ranks(r["ms"], world)
    e2e_ms = max_over_ranks(r["e2e_ms"], world)
    flops = counted_flops(w)
    value = world * flops / (ms * 1e-3) / 1e12
    e2e_value = world * flops / (e2e_ms * 1e-3) / 1e12
    acc = accumulates(mode)
    # Dominant kernel: the key/value-major backward. Its algorithmic work is the
    # S, dP, dV and dK contractions (8*d FLOPs per allowed pair), plus dQ (2*d)
    # when it accumulates dQ (atomic, ordered).
    kv_ms = r["stage_ms"][1]
    kv_flops = causal_pairs(w) * w.d * (10.0 if acc else 8.0)
    kv_tflops = kv_flops / (kv_ms * 1e-3) / 1e12
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    hbm_peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    esz = 4 if w.dtype == "f32" else 2
    n_pad = -(-w.N // 128) * 128
    # O and dO read, L read, -D and -L*log2e written; atomic mode also zero-fills the fp32 dQ accumulator
    pre_bytes = w.B * w.H * (w.N * (2 * w.d * esz + 4) + n_pad * 8 + (n_pad * w.d * 4 if acc else 0))
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else w.dtype, "data": "synthetic",
        "config": config,
        "pct_of_dense_bf16_peak": 100.0 * value / peak,
        "stages_ms": {"preprocess": r["stage_ms"][0], "dkdv": r["stage_ms"][1],
                      ("dq_convert" if acc else "dq_qmajor"): r["stage_ms"][2]},
        # the D pass: reads O and dO, writes -D and -L*log2e (HBM-bound)
        "preprocess_hbm": {"bytes": pre_bytes, "gbs": pre_bytes / (r["stage_ms"][0] * 1e-3) / 1e9,
                           "peak_gbs": hbm_peak,
                           "frac": pre_bytes / (r["stage_ms"][0] * 1e-3) / 1e9 / hbm_peak,
                           "peak_source": f"{peak_src} copy bandwidth"},
        "roofline": {"kernel": "bwd_dkdv (key/value-major, tcgen05)", "bound": "tensor", "achieved": kv_tflops,
                     "peak": peak, "unit": "TFLOP/s", "frac": kv_tflops / peak,
                     "traffic": dkdv_traffic(w, not acc),
                     "peak_source": f"{peak_src} burst bf16"},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": 3 * a.steps,
        # forward: 4*d FLOP per allowed pair (QK^T and PV), the usual forward count
        "forward": {"ms": r["fwd_ms"], "tflops": 0.4 * flops / (r["fwd_ms"] * 1e-3) / 1e12,
                    "bwd_over_fwd_speed": (flops / (r["ms"] * 1e-3)) / (0.4 * flops / (r["fwd_ms"] * 1e-3))},
        "clocks": r["clocks"],
        # every dQ algorithm on the same workload (recompute and ordered are the
        # deterministic ones), timed the same way as `value`
        "dq_modes": {name: {"ms_per_step": ms_m, "value": flops / (ms_m * 1e-3) / 1e12, "unit": "TFLOP/s",
                            "deterministic": name != "atomic"} for name, ms_m in r["mode_ms"].items()},
    }
    if rank == 0 and not a.no_workloads:
        # every other workload of the plan, every dQ algorithm, timed the same way
        import flashattention_backward_fa_gb300 as fa
        line["workloads"] = {name: time_workload(fa, wl) for name, wl in sorted(WORKLOADS.items())
                             if name != w.name}
        torch.cuda.empty_cache()
    if rank == 0 and not a.no_cpu_baseline:
        # a bounded sample: one warm-up and up to four timed heads, about 30 s at most
        tf, sample, cores, _ = run_reference_steps(w, steps=4, warmup=1, budget_s=30.0)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Benchmark of the fused exact-attention forward on GB300.

One step = one fa_fwd call over the whole workload (all heads, all query
tiles, every visible K/V tile).  Default workload: long context, B=4 H=32
Nq=Nk=8192 d=128, non-causal, bf16 Q/K/V ~ N(0, 1) (synthetic, seeded).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  Metric: attention forward TFLOP/s with
FLOPs = 4*B*H*Nq*Nk*d (halved when causal), plus the fraction of the measured
dense-bf16 peak.  Under torchrun each rank runs the same workload on its own
GPU (independent replicas, weak scaling); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "attention fwd TFLOP/s and % of GB300 dense BF16 peak (1 GPU)"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "long_8192_d128"
L2_BYTES = 129 * 1024 * 1024
KERNEL_SOURCES = ["exact_attention_19_gb300/csrc/fa_fwd_kernel.cuh", "exact_attention_19_gb300/csrc/fa_fwd_persist.cuh",
                  "exact_attention_19_gb300/csrc/fa_ptx.cuh", "exact_attention_19_gb300/csrc/fa_api.cu"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fa_fwd_kernel_dram_traffic.md")
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
NOMINAL_BF16_TFLOPS = 2250.0  # nominal dense bf16 tensor peak of one GB300 (not measured; context only)


# ----------------------------------------------------------------------------
# small helpers (host logic, testable without a GPU)
# ----------------------------------------------------------------------------
def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_name(w, n_splits, sms: int = 152) -> str:
    """The forward kernel the library launches for this workload: the persistent one for a single
    pass (fa_fwd and fa_fwd_splitkv with one split) without a mask at d = 128 or at d = 64 with at
    most 2048 keys, causal at d = 64 with more than 2048 keys and at least 6 query-tile pairs per
    SM, causal at d = 128 with at least 20 pairs per SM, and a window bounded on both sides
    with Nq <= Nk and at least 4 pairs per SM; else fa_fwd_kernel."""
    single = n_splits is None or n_splits <= 1
    if w.window is not None:
        wl, wr = w.window
        pairs = w.B * w.H * ((w.Nq + 255) // 256)
        if wl >= 0 and wr >= 0 and w.Nq <= w.Nk and pairs >= 4 * sms:
            return "fa_fwd_persist_kernel"
        return "fa_fwd_kernel"
    if single:
        if not w.causal and (w.d == 128 or w.Nk <= 2048):
            return "fa_fwd_persist_kernel"
        pairs = w.B * w.H * ((w.Nq + 255) // 256)
        if w.causal and w.d == 64 and w.Nk > 2048 and pairs >= 6 * sms:
            return "fa_fwd_persist_kernel"
        if w.causal and w.d == 128 and pairs >= 20 * sms:
            return "fa_fwd_persist_kernel"
    return "fa_fwd_kernel"


def read_traffic(workload: str, src_hash: str):
    """DRAM bytes per launch recorded by an ncu capture of this exact kernel source, else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    pat = re.compile(r"^\|\s*" + re.escape(workload) + r"\s*\|\s*([0-9a-f]{16})\s*\|\s*([0-9.eE+]+)\s*\|")
    with open(TRAFFIC_FILE) as f:
        for line in f:
            m = pat.match(line.strip())
            if m and m.group(1) == src_hash:
                return float(m.group(2))
    return None


def timed_steps(torch, step, steps, stream, flush):
    """Device time of `steps` calls of step(), with an event on the launching stream at every step
    boundary.  Inputs larger than L2 run back to back; otherwise the L2 is flushed before each
    step, outside its events.  Returns (total ms, per-step ms)."""
    if flush is None:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        ev[0].record(stream)
        for i in range(steps):
            step()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[steps]), [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    total, per = 0.0, []
    for _ in range(steps):
        flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1)
        per.append(t)
        total += t
    return total, per


def step_stats(per_step_ms):
    """Median and 10th / 90th percentiles of the per-step device times (ms)."""
    xs = sorted(per_step_ms)
    if not xs:
        return None

    def pct(q):
        return xs[min(len(xs) - 1, max(0, int(round(q * (len(xs) - 1)))))]

    return {"median": pct(0.5), "p10": pct(0.1), "p90": pct(0.9)}


def roofline_entry(flops, algo_bytes, achieved_tflops, achieved_gbs, peak_tflops, peak_gbs):
    """The binding roofline of a workload: the tensor pipe when its intensity
    (FLOPs per compulsory byte) is at or above the ridge peak_tflops / peak_gbs,
    HBM below it.  Both achieved figures are kept."""
    intensity = flops / algo_bytes
    ridge = peak_tflops * 1e12 / (peak_gbs * 1e9)
    if intensity >= ridge:
        out = {"bound": "tensor", "achieved": achieved_tflops, "peak": peak_tflops, "unit": "TFLOP/s",
               "frac": achieved_tflops / peak_tflops, "peak_kind": "bf16 burst"}
    else:
        out = {"bound": "hbm", "achieved": achieved_gbs, "peak": peak_gbs, "unit": "GB/s",
               "frac": achieved_gbs / peak_gbs, "peak_kind": "HBM copy"}
    out.update({"intensity_flop_per_byte": intensity, "ridge_flop_per_byte": ridge,
                "achieved_tflops": achieved_tflops, "achieved_gbs": achieved_gbs})
    return out


def e2e_entry(pipe_value, pipe_ms, serial_value, serial_ms, h2d_bytes, d2h_bytes, steps):
    """End-to-end line: the faster of the two ways of running the steps (both
    move every step's inputs in and results out inside the timed region), with
    both figures kept."""
    use_pipe = not (serial_value > pipe_value)  # NaN-safe: a missing serial run picks the pipelined one
    return {"value": pipe_value if use_pipe else serial_value, "unit": UNIT,
            "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
            "ms_per_step": pipe_ms if use_pipe else serial_ms, "steps": steps,
            "mode": "pipelined" if use_pipe else "serial",
            "pipelined_value": pipe_value, "pipelined_ms_per_step": pipe_ms,
            "serial_value": serial_value, "serial_ms_per_step": serial_ms,
            "how": "pinned host inputs copied in and O, LSE read back every step; serial: copies and kernel on "
                   "one stream; pipelined: two device buffer sets, copies on two copy streams overlapping the "
                   "previous step's kernel"}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def visible_keys(w: synth.Workload, rows: np.ndarray) -> np.ndarray:
    """Keys each flat query row attends to: all Nk, i + 1 under the causal mask,
    or the keys its sliding window keeps (bottom-right alignment, -1 = open side)."""
    i = rows % w.Nq
    if w.window is not None:
        wl, wr = w.window
        s = w.Nk - w.Nq
        lo = np.maximum(0, i + s - wl) if wl >= 0 else np.zeros_like(i)
        hi = np.minimum(w.Nk, i + s + wr + 1) if wr >= 0 else np.full(i.shape, w.Nk)
        return np.maximum(0, hi - lo)
    return np.minimum(i + 1, w.Nk) if w.causal else np.full(rows.shape, w.Nk)


def flops_of(w: synth.Workload) -> float:
    """Counted forward FLOPs: 4*B*H*Nq*Nk*d, halved under the causal mask (the
    metric's convention); under a window, 4*d per (row, key) pair it keeps."""
    if w.window is None:
        return w.flops
    kept = float(np.sum(visible_keys(w, np.arange(w.Nq))))
    return 4.0 * w.B * w.H * kept * w.d


def pairs_of(w: synth.Workload) -> float:
    """(row, key) pairs whose exponential is taken per step."""
    return flops_of(w) / (4.0 * w.d)


def sample_rows_even(w: synth.Workload, n: int) -> np.ndarray:
    total = w.B * w.H * w.Nq
    n = max(1, min(n, total))
    return np.unique(np.linspace(0, total - 1, n).round().astype(np.int64))


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise max of a list of floats over all ranks (identity without a process group)."""
    if dist is None:
        return [float(x) for x in values]
    import torch

    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def aggregate(elapsed_ms_per_rank, flops_per_rank):
    """Whole-job throughput: all ranks' FLOPs over the slowest rank's time."""
    t = max(elapsed_ms_per_rank)
    return sum(flops_per_rank) / (t * 1e-3) / 1e12, t


class ClockSampler:
    """nvidia-smi sampled every 100 ms in the background; keep (time, row)."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        self.thread = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        inside = [s for (t, s) in self.samples if t0 <= t <= t1]
        if not inside and self.samples:  # region shorter than the sampling period: nearest sample
            mid = 0.5 * (t0 + t1)
            inside = [min(self.samples, key=lambda ts: abs(ts[0] - mid))[1]]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(s[0]) for s in inside if num(s[0]) is not None]
        smax = [num(s[1]) for s in inside if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4) if s[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside)}


# ----------------------------------------------------------------------------
# CPU oracle leg (the reference arm and the cpu_baseline field)
# ----------------------------------------------------------------------------
def time_oracle(w: synth.Workload, q, k, v, budget_s: float, max_rows: int | None = None):
    """Run the oracle on an even sample of rows sized to about budget_s.

    Returns (TFLOP/s, seconds, rows, threads)."""
    import oracle

    # calibrate: a warm-up call (thread pool, page faults), then grow the
    # sample until one call takes a measurable fraction of the budget
    n_probe = 16
    oracle.attention_rows(q, k, v, sample_rows_even(w, n_probe), w.scale, w.causal, window=w.window)
    while True:
        probe = sample_rows_even(w, n_probe)
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, probe, w.scale, w.causal, window=w.window)
        t_probe = max(time.perf_counter() - t0, 1e-6)
        if t_probe >= 0.05 * budget_s or probe.size >= w.B * w.H * w.Nq:
            break
        n_probe *= 4
    n = int(len(probe) * budget_s / t_probe)
    if max_rows:
        n = min(n, max_rows)
    rows = sample_rows_even(w, max(n, 16))
    t0 = time.perf_counter()
    oracle.attention_rows(q, k, v, rows, w.scale, w.causal, window=w.window)
    secs = time.perf_counter() - t0
    flops = float(np.sum(4.0 * visible_keys(w, rows) * w.d))
    return flops / secs / 1e12, secs, int(rows.size), oracle.threads()


def run_reference(args, w: synth.Workload, rank: int):
    if rank != 0:
        return 0
    import oracle

    oracle.build()
    q, k, v = w.make()
    steps, warmup = args.steps, args.warmup
    per_step = max(0.05, min(2.0, 150.0 / max(1, steps + warmup)))
    for _ in range(warmup):
        time_oracle(w, q, k, v, per_step)
    total_flops, total_s, total_rows, threads = 0.0, 0.0, 0, oracle.threads()
    for _ in range(steps):
        tflops, secs, n, threads = time_oracle(w, q, k, v, per_step)
        total_flops += tflops * 1e12 * secs
        total_s += secs
        total_rows += n
    value = total_flops / total_s / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": warmup, "ms_per_step": total_s / steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{total_rows // steps} evenly spaced query rows of {w.name} per step "
                                   f"(of {w.B * w.H * w.Nq}); fp64 C oracle, OpenMP"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w: synth.Workload, l2_note: str | None = None):
    c = {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d, "causal": w.causal,
         "scale": w.scale, "inputs": f"bf16 q~N(0,{w.sigma_q:g}^2), k,v~N(0,1), seed {w.seed}",
         "flops_per_step": flops_of(w)}
    if w.window is not None:
        c["window"] = list(w.window)
    if l2_note:
        c["l2"] = l2_note
    return c


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def run_gpu(args, w: synth.Workload, rank: int, world: int, local_rank: int):
    import torch

    import exact_attention_19_gb300 as fa
    from exact_attention_19_gb300 import build as fa_build

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    fa_build.build()
    fa.load()

    dist = None
    if world > 1:
        import torch.distributed as dist

    q_h, k_h, v_h = w.make()  # bf16 bits, host

    def pinned(bits):
        t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
        return t.pin_memory()

    q_p, k_p, v_p = pinned(q_h), pinned(k_h), pinned(v_h)
    q, k, v = q_p.to(dev), k_p.to(dev), v_p.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    in_bytes = 2 * (q.numel() + k.numel() + v.numel())
    big_inputs = in_bytes > L2_BYTES
    flush = None if big_inputs else torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    l2_note = (f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB > {L2_BYTES / 1e6:.0f} MB)" if big_inputs
               else f"L2 flushed between timed steps ({2 * L2_BYTES / 1e6:.0f} MB write)")

    # split-KV (the library's choice for grids that would leave SMs idle) runs
    # two kernels per step: the sliced forward and the merge
    n_splits = fa.fa_splitkv_heuristic(w.B, w.H, w.Nq, w.Nk, w.d, int(w.causal))
    workspace = None
    if n_splits > 1:
        workspace = torch.empty(fa.fa_splitkv_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d, n_splits),
                                dtype=torch.uint8, device=dev)
    launches_per_step = 2 if n_splits > 1 else 1

    def step():
        fa.fwd(q, k, v, causal=w.causal, scale=w.scale, window=w.window, out=o, lse=lse, stream=stream,
               n_splits=n_splits, workspace=workspace)

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, word = fa.fa_fwd_status(None, clear=True)
    if st != 0:
        raise RuntimeError(f"kernel reported a wait timeout during warm-up (status {word:#x})")

    # denominator of the exponential-unit roofline, measured before the timed region
    ex2_peak = fa.fa_probe_exp2(0, stream)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count

    try:
        props = torch.cuda.get_device_properties(dev)
        gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(local_rank)
    except Exception:
        gpu_id = str(local_rank)
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)

    # ---- device-timed steps ------------------------------------------------
    barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    elapsed, per_step = timed_steps(torch, step, args.steps, stream, flush)
    barrier()
    torch.cuda.synchronize()
    wall1 = time.time()
    time.sleep(0.15)
    sampler.stop()
    clocks = sampler.summary(wall0, wall1)
    st, word = fa.fa_fwd_status(None, clear=True)
    if st != 0:
        raise RuntimeError(f"kernel reported a wait timeout (status {word:#x})")

    # ---- end-to-end through the public API with host buffers ----------------
    # Every step copies its inputs from pinned host memory, runs fa.fwd and
    # reads O and LSE back into pinned host memory.  Serial: all on one stream.
    # Pipelined (the reported e2e): two device buffer sets, host->device copies
    # on one copy stream and device->host reads on another, so step k+1's
    # inputs travel while step k computes; each step still moves its own bytes.
    o_host = [torch.empty(o.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    lse_host = [torch.empty(lse.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    e2e_steps = max(1, min(args.steps, 50))
    e2e_ms = e2e_serial_ms = float("nan")
    if not args.no_e2e:
        qd, kd, vd = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

        def e2e_serial_step():
            qd.copy_(q_p, non_blocking=True)
            kd.copy_(k_p, non_blocking=True)
            vd.copy_(v_p, non_blocking=True)
            fa.fwd(qd, kd, vd, causal=w.causal, scale=w.scale, window=w.window, out=o, lse=lse, stream=stream,
                   n_splits=n_splits, workspace=workspace)
            o_host[0].copy_(o, non_blocking=True)
            lse_host[0].copy_(lse, non_blocking=True)

        sets = [(qd, kd, vd, o, lse),
                (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(o),
                 torch.empty_like(lse))]
        h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_kernel = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def e2e_pipelined(n):
            for i in range(n):
                b = i & 1
                qb, kb, vb, ob, lb = sets[b]
                if i >= 2:
                    h2d_stream.wait_event(ev_kernel[b])  # step i-2 has finished reading this input set
                with torch.cuda.stream(h2d_stream):
                    qb.copy_(q_p, non_blocking=True)
                    kb.copy_(k_p, non_blocking=True)
                    vb.copy_(v_p, non_blocking=True)
                ev_in[b].record(h2d_stream)
                stream.wait_event(ev_in[b])
                if i >= 2:
                    stream.wait_event(ev_out[b])  # step i-2's outputs have been read back
                fa.fwd(qb, kb, vb, causal=w.causal, scale=w.scale, window=w.window, out=ob, lse=lb, stream=stream,
                       n_splits=n_splits, workspace=workspace)
                ev_kernel[b].record(stream)
                d2h_stream.wait_event(ev_kernel[b])
                with torch.cuda.stream(d2h_stream):
                    o_host[b].copy_(ob, non_blocking=True)
                    lse_host[b].copy_(lb, non_blocking=True)
                ev_out[b].record(d2h_stream)
            stream.wait_stream(h2d_stream)
            stream.wait_stream(d2h_stream)

        def timed(fn):
            barrier()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            barrier()
            return e0.elapsed_time(e1) / e2e_steps

        for _ in range(min(args.warmup, 3)):
            e2e_serial_step()
        e2e_pipelined(min(args.warmup, 3))
        e2e_serial_ms = timed(lambda: [e2e_serial_step() for _ in range(e2e_steps)])
        e2e_ms = timed(lambda: e2e_pipelined(e2e_steps))
        st, word = fa.fa_fwd_status(None, clear=True)
        if st != 0:
            raise RuntimeError(f"kernel reported a wait timeout in the end-to-end run (status {word:#x})")

    # ---- max over ranks -------------------------------------------------------
    t_max_elapsed, t_max_e2e, t_max_e2e_serial = max_over_ranks([elapsed, e2e_ms, e2e_serial_ms], dist, dev)
    times = [t_max_elapsed] * world
    value, t_max = aggregate(times, [flops_of(w) * args.steps] * world)
    e2e_value, _ = aggregate([t_max_e2e] * world, [flops_of(w)] * world)
    e2e_serial_value, _ = aggregate([t_max_e2e_serial] * world, [flops_of(w)] * world)
    ms_per_step = t_max / args.steps

    if rank != 0:
        return 0

    peaks, peaks_kind = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved = flops_of(w) / (ms_per_step * 1e-3) / 1e12
    achieved_gbs = w.algorithmic_bytes / (ms_per_step * 1e-3) / 1e9
    src_hash = kernel_source_hash()
    traffic = read_traffic(w.name, src_hash)
    roofline = roofline_entry(flops_of(w), w.algorithmic_bytes, achieved, achieved_gbs, peak, hbm)
    roofline.update({"traffic": traffic, "peak_kind": f"{roofline['peak_kind']}, {peaks_kind}",
                     "frac_of_sustained": achieved / float(peaks.get("bf16_tflops_sustained", peak)),
                     "frac_of_nominal": achieved / NOMINAL_BF16_TFLOPS,
                     "kernel": kernel_name(w, n_splits), "kernel_source": src_hash,
                     "algorithmic_bytes": w.algorithmic_bytes})

    # third roofline: exponentials (one ex2 per visible score) per SM clock
    # against the probe's rate, at the median SM clock seen under load
    ex2_per_step = pairs_of(w)
    mufu = None
    if clocks.get("sm_mhz"):
        rate = ex2_per_step / (ms_per_step * 1e-3) / (float(clocks["sm_mhz"]) * 1e6) / n_sm
        mufu = {"bound": "mufu", "achieved": rate, "peak": ex2_peak, "unit": "ex2/clk/SM", "frac": rate / ex2_peak,
                "ex2_per_step": ex2_per_step, "sm_mhz": clocks["sm_mhz"], "sms": n_sm,
                "peak_kind": "measured by fa_probe_exp2 (ex2.approx) on this GPU"}

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        q_np, k_np, v_np = q_h, k_h, v_h
        c_val, c_secs, c_rows, c_threads = time_oracle(w, q_np, k_np, v_np, args.cpu_seconds)
        cpu = {"value": c_val, "unit": UNIT, "cores": c_threads, "kind": "oracle",
               "sample": f"{c_rows} evenly spaced query rows of {w.B * w.H * w.Nq} ({c_secs:.1f} s, fp64 C "
                         f"oracle, OpenMP)"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(config_of(w, l2_note), n_splits=n_splits),
        "roofline": roofline, "mufu_roofline": mufu, "cpu_baseline": cpu,
        "e2e": e2e_entry(e2e_value, e2e_ms, e2e_serial_value, e2e_serial_ms, int(in_bytes),
                         int(2 * o.numel() + 4 * lse.numel()), e2e_steps),
        "gpu_launches": args.steps * launches_per_step, "clocks": clocks,
        "pct_of_peak": 100.0 * achieved / peak,  # of the dense bf16 peak, whatever the binding roofline
        "ms_step_stats": step_stats(per_step), "peak_mem_bytes": int(torch.cuda.max_memory_allocated(dev)),
    }
    print(json.dumps(line), flush=True)
    return 0


def bwd_algorithmic_bytes(w: synth.Workload) -> int:
    """Compulsory HBM bytes of one fa_bwd: Q, K, V, O, dO and LSE read, dQ, dK, dV written,
    and the fp32 L and D workspace written by the first kernel and read by the second."""
    bhnd = w.B * w.H * w.Nq * w.d
    rows = w.B * w.H * w.Nq
    return 2 * (5 + 3) * bhnd + 4 * rows + 2 * 8 * rows


def run_bwd(args, w: synth.Workload, local_rank: int):
    """Backward-pass timing line (not the headline metric): one fa_bwd per step.
    FLOPs are counted as 2.5x the forward's; the two kernels execute 3.5x (S and dP
    are recomputed in each), reported as roofline.executed_tflops."""
    import torch

    import exact_attention_19_gb300 as fa
    from exact_attention_19_gb300 import build as fa_build

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    fa_build.build()
    q_h, k_h, v_h = w.make()
    do_h = synth.normal_bf16(w.seed + 7, 3, w.q_shape())

    def up(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    q, k, v, do = up(q_h), up(k_h), up(v_h), up(do_h)
    o, lse = fa.fwd(q, k, v, causal=w.causal, scale=w.scale, window=w.window, n_splits=1)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.Nq), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    algo_bytes = bwd_algorithmic_bytes(w)
    in_bytes = 2 * (q.numel() + k.numel() + v.numel() + o.numel() + do.numel())
    big_inputs = in_bytes > L2_BYTES
    flush = None if big_inputs else torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    l2_note = (f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB > {L2_BYTES / 1e6:.0f} MB)" if big_inputs
               else f"L2 flushed between timed steps ({2 * L2_BYTES / 1e6:.0f} MB write)")

    def step():
        fa.bwd(q, k, v, o, lse, do, causal=w.causal, scale=w.scale, window=w.window, dq=dq, dk=dk, dv=dv,
               workspace=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    try:
        props = torch.cuda.get_device_properties(dev)
        gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(local_rank)
    except Exception:
        gpu_id = str(local_rank)
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)
    torch.cuda.synchronize()
    wall0 = time.time()
    elapsed, per_step = timed_steps(torch, step, args.steps, stream, flush)
    torch.cuda.synchronize()
    wall1 = time.time()
    time.sleep(0.15)
    sampler.stop()
    clocks = sampler.summary(wall0, wall1)
    st, word = fa.fa_fwd_status(None, clear=True)
    if st != 0:
        raise RuntimeError(f"kernel reported a wait timeout (status {word:#x})")
    ms = elapsed / args.steps
    flops = 2.5 * flops_of(w)
    peaks, kind = load_peaks()
    value = flops / (ms * 1e-3) / 1e12
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_gbs = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    roofline = roofline_entry(flops, algo_bytes, value, algo_bytes / (ms * 1e-3) / 1e9, peak_tf, peak_gbs)
    roofline.update({"traffic": None, "peak_kind": f"{roofline['peak_kind']}, {kind}", "kernel": "fa_bwd (dQ + dK/dV)",
                     "algorithmic_bytes": algo_bytes, "executed_tflops": 1.4 * value,
                     "executed_frac": 1.4 * value / peak_tf})
    config = dict(config_of(w))
    config["l2"] = l2_note
    print(json.dumps({"metric": "attention bwd TFLOP/s (2.5x forward FLOPs)", "value": value, "unit": UNIT,
                      "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                      "higher_is_better": True, "dtype": "bf16", "data": "synthetic", "config": config,
                      "frac_of_peak": value / peak_tf, "roofline": roofline, "clocks": clocks,
                      "ms_step_stats": step_stats(per_step), "peak_mem_bytes": int(torch.cuda.max_memory_allocated(dev)),
                      "gpu_launches": 2 * args.steps}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--pass", dest="which", choices=["fwd", "bwd"], default="fwd",
                    help="bwd: time fa_bwd instead (FLOPs counted as 2.5x the forward's)")
    ap.add_argument("--window", default=None, metavar="LEFT,RIGHT",
                    help="sliding-window mask over the workload (bottom-right, -1 = open side); "
                         "FLOPs then count 4*d per kept (row, key) pair")
    ap.add_argument("--causal", action="store_true",
                    help="apply the causal mask to the workload (square workloads only; FLOPs halved)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference" and args.which == "bwd":
        ap.error("the reference arm times the forward oracle only; --pass bwd has none")
    w = synth.WORKLOADS[args.workload]
    if args.window is not None:
        try:
            wl, wr = (int(x) for x in args.window.split(","))
        except ValueError:
            ap.error("--window takes two integers: LEFT,RIGHT")
        if wl < -1 or wr < -1:
            ap.error("--window bounds must be >= -1")
        # its own name: the window's launch has its own DRAM traffic (and config)
        w = w.with_(window=(wl, wr), causal=False, name=f"{w.name}_window_{wl}_{wr}")
    if args.causal:
        if args.window is not None:
            ap.error("--causal and --window exclude each other")
        if w.Nq != w.Nk:
            ap.error("--causal needs a square workload (Nq == Nk)")
        if not w.causal:
            w = w.with_(causal=True, name=w.name + "_causal")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, w, rank)
    if args.which == "bwd":
        return run_bwd(args, w, local_rank)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    try:
        return run_gpu(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())

#!/usr/bin/env python
"""Throughput of exact IO-aware attention (forward + backward) on GB300.

One step = one forward (fa_fwd) and one backward (fa_bwd) over one batch of
the long-context workload: B=1, H=16, N=16384, d=128, causal, bf16 inputs
(seeded synthetic N(0,1) data with a sink key row, as in the workload table).
Counted FLOPs: 4*B*H*N^2*d forward, x2.5 backward, halved for causal.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  N > 1 runs N independent replicas (one per
GPU, launched by torchrun); the path has no exchange step, so there is no
data-path collective, only a barrier and a max over ranks for timing.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("attention fwd and fwd+bwd TFLOP/s (bf16, causal) and % of GB300 dense BF16 peak")
DEFAULT_WORKLOAD = "long_sink_b1h16_n16384_d128_causal"
L2_FLUSH_BYTES = 512 << 20          # > the 129 MB L2, written between timed steps
ISSUE_FLOP_PER_CLK_SM = 8192        # dense bf16 tcgen05 rate per SM per clock (measured)
NUM_SMS = 152
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


# --------------------------------------------------------------- helpers ----
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(world: int, device=None):
    import torch.distributed as dist
    if world > 1:
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of a float over ranks (identity at world size 1)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(flops_per_step: float, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job TFLOP/s: every rank ran `steps` replica steps; the job took the
    slowest rank's time."""
    return world * steps * flops_per_step / max_seconds / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_io_aware_12_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            doc = json.load(f)
    except (OSError, ValueError):
        return None
    if doc.get("source_hash") != kernel_source_hash():
        return None
    ent = doc.get("kernels", {}).get(kernel)
    return None if ent is None else ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons; samples are
    timestamped so the summary covers only the timed window (mark_start /
    mark_end)."""

    FIELDS = "timestamp," + CLOCK_FIELDS
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index: int, period_ms: int = 50, path=None):
        self.index, self.period_ms, self.proc, self.path = index, period_ms, None, path
        self.t_start = self.t_end = None
        self.tmpdir = None

    def __enter__(self):
        if self.path is None:      # a private temporary file unless --clock-csv names one
            import tempfile
            self.tmpdir = tempfile.mkdtemp(prefix="fa_clocks_")
            self.path = os.path.join(self.tmpdir, f"clocks_gpu{self.index}.csv")
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period_ms}"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.5)
        except (OSError, ValueError):
            self.proc = None
        return self

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def cleanup(self):
        """Remove the temporary CSV (after summary())."""
        if self.tmpdir is not None:
            import shutil
            shutil.rmtree(self.tmpdir, ignore_errors=True)
            self.tmpdir = None

    @staticmethod
    def _parse_time(ts: str):
        from datetime import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.strptime(ts.strip(), fmt).timestamp()
            except ValueError:
                continue
        return None

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        samples = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                samples.append((self._parse_time(parts[0]), float(parts[2]), float(parts[3]),
                                float(parts[4]), parts[6:10]))
            except ValueError:
                continue
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        inside = samples
        if self.t_start is not None and self.t_end is not None and samples[0][0] is not None:
            inside = [x for x in samples if x[0] is not None and
                      self.t_start - 0.05 <= x[0] <= self.t_end + 0.05]
            if not inside:   # window shorter than the sampling period: nearest sample
                mid = 0.5 * (self.t_start + self.t_end)
                inside = [min(samples, key=lambda x: abs((x[0] or 0) - mid))]
        reasons = sorted({n for x in inside for n, v in zip(self.REASONS, x[4])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(x[1] for x in inside),
                "sm_max_mhz": max(x[2] for x in inside), "reasons": reasons,
                "samples_in_window": len(inside),
                "power_w_max": max(x[3] for x in inside)}


def pick_workload(args):
    """The named workload, or (--shape B,H,N,d,causal) a same-recipe variant
    used for profiling captures of a smaller case."""
    from exact_io_aware_12_gb300.workloads import BY_NAME, Workload
    w = BY_NAME[args.workload]
    if args.shape:
        B, H, N, d, c = (int(v) for v in args.shape.split(","))
        w = Workload(f"{w.name}@{B}x{H}x{N}x{d}{'c' if c else ''}", B, H, N, d, bool(c), w.seed,
                     w.qk_scale, w.sink)
    return w


# ------------------------------------------------------------ our impl ----
def run_ours(args):
    import torch
    from exact_io_aware_12_gb300 import api, _lib
    from exact_io_aware_12_gb300.workloads import flops_fwd, flops_bwd, make_inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    if rank == 0:
        _lib.load()               # builds if needed, once
    barrier(world, dev)
    _lib.load()

    w = pick_workload(args)
    B, H, N, d = w.shape
    f_fwd = flops_fwd(B, H, N, d, w.causal)
    f_bwd = flops_bwd(B, H, N, d, w.causal)
    f_step = f_fwd + f_bwd
    x = make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(api.workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        api.fwd(q, k, v, w.causal, w.tau, out=o, lse=lse)
        api.bwd(q, k, v, o, do, lse, w.causal, w.tau, dq=dq, dk=dk, dv=dv, workspace=ws)

    ev = lambda: torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize(dev)
    if api.last_device_error(dev) != _lib.FA_OK:
        raise RuntimeError("kernel watchdog fired during warm-up")

    # events: whole step, forward kernel, backward main kernel (per step)
    st_s, st_e = [ev() for _ in range(args.steps)], [ev() for _ in range(args.steps)]
    kf_s, kf_e = [ev() for _ in range(args.steps)], [ev() for _ in range(args.steps)]
    kb_s, kb_e = [ev() for _ in range(args.steps)], [ev() for _ in range(args.steps)]
    for e in st_s + st_e + kf_s + kf_e + kb_s + kb_e:
        e.record(stream)           # materialise the handles
    torch.cuda.synchronize(dev)

    with ClockSampler(local, path=args.clock_csv) as clocks:
        barrier(world, dev)
        torch.cuda.synchronize(dev)
        clocks.mark_start()
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))                      # L2 flush, outside the step events
            st_s[i].record(stream)
            _lib.check(_lib.fa_set_timing_events(kf_s[i].cuda_event, kf_e[i].cuda_event), "timing")
            api.fwd(q, k, v, w.causal, w.tau, out=o, lse=lse)
            _lib.check(_lib.fa_set_timing_events(kb_s[i].cuda_event, kb_e[i].cuda_event), "timing")
            api.bwd(q, k, v, o, do, lse, w.causal, w.tau, dq=dq, dk=dk, dv=dv, workspace=ws)
            _lib.check(_lib.fa_set_timing_events(None, None), "timing")
            st_e[i].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        clocks.mark_end()
        barrier(world, dev)
    if api.last_device_error(dev) != _lib.FA_OK:
        raise RuntimeError("kernel watchdog fired during the timed steps")

    step_ms = [a.elapsed_time(b) for a, b in zip(st_s, st_e)]
    fwd_ms = [a.elapsed_time(b) for a, b in zip(kf_s, kf_e)]
    bwd_ms = [a.elapsed_time(b) for a, b in zip(kb_s, kb_e)]
    total_s = reduce_max(sum(step_ms) / 1e3, world, dev)
    value = aggregate_value(f_step, args.steps, world, total_s)
    fwd_avg = reduce_max(sum(fwd_ms) / len(fwd_ms), world, dev)
    bwd_avg = reduce_max(sum(bwd_ms) / len(bwd_ms), world, dev)

    peaks, peak_src = measured_peaks()
    peak = float(peaks["bf16_tflops"])
    fwd_tf = f_fwd / (fwd_avg / 1e3) / 1e12
    bwdk_tf = f_bwd / (bwd_avg / 1e3) / 1e12
    step_avg_ms = total_s * 1e3 / args.steps
    # the dominant kernel by device time
    if bwd_avg >= fwd_avg:
        dom, dom_tf, dom_name = "fa_bwd_main_kernel", bwdk_tf, "bwd_main"
    else:
        dom, dom_tf, dom_name = "fa_fwd_kernel", fwd_tf, "fwd"
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(dom_tf, 2),
                "peak": peak, "unit": "TFLOP/s", "frac": round(dom_tf / peak, 4),
                "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json bf16_tflops)",
                "traffic": profiled_traffic(dom_name)}

    clk = clocks.summary()
    clocks.cleanup()
    # the tensor pipe's issue-rate ceiling at the clock seen during the timed steps:
    # 8192 dense bf16 FLOP per clock per SM (a 128x128x16 MMA every 64 cycles, measured)
    sm_mhz = clk.get("sm_mhz") or clk.get("sm_max_mhz") or 2070.0
    issue_ceiling = ISSUE_FLOP_PER_CLK_SM * NUM_SMS * sm_mhz * 1e6 / 1e12
    roofline["issue_ceiling_tflops"] = round(issue_ceiling, 1)
    roofline["frac_of_issue_ceiling"] = round(dom_tf / issue_ceiling, 4)
    roofline["issue_ceiling_source"] = (f"{ISSUE_FLOP_PER_CLK_SM} FLOP/clk/SM x {NUM_SMS} SMs x "
                                        f"median SM clock {sm_mhz:.0f} MHz in the timed steps")

    configs_leg = measure_configs(w, dev, min(args.steps, 20), peak) if args.configs else None
    window_leg = (measure_window(w, q, k, v, do, dev, args.window, min(args.steps, 20), peak)
                  if args.window > 0 and w.causal else None)
    blocks_leg = (measure_blocks(w, q, k, v, do, dev, min(args.steps, 20), peak)
                  if args.blocks and w.causal else None)
    decode_leg = (measure_decode(dev, min(args.steps, 20), peaks,
                                 tuple(int(v) for v in args.decode_shape.split(",")))
                  if args.decode else None)
    fp8_leg = (measure_fp8(w, dev, min(args.steps, 20), peak)
               if args.fp8 and d == 128 else None)
    e2e = run_e2e(args, w, x, dev, f_step) if not args.no_e2e else None
    cpu = run_cpu_baseline(w, budget_s=args.cpu_seconds) if (rank == 0 and not args.no_cpu) else None

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_avg_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, key row 0 = 4 x mean query per head)",
        "config": {"workload": w.name, "B": B, "H": H, "N": N, "d": d, "causal": w.causal,
                   "step": "fa_fwd + fa_bwd", "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed before every timed step (512 MiB write, outside the step events)"},
        "frac_of_peak": round(value / world / peak, 4),
        "fwd": {"ms": round(fwd_avg, 4), "tflops": round(fwd_tf, 2), "frac": round(fwd_tf / peak, 4)},
        "bwd_main_kernel": {"ms": round(bwd_avg, 4), "tflops": round(bwdk_tf, 2),
                            "frac": round(bwdk_tf / peak, 4)},
        "fwd_bwd_step": {"ms": round(step_avg_ms, 4), "tflops_per_gpu": round(value / world, 2)},
        "roofline": roofline,
        "configs": configs_leg,
        "sliding_window": window_leg,
        "block_sparse": blocks_leg,
        "decode": decode_leg,
        "fp8": fp8_leg,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 4 * args.steps,
        "clocks": clk,
        "wall_s_timed_loop": round(wall, 3),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def measure_configs(headline, dev, steps, peak):
    """Every other named workload (the tiny check, the two GPT-2 shapes and the
    128k forward-only one), timed like the headline: L2 flushed before each
    step, CUDA events around the forward kernel, the backward main kernel and
    the whole fa_fwd + fa_bwd step (pre and post kernels included)."""
    import torch
    from exact_io_aware_12_gb300 import api, _lib
    from exact_io_aware_12_gb300.workloads import WORKLOADS, flops_fwd, flops_bwd, make_inputs

    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    out = {}
    for w in WORKLOADS:
        if w.name == headline.name:
            continue
        B, H, N, d = w.shape
        x = make_inputs(w)
        q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
        do = x["do"].to(dev) if w.backward else None
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        if w.backward:
            dq, dk, dv = (torch.empty_like(q) for _ in range(3))
            ws = torch.empty(api.workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)

        def run(i=None, ev=None):
            if ev is not None:
                ev[0].record(stream)
                _lib.check(_lib.fa_set_timing_events(ev[1].cuda_event, ev[2].cuda_event), "timing")
            api.fwd(q, k, v, w.causal, w.tau, out=o, lse=lse)
            if w.backward:
                if ev is not None:
                    _lib.check(_lib.fa_set_timing_events(ev[3].cuda_event, ev[4].cuda_event), "timing")
                api.bwd(q, k, v, o, do, lse, w.causal, w.tau, dq=dq, dk=dk, dv=dv, workspace=ws)
            if ev is not None:
                _lib.check(_lib.fa_set_timing_events(None, None), "timing")
                ev[5].record(stream)

        for _ in range(3):
            run()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
        for e in sum(ev, []):
            e.record(stream)
        torch.cuda.synchronize(dev)
        for i in range(steps):
            flush.fill_(float(i))
            run(i, ev[i])
        torch.cuda.synchronize(dev)
        if api.last_device_error(dev) != _lib.FA_OK:
            raise RuntimeError(f"kernel watchdog fired in the {w.name} leg")
        ff, fb = flops_fwd(B, H, N, d, w.causal), flops_bwd(B, H, N, d, w.causal)
        fms = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
        sms = sum(e[0].elapsed_time(e[5]) for e in ev) / steps
        ent = {"B": B, "H": H, "N": N, "d": d, "causal": w.causal, "steps": steps,
               "fwd": {"ms": round(fms, 4), "tflops": round(ff / fms / 1e9, 2),
                       "frac": round(ff / fms / 1e9 / peak, 4)}}
        if w.backward:
            bms = sum(e[3].elapsed_time(e[4]) for e in ev) / steps
            ent["bwd_main_kernel"] = {"ms": round(bms, 4), "tflops": round(fb / bms / 1e9, 2),
                                      "frac": round(fb / bms / 1e9 / peak, 4)}
            ent["fwd_bwd_step"] = {"ms": round(sms, 4), "tflops": round((ff + fb) / sms / 1e9, 2),
                                   "frac": round((ff + fb) / sms / 1e9 / peak, 4)}
        else:
            ent["step"] = "fa_fwd only (the workload has no backward)"
        out[w.name] = ent
        del q, k, v, do, o, lse, x
        if w.backward:
            del dq, dk, dv, ws
        torch.cuda.empty_cache()
    return out


def window_flops_fwd(B, H, N, d, window):
    """Counted forward FLOPs with a causal window: 4 d per visible score, and row
    i sees min(i + 1, window) keys."""
    n_in = min(N, window)
    visible = n_in * (n_in + 1) // 2 + (N - n_in) * window
    return 4.0 * B * H * d * visible


def blocks_flops_fwd(B, H, N, d, causal, mask):
    """Counted forward FLOPs with a block mask: 4 d per visible score.  Block
    (i, j) holds rows_i x keys_j scores; with causal, the diagonal block holds
    rows_i (rows_i + 1) / 2 and blocks above it none.  mask: [nb, nb] (one for
    every head) or [B*H, nb, nb]."""
    import numpy as np
    nb = mask.shape[-1]
    sizes = np.minimum(128, N - 128 * np.arange(nb)).astype(np.float64)
    cnt = np.outer(sizes, sizes)
    if causal:
        cnt = np.tril(cnt, -1) + np.diag(sizes * (sizes + 1) / 2)
    m = (np.asarray(mask) != 0).reshape(-1, nb, nb)
    visible = float((m * cnt).sum()) * (B * H if m.shape[0] == 1 else 1)
    return 4.0 * d * visible


def measure_variant(w, q, k, v, do, dev, steps, peak, ff, **mask):
    """The same workload with a mask variant (window=... or blocks=..., passed
    to api.fwd / api.bwd): per-kernel CUDA-event times and TFLOP/s on the
    variant's counted forward FLOPs ff (backward = 2.5 x forward)."""
    import torch
    from exact_io_aware_12_gb300 import api, _lib

    B, H, N, d = w.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(api.workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(3):
        api.fwd(q, k, v, True, w.tau, out=o, lse=lse, **mask)
        api.bwd(q, k, v, o, do, lse, True, w.tau, dq=dq, dk=dk, dv=dv, workspace=ws, **mask)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for e in sum(ev, []):
        e.record(stream)
    torch.cuda.synchronize(dev)
    for i in range(steps):
        flush.fill_(float(i))
        _lib.check(_lib.fa_set_timing_events(ev[i][0].cuda_event, ev[i][1].cuda_event), "timing")
        api.fwd(q, k, v, True, w.tau, out=o, lse=lse, **mask)
        _lib.check(_lib.fa_set_timing_events(ev[i][2].cuda_event, ev[i][3].cuda_event), "timing")
        api.bwd(q, k, v, o, do, lse, True, w.tau, dq=dq, dk=dk, dv=dv, workspace=ws, **mask)
        _lib.check(_lib.fa_set_timing_events(None, None), "timing")
    torch.cuda.synchronize(dev)
    if api.last_device_error(dev) != _lib.FA_OK:
        raise RuntimeError(f"kernel watchdog fired in the {sorted(mask)} leg")
    fms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    bms = sum(e[2].elapsed_time(e[3]) for e in ev) / steps
    return {"steps": steps,
            "fwd": {"ms": round(fms, 4), "tflops": round(ff / fms / 1e9, 2),
                    "frac": round(ff / fms / 1e9 / peak, 4)},
            "bwd_main_kernel": {"ms": round(bms, 4), "tflops": round(2.5 * ff / bms / 1e9, 2),
                                "frac": round(2.5 * ff / bms / 1e9 / peak, 4)},
            "flops_fwd": ff}


SWEEP_TOKENS = 16 * 16384  # B*H*N of every sweep shape (the 16k workload's)


def run_sweep(args):
    """Shape sweep (--sweep): d in {64, 128}, causal and not, N = 1024 ... 32768
    at a fixed token count B*H*N (H = 16, B = tokens / (16 N), or H = 8 at
    N = 32768); per shape the forward and backward main kernels' CUDA-event
    times over --steps calls (L2 flushed before each), one JSON line each.
    Seeded N(0, 1) inputs; TFLOP/s on the causal-halved FLOP count."""
    import torch
    from exact_io_aware_12_gb300 import api, _lib
    from exact_io_aware_12_gb300.workloads import draw, flops_fwd

    dev = torch.device("cuda", 0)
    peaks, src = measured_peaks()
    peak = float(peaks["bf16_tflops"])
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for d in (64, 128):
        for causal in (True, False):
            for N in (1024, 2048, 4096, 8192, 16384, 32768):
                H = 16 if N < 32768 else 8
                B = max(1, SWEEP_TOKENS // (H * N))
                x = draw(B, H, N, d, seed=N + d)
                q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
                tau = 1 / math.sqrt(d)
                o = torch.empty_like(q)
                lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
                dq, dk, dv = (torch.empty_like(q) for _ in range(3))
                ws = torch.empty(api.workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
                for _ in range(args.warmup):
                    api.fwd(q, k, v, causal, tau, out=o, lse=lse)
                    api.bwd(q, k, v, o, do, lse, causal, tau, dq=dq, dk=dk, dv=dv, workspace=ws)
                ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
                for e in sum(ev, []):
                    e.record(stream)
                torch.cuda.synchronize(dev)
                for i in range(args.steps):
                    flush.fill_(float(i))
                    _lib.check(_lib.fa_set_timing_events(ev[i][0].cuda_event, ev[i][1].cuda_event), "timing")
                    api.fwd(q, k, v, causal, tau, out=o, lse=lse)
                    _lib.check(_lib.fa_set_timing_events(ev[i][2].cuda_event, ev[i][3].cuda_event), "timing")
                    api.bwd(q, k, v, o, do, lse, causal, tau, dq=dq, dk=dk, dv=dv, workspace=ws)
                    _lib.check(_lib.fa_set_timing_events(None, None), "timing")
                torch.cuda.synchronize(dev)
                if api.last_device_error(dev) != _lib.FA_OK:
                    raise RuntimeError("kernel watchdog fired in the sweep")
                fms = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
                bms = sum(e[2].elapsed_time(e[3]) for e in ev) / args.steps
                ff = flops_fwd(B, H, N, d, causal)
                print(json.dumps({"sweep": True, "B": B, "H": H, "N": N, "d": d, "causal": causal,
                                  "fwd_ms": round(fms, 4), "fwd_tflops": round(ff / fms / 1e9, 1),
                                  "fwd_frac": round(ff / fms / 1e9 / peak, 4),
                                  "bwd_main_ms": round(bms, 4),
                                  "bwd_tflops": round(2.5 * ff / bms / 1e9, 1),
                                  "bwd_frac": round(2.5 * ff / bms / 1e9 / peak, 4),
                                  "peak_tflops": peak, "peak_source": src}), flush=True)
                del q, k, v, do, o, lse, dq, dk, dv, ws, x


def measure_window(w, q, k, v, do, dev, window, steps, peak):
    """Causal sliding window of `window` keys (fa_fwd_window / fa_bwd_window)."""
    B, H, N, d = w.shape
    ff = window_flops_fwd(B, H, N, d, window)
    return {"window": window, **measure_variant(w, q, k, v, do, dev, steps, peak, ff, window=window)}


def measure_blocks(w, q, k, v, do, dev, steps, peak):
    """Block-sparse causal attention (fa_fwd_blocks / fa_bwd_blocks) with a
    seeded per-head local + global-anchor mask: 4 local blocks (512 tokens),
    2 anchor blocks (256 tokens), 2% random extra blocks."""
    import torch
    from exact_io_aware_12_gb300.workloads import local_global_block_mask

    B, H, N, d = w.shape
    nb = (N + 127) // 128
    m = local_global_block_mask(nb, local=4, anchors=2, heads=B * H, extra=0.02, seed=3)
    ff = blocks_flops_fwd(B, H, N, d, True, m)
    dense = 4.0 * B * H * N * N * d / 2
    mt = torch.from_numpy(m).to(dev).reshape(B, H, nb, nb)
    out = {"mask": "per head: 4 local + 2 anchor blocks of 128, 2% random extra (seed 3)",
           "causal_work_fraction": round(ff / dense, 4),
           **measure_variant(w, q, k, v, do, dev, steps, peak, ff, blocks=mt)}
    # the first two heads alone: few key tiles per SM, where the backward splits the
    # anchor key tiles (seen by every query tile) over helper CTAs
    if B * H > 2:
        w2 = dataclasses.replace(w, B=1, H=2)
        sl = [t.reshape(B * H, N, d)[:2].reshape(1, 2, N, d).contiguous() for t in (q, k, v, do)]
        f2 = blocks_flops_fwd(1, 2, N, d, True, m[:2])
        out["two_heads"] = {"shape": [1, 2, N, d], **measure_variant(w2, *sl, dev, steps, peak, f2,
                                                                     blocks=mt.reshape(B * H, nb, nb)[:2]
                                                                     .reshape(1, 2, nb, nb).contiguous())}
    return out


def measure_decode(dev, steps, peaks, shape=None):
    """Decode step (fa_fwd_decode: split kernel + combine kernel) on the decode
    workload: CUDA-event time around both kernels, and GB/s of the algorithmic
    bytes (Q, K, V read once; O and LSE written once) against the measured HBM
    copy bandwidth.  K and V (2.1 GB) exceed L2; L2 is flushed anyway."""
    import torch
    from exact_io_aware_12_gb300 import api, _lib
    from exact_io_aware_12_gb300.workloads import DECODE_BY_NAME, draw_decode

    w = DECODE_BY_NAME["decode_b8h16_nq1_nk32768_d128"]
    name = w.name
    if shape is not None and shape != (w.B, w.H, w.Nq, w.Nk, w.d):
        # a smaller case of the same recipe (profiling)
        w = type(w)("decode_b%dh%d_nq%d_nk%d_d%d" % shape, *shape, w.causal, w.seed)
        name = w.name
    x = draw_decode(w.B, w.H, w.Nq, w.Nk, w.d, w.seed)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    need = api.decode_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(3):
        api.fwd_decode(q, k, v, w.causal, w.tau, out=o, lse=lse, workspace=ws)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for e in sum(ev, []):
        e.record(stream)
    torch.cuda.synchronize(dev)
    for i in range(steps):
        flush.fill_(float(i))
        _lib.check(_lib.fa_set_timing_events(ev[i][0].cuda_event, ev[i][1].cuda_event), "timing")
        api.fwd_decode(q, k, v, w.causal, w.tau, out=o, lse=lse, workspace=ws)
        _lib.check(_lib.fa_set_timing_events(None, None), "timing")
    torch.cuda.synchronize(dev)
    if api.last_device_error(dev) != _lib.FA_OK:
        raise RuntimeError("kernel watchdog fired in the decode leg")
    ms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    nbytes = 2 * (q.numel() + k.numel() + v.numel() + o.numel()) + 4 * lse.numel()
    gbs = nbytes / (ms / 1e3) / 1e9
    peak = float(peaks["hbm_gbs"])
    return {"workload": name, "steps": steps, "ms": round(ms, 4),
            "bytes": nbytes, "gbs": round(gbs, 1), "peak_gbs": peak,
            "frac": round(gbs / peak, 4), "bound": "hbm",
            "kernels": "fa_decode_split_kernel" + (" + fa_decode_combine_kernel" if need else ""),
            "traffic": profiled_traffic("decode_split")}


def measure_fp8(w, dev, steps, peak_bf16):
    """FP8 forward (fa_fwd_fp8) on the same shape with seeded e4m3 inputs
    (per-tensor scale amax / 448): CUDA-event time of the kernel and TFLOP/s on
    the causal count, against the fp8 peak = measured bf16 peak x 2 (the
    nominal dense fp8 / bf16 ratio, 4.5 / 2.25 PFLOP/s)."""
    import torch
    from exact_io_aware_12_gb300 import api, _lib
    from exact_io_aware_12_gb300.workloads import draw_fp8, flops_fwd

    B, H, N, d = w.shape
    x = draw_fp8(B, H, N, d, w.seed)
    q8, k8, v8 = (x[n].to(dev) for n in ("q8", "k8", "v8"))
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    sc = (x["q_scale"], x["k_scale"], x["v_scale"])
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(3):
        api.fwd_fp8(q8, k8, v8, *sc, w.causal, w.tau, out=o, lse=lse)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for e in sum(ev, []):
        e.record(stream)
    torch.cuda.synchronize(dev)
    for i in range(steps):
        flush.fill_(float(i))
        _lib.check(_lib.fa_set_timing_events(ev[i][0].cuda_event, ev[i][1].cuda_event), "timing")
        api.fwd_fp8(q8, k8, v8, *sc, w.causal, w.tau, out=o, lse=lse)
        _lib.check(_lib.fa_set_timing_events(None, None), "timing")
    torch.cuda.synchronize(dev)
    if api.last_device_error(dev) != _lib.FA_OK:
        raise RuntimeError("kernel watchdog fired in the fp8 leg")
    ms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    ff = flops_fwd(B, H, N, d, w.causal)
    peak = 2.0 * peak_bf16
    tf = ff / ms / 1e9
    return {"steps": steps, "fwd": {"ms": round(ms, 4), "tflops": round(tf, 2),
                                    "frac": round(tf / peak, 4)},
            "peak_tflops": peak, "peak_source": "measured bf16 burst x 2 (nominal fp8/bf16 ratio)",
            "dtype": "e4m3 in, bf16 O", "traffic": profiled_traffic("fwd_fp8")}


def run_e2e(args, w, x, dev, f_step):
    """Same step through the C ABI with host buffers (the library's native host
    pipeline, fa_host_pipeline_*, via api.HostPipeline): every step copies its
    pinned host inputs in and its outputs (O, LSE, dQ, dK, dV) back, inside the
    timing; the copies of neighbouring steps overlap the kernels, two device
    buffer sets deep."""
    import torch
    from exact_io_aware_12_gb300 import api

    world, _, _ = dist_env()
    B, H, N, d = w.shape
    hin = {n: x[n].pin_memory() for n in ("q", "k", "v", "do")}
    dq_, dk_, dv_, o_ = (torch.empty(w.shape, dtype=torch.bfloat16).pin_memory() for _ in range(4))
    lse_ = torch.empty((B, H, N), dtype=torch.float32).pin_memory()

    # the public API's host-buffer pipeline: each step copies its inputs in and
    # its results out; neighbouring steps' copies overlap each other's kernels
    pipe = api.HostPipeline(B, H, N, d, w.causal, w.tau, device=dev)

    def step():
        pipe.step(hin["q"], hin["k"], hin["v"], hin["do"], o_, lse_, dq_, dk_, dv_)

    for _ in range(max(1, args.warmup)):
        step()
    pipe.synchronize()
    barrier(world, dev)
    s = pipe.mark()     # after the warm-up; the first timed copy starts after it
    for _ in range(args.steps):
        step()
    e = pipe.mark()     # after the last timed step's copies out
    e.synchronize()
    t = reduce_max(s.elapsed_time(e) / 1e3, world, dev)
    pipe.close()
    h2d = sum(t_.numel() * t_.element_size() for t_ in hin.values())
    d2h = sum(t_.numel() * t_.element_size() for t_ in (o_, lse_, dq_, dk_, dv_))
    return {"value": round(aggregate_value(f_step, args.steps, world, t), 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(t * 1e3 / args.steps, 4)}


# ------------------------------------------------------------ CPU oracle ----
def oracle_sample(w, budget_s: float):
    """Times the fp64 oracle on a bounded sample of the workload: the forward on
    sampled query rows of every head and the backward on a causal prefix.
    Returns (flops, seconds, description)."""
    import numpy as np
    import oracle
    from exact_io_aware_12_gb300.workloads import flops_fwd, flops_bwd, make_inputs

    x = make_inputs(w)
    B, H, N, d = w.shape
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "do"))
    # calibrate: a few rows, then size the sample to ~budget/2 for each half
    rng = np.random.default_rng(7)
    probe_rows = (np.arange(B * H) * N)[:, None] + rng.integers(0, N, size=(B * H, 2))
    t0 = time.perf_counter()
    oracle.fwd_rows(q, k, v, w.tau, w.causal, probe_rows.ravel())
    t_probe = time.perf_counter() - t0
    f_probe = sum(4.0 * d * ((r % N) + 1 if w.causal else N) for r in probe_rows.ravel())
    rate = f_probe / max(t_probe, 1e-6)
    per_row = 4.0 * d * (N / 2 if w.causal else N)
    n_rows = int(max(B * H, min(B * H * N, (budget_s / 2) * rate / per_row)))
    per_head = max(1, n_rows // (B * H))
    rows = ((np.arange(B * H) * N)[:, None] + rng.integers(0, N, size=(B * H, per_head))).ravel()
    t0 = time.perf_counter()
    oracle.fwd_rows(q, k, v, w.tau, w.causal, rows)
    t_f = time.perf_counter() - t0
    f_f = sum(4.0 * d * ((r % N) + 1 if w.causal else N) for r in rows)
    # backward on a prefix sized to the other half of the budget
    n_b = 64
    while n_b * 2 <= N and flops_bwd(B, H, n_b * 2, d, w.causal) / rate * 3 < budget_s / 2:
        n_b *= 2
    sl = lambda a: np.ascontiguousarray(a[:, :, :n_b])
    t0 = time.perf_counter()
    oracle.bwd(sl(q), sl(k), sl(v), sl(do), w.tau, w.causal)
    t_b = time.perf_counter() - t0
    f_b = flops_bwd(B, H, n_b, d, w.causal)
    desc = (f"forward on {rows.size} random query rows ({per_head}/head) + backward on the "
            f"{n_b}-token causal prefix, all {B * H} heads; FLOPs counted as on the GPU")
    return f_f + f_b, t_f + t_b, desc, rows.size / t_f


def run_cpu_baseline(w, budget_s: float):
    """The oracle on the host cores: all of them, then one thread on a quarter
    of the budget. Besides TFLOP/s it reports the forward's query rows per
    second and the time a whole step (forward + backward of the full workload)
    would take at each rate, labelled as extrapolated."""
    import oracle
    from exact_io_aware_12_gb300.workloads import flops_fwd, flops_bwd

    n_all = oracle.num_threads()
    flops, secs, desc, rows_s = oracle_sample(w, budget_s)
    oracle.set_num_threads(1)
    try:
        f1, s1, _, rows_s1 = oracle_sample(w, budget_s / 4)
    finally:
        oracle.set_num_threads(n_all)
    B, H, N, d = w.shape
    full = flops_fwd(B, H, N, d, w.causal) + flops_bwd(B, H, N, d, w.causal)
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": n_all,
            "kind": "oracle", "sample": desc, "seconds": round(secs, 2),
            "fwd_rows_per_s": round(rows_s, 1),
            "single_thread": {"value": round(f1 / s1 / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
                              "fwd_rows_per_s": round(rows_s1, 2), "seconds": round(s1, 2)},
            "extrapolated_full_step_s": {"all_cores": round(full / (flops / secs), 1),
                                         "single_thread": round(full / (f1 / s1), 1)}}


def run_reference(args):
    """The oracle as the reference arm: rank 0 only, host cores."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    w = pick_workload(args)
    per_step = max(1.0, min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, per_step)
    tot_f, tot_s, desc = 0.0, 0.0, ""
    for _ in range(args.steps):
        f, s, desc, _ = oracle_sample(w, per_step)
        tot_f += f
        tot_s += s
    value = tot_f / tot_s / 1e12
    B, H, N, d = w.shape
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_s * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": B, "H": H, "N": N, "d": d, "causal": w.causal},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "kind": "oracle",
                             "cores": oracle.num_threads(), "sample": desc},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--shape", default=None,
                    help="B,H,N,d,causal: a smaller same-recipe case (profiling only)")
    ap.add_argument("--cpu-seconds", type=float, default=20.0,
                    help="CPU time budget of the oracle baseline sample")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--window", type=int, default=4096,
                    help="also time the causal sliding-window kernels with this window (0: skip)")
    ap.add_argument("--no-blocks", dest="blocks", action="store_false",
                    help="skip the block-sparse leg")
    ap.add_argument("--no-decode", dest="decode", action="store_false",
                    help="skip the decode leg")
    ap.add_argument("--no-fp8", dest="fp8", action="store_false", help="skip the FP8 leg")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip timing the other named workloads")
    ap.add_argument("--clock-csv", default=None,
                    help="keep the nvidia-smi clock samples in this file (default: a temp file)")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the bench line: forward/backward TFLOP/s over d, causal and N")
    ap.add_argument("--decode-shape", default="8,16,1,32768,128",
                    help="B,H,Nq,Nk,d of the decode leg (a smaller case: profiling only)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, _, _ = dist_env()
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world} (launch N>1 with torchrun)")
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

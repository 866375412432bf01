#!/usr/bin/env python
"""Benchmark of the Linformer attention forward on GB300: prints ONE JSON line.

A step is one pass of the whole forward (projection + compressed attention) over
one batch of the long-sequence workload: b=16, h=12, n=4096, d=64, k=256, one
layerwise-shared E = F, bf16 in and out, synthetic N(0,1) inputs and N(0,1/k)
projections.  Throughput is b*h*n tokens per second.

  python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference]

--impl ours (default): inputs resident in HBM, K steps timed with CUDA events on
the launching stream, barrier + synchronize on both sides, max over ranks (each
rank runs its own full batch: weak scaling, no collective on the data path).
Also reported: the dominant kernel against its roofline (per-kernel CUDA events
from a second, profiled pass of K steps), the end-to-end rate through the
host-buffer entry point (copies in the timed region), SM clocks sampled by
nvidia-smi during the run, and the fp64 oracle timed on the host cores on a
bounded sample of the same workload.

--impl reference: the fp64 CPU oracle on the host cores, each step a bounded
sample (whole batches) of the same workload; rank 0 only.

--approx-error: not a benchmark step but the method's own approximation error
against exact softmax attention, over n and k on the same synthetic inputs (one
JSON line with a row per (n, k)); see approx_error_rows().
"""
from __future__ import annotations

import argparse
import csv
import dataclasses
import io
import json
import os
import signal
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from rank_linear_complexity_gb300.workloads import HEADLINE, WORKLOADS, workload_inputs  # noqa

METRIC = "Linformer attn fwd Mtokens/s at n=4096,k=256 bf16; % of HBM/TC roofline"
UNIT = "Mtokens/s"
L2_BYTES = 129e6


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def algorithmic(w):
    """Compulsory bytes and algorithmic FLOPs of the forward, and per kernel."""
    es = 4 if w.dtype == 0 else 2
    os_ = 2 if w.dtype == 1 else 4
    units = w.units
    qkv_each = units * w.n * w.d * es
    groups = w.h if w.share_mode in (0, 1) else 1
    n_proj = 2 if w.share_mode in (0, 2) else 1
    ef = groups * n_proj * w.k * w.n * es
    o_bytes = units * w.n * w.d * os_
    flop_proj = 4.0 * w.n * w.k * w.d * units
    flop_attn = 4.0 * w.n * w.k * w.d * units
    return {
        "total_bytes": 3 * qkv_each + ef + o_bytes,
        "total_flop": flop_proj + flop_attn,
        "project": {"bytes": 2 * qkv_each + ef, "flop": flop_proj},
        "attend": {"bytes": qkv_each + o_bytes, "flop": flop_attn},
    }


def valid_rows_algorithmic(w, lengths):
    """Compulsory bytes and FLOPs over the valid rows only (ragged batches): Q, K, V and
    the FLOPs of rows t < L_b, all of O (padded rows are written as zero), E and F once."""
    es = 4 if w.dtype == 0 else 2
    os_ = 2 if w.dtype == 1 else 4
    rows = sum(min(max(int(L), 0), w.n) for L in lengths) * w.h
    groups = w.h if w.share_mode in (0, 1) else 1
    n_proj = 2 if w.share_mode in (0, 2) else 1
    return {"total_bytes": 3 * rows * w.d * es + w.units * w.n * w.d * os_
                           + groups * n_proj * w.k * w.n * es,
            "total_flop": 8.0 * rows * w.k * w.d}


def flushed_median(step, stream, steps: int, scratch_bytes: int = 1 << 30):
    """Per-step device time with L2 flushed before every step (a 1 GB write between the
    steps, outside the events): median and spread over `steps` steps, in ms."""
    scratch = torch.empty(scratch_bytes, dtype=torch.uint8, device=stream.device)
    pairs = []
    for i in range(steps):
        scratch.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        pairs.append((a, b))
    torch.cuda.synchronize()
    ms = sorted(a.elapsed_time(b) for a, b in pairs)
    del scratch
    return {"median_ms": statistics.median(ms), "min_ms": ms[0], "max_ms": ms[-1],
            "steps": steps, "flush": f"{scratch_bytes >> 20} MB write before each step"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the GPU works.  Each sample is
    stamped with the host clock when it arrives, so that windows of the run (the timed
    steps, the sustained pass) can be summarised separately."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int, interval_ms: int = 50):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.thread = None
        self.samples = []  # (host monotonic time, row)

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                row = next(csv.reader([line]), [])
                if len(row) >= 9:
                    self.samples.append((time.monotonic(), row))

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def wait_first(self, timeout_s: float = 5.0):
        """Blocks until the first sample has arrived (nvidia-smi takes a moment to start)."""
        t0 = time.monotonic()
        while self.proc is not None and not self.samples and time.monotonic() - t0 < timeout_s:
            time.sleep(0.01)

    def stop(self):
        if self.proc is not None:
            self.proc.send_signal(signal.SIGTERM)
            try:
                self.proc.wait(timeout=10)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=10)

    def summary(self, t0: float = None, t1: float = None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        sm, smax, power, reasons = [], [], [], set()
        for t, r in self.samples:
            if (t0 is not None and t < t0) or (t1 is not None and t > t1):
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                power.append(float(r[3]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def sustained_pass(step, stream, seconds: float, batch: int = 100):
    """Back-to-back steps for at least `seconds` (batches of `batch` steps, synchronised
    after each), timed with CUDA events; returns (ms per step, steps, host t0, host t1)."""
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.monotonic()
    ev0.record(stream)
    steps = 0
    while True:
        for _ in range(batch):
            step()
        steps += batch
        torch.cuda.synchronize()
        if time.monotonic() - t0 >= seconds:
            break
    ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.monotonic()
    return ev0.elapsed_time(ev1) / steps, steps, t0, t1


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(tokens_per_rank: int, ms_per_step_max: float, world: int) -> float:
    """Whole-job Mtokens/s: every rank's tokens over the slowest rank's step time."""
    return world * tokens_per_rank / (ms_per_step_max * 1e-3) / 1e6


def oracle_sample(w, x, units: int, nthreads: int = 0):
    """Time the oracle on the first `units` units (batch-major); returns
    (seconds, tokens, threads used)."""
    from oracle import oracle as orc
    units = max(1, min(units, w.units))
    if units < w.h:
        bsl, hsl = slice(0, 1), slice(0, units)
    else:
        bsl, hsl = slice(0, units // w.h), slice(0, w.h)
        units = (units // w.h) * w.h
    per_head = w.share_mode in (0, 1)
    E = x["E"][hsl] if per_head else x["E"]
    F = None if x["F"] is None else (x["F"][hsl] if per_head else x["F"])
    args = [x["Q"][bsl, hsl], x["K"][bsl, hsl], x["V"][bsl, hsl], E, F,
            None if x["lengths"] is None else x["lengths"][bsl]]
    t0 = time.perf_counter()
    _, used = orc.linformer_fwd(*args, w.share_mode, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return dt, units * w.n, used


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = HEADLINE
    from oracle import oracle as orc
    orc.build()
    x = workload_inputs(w)
    # Size each step so that warm-up + timed steps take about REF_BUDGET_S seconds.
    t_unit, _, _ = oracle_sample(w, x, 1)
    per_step = args.ref_budget_s / (args.steps + args.warmup)
    units = int(max(1, min(w.units, per_step / max(t_unit, 1e-6))))
    for _ in range(args.warmup):
        oracle_sample(w, x, units)
    times, used, tokens = [], 1, 0
    for _ in range(args.steps):
        dt, tokens, used = oracle_sample(w, x, units)
        times.append(dt)
    total = sum(times)
    value = tokens * len(times) / total / 1e6
    sample = (f"{tokens // w.n} of {w.units} units ({tokens} tokens) per step, fp64 oracle, "
              f"OpenMP on {used} threads of {host_cores()} host cores")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": w.describe(),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_ours(args):
    import rank_linear_complexity_gb300.linformer as lf
    from rank_linear_complexity_gb300 import build as libbuild
    libbuild.build()
    world, rank, local = dist_setup(args.gpus)
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload] if args.workload is not None else HEADLINE
    if args.batch:
        w = dataclasses.replace(w, b=args.batch, name=f"{w.name}_b{args.batch}")
    x = workload_inputs(w)
    g = {kk: (v.to(dev) if v is not None else None) for kk, v in x.items()}
    out_dt = torch.bfloat16 if w.dtype == 1 else torch.float32
    O = torch.empty((w.b, w.h, w.n, w.d), dtype=out_dt, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        st = lf.linformer_attn_fwd(g["Q"], g["K"], g["V"], g["E"], g["F"], g["lengths"], O,
                                   w.b, w.h, w.n, w.d, w.k, w.share_mode, w.dtype, stream)
        if st != 0:
            raise lf.LinformerError(st, "linformer_attn_fwd")

    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    sampler.start()
    sampler.wait_first()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if lf.linformer_debug_read_device_status(stream) != 0:
        raise RuntimeError("device status set during warm-up")

    # --- headline: K steps, CUDA events on the launching stream -----------------------
    launches0 = lf.linformer_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_timed0 = time.monotonic()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_timed1 = time.monotonic()
    barrier(world)
    launches = lf.linformer_launch_count() - launches0
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), world)
    ms_step = ms_total / args.steps

    # --- clocks under load: a sustained pass of back-to-back forwards right after the
    # timed steps (those last milliseconds, less than the sampling interval) -----------
    sustained = None
    if args.sustain_s > 0:
        s_ms, s_steps, s_t0, s_t1 = sustained_pass(step, stream, args.sustain_s)
        sustained = {"ms_per_step": s_ms, "steps": s_steps, "seconds": s_t1 - s_t0,
                     "clocks": sampler.summary(s_t0, s_t1)}
    sampler.stop()
    timed_clocks = sampler.summary(t_timed0, t_timed1)
    if sustained and sustained["clocks"]["samples"]:
        clocks = dict(sustained["clocks"], window="sustained pass of back-to-back forwards "
                      "directly after the timed steps", timed_region_samples=timed_clocks["samples"])
    else:
        clocks = dict(sampler.summary(), window="whole run")
    value = aggregate_throughput(w.tokens, ms_step, world)

    # --- per-kernel durations: a second pass of K steps with library events -----------
    lf.linformer_profile_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    lf.linformer_profile_enable(False)
    per_kernel = lf.linformer_profile_collect()
    if lf.linformer_debug_read_device_status(stream) != 0:
        raise RuntimeError("device status set during the timed region")

    peaks = load_peaks()
    alg = algorithmic(w)
    kernels = {}
    for name, (ms, cnt) in per_kernel.items():
        part = "project" if "project" in name else "attend"
        avg_s = ms / cnt * 1e-3
        t_mem = alg[part]["bytes"] / (peaks["hbm_gbs"] * 1e9)
        t_tc = alg[part]["flop"] / (peaks["bf16_tflops"] * 1e12)
        bound = "hbm" if t_mem >= t_tc else "tensor"
        if bound == "hbm":
            achieved, peak, unit = alg[part]["bytes"] / avg_s / 1e9, peaks["hbm_gbs"], "GB/s"
        else:
            achieved, peak, unit = alg[part]["flop"] / avg_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
        kernels[name] = {"avg_us": avg_s * 1e6, "launches": cnt, "bound": bound,
                         "achieved": achieved, "peak": peak, "unit": unit,
                         "frac": achieved / peak}
    dominant = max(kernels, key=lambda k: kernels[k]["avg_us"]) if kernels else None
    mhz = clocks.get("sm_mhz")
    for kd in kernels.values():  # clock-normalised duration, comparable across boxes
        kd["kcycles_at_median_sm_clock"] = kd["avg_us"] * mhz / 1e3 if mhz else None
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if dominant and os.path.exists(tfile):
        try:
            # dram bytes per launch from an ncu capture, keyed by workload then kernel
            traffic = json.load(open(tfile)).get(w.name, {}).get(dominant)
        except Exception:
            traffic = None
    roofline = None
    if dominant:
        kd = kernels[dominant]
        roofline = {"kernel": dominant, "bound": kd["bound"], "achieved": kd["achieved"],
                    "peak": kd["peak"], "unit": kd["unit"], "frac": kd["frac"],
                    "traffic": traffic, "peak_source": peaks["source"] + " (burst)"}
    t_roof = max(alg["total_bytes"] / (peaks["hbm_gbs"] * 1e9),
                 alg["total_flop"] / (peaks["bf16_tflops"] * 1e12))
    path_frac = t_roof / (ms_step * 1e-3)
    valid_frac = None
    if x["lengths"] is not None:
        va = valid_rows_algorithmic(w, x["lengths"].tolist())
        valid_frac = max(va["total_bytes"] / (peaks["hbm_gbs"] * 1e9),
                         va["total_flop"] / (peaks["bf16_tflops"] * 1e12)) / (ms_step * 1e-3)

    # --- L2 flushed before every step: median of up to 50 single-step timings ---------
    flushed = None
    if not args.no_flush_pass:
        try:
            flushed = flushed_median(step, stream, max(1, min(args.steps, 50)))
            flushed["value"] = aggregate_throughput(w.tokens, flushed["median_ms"], world)
        except (RuntimeError, torch.cuda.OutOfMemoryError) as e:  # no room for the scratch
            flushed = {"unavailable": str(e).splitlines()[0][:200]}
        if lf.linformer_debug_read_device_status(stream) != 0:
            raise RuntimeError("device status set during the flushed pass")

    # --- end to end through the host-buffer entry point -------------------------------
    e2e = None
    if not args.no_e2e:
        pin = {kk: (v.pin_memory() if v is not None else None) for kk, v in x.items()}
        Oh = torch.empty((w.b, w.h, w.n, w.d), dtype=out_dt).pin_memory()

        def host_step():
            st = lf.linformer_attn_fwd_host(pin["Q"], pin["K"], pin["V"], pin["E"], pin["F"],
                                            pin["lengths"], Oh, w.b, w.h, w.n, w.d, w.k,
                                            w.share_mode, w.dtype, stream)
            if st != 0:
                raise lf.LinformerError(st, "linformer_attn_fwd_host")

        for _ in range(min(3, args.warmup)):
            host_step()
        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            host_step()
        dt = max_over_ranks(time.perf_counter() - t0, world)
        h2d = sum(v.numel() * v.element_size() for v in pin.values() if v is not None)
        e2e = {"value": world * w.tokens * e2e_steps / dt / 1e6, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": Oh.numel() * Oh.element_size(),
               "steps": e2e_steps, "ms_per_step": 1e3 * dt / e2e_steps}

    # --- CPU baseline: the oracle on a bounded sample, rank 0 at N = 1 -----------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, tokens, used = oracle_sample(w, x, args.cpu_units)
        cpu = {"value": tokens / dt / 1e6, "unit": UNIT, "cores": used, "kind": "oracle",
               "sample": f"first {tokens // w.n} of {w.units} units ({tokens} tokens), one pass, "
                         f"{dt:.2f} s wall, {used} OpenMP threads on {host_cores()} host cores"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype != 0 else "f32", "data": "synthetic",
            "config": dict(w.describe(), parallelism=f"replicas{world}",
                           l2=("no flush: inputs larger than L2 "
                               f"(Q+K+V {3 * w.tokens * w.d * 2 / 1e6:.0f} MB vs "
                               f"{L2_BYTES / 1e6:.0f} MB L2)")),
            "tflops": alg["total_flop"] / (ms_step * 1e-3) / 1e12,
            "path_roofline_frac": path_frac,
            "path_roofline_frac_valid_rows": valid_frac,
            "l2_flushed": flushed,
            "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches, "clocks": clocks, "sustained": sustained,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# --- approximation error of the method (pages: "Linformer ... 요약 설명", sections
# "Self-Attention is Low Rank" and "Model": the first theorem, a random projection of
# the attention output via the Johnson-Lindenstrauss lemma, rank of order log n for a
# fixed error; the second, a projection size that depends on the head dimension and
# the error but not on n).  Exact references in fp64 with plain PyTorch.

def full_attention64(Q, K, V):
    """P = softmax(Q K^T / sqrt(d)) and O = P V per unit, fp64 ([..., n, d] inputs)."""
    Q, K, V = Q.double(), K.double(), V.double()
    P = torch.softmax(Q @ K.transpose(-1, -2) / (Q.shape[-1] ** 0.5), dim=-1)
    return P, P @ V


def linformer64(Q, K, V, R):
    """The method in exact arithmetic with E = F = R (k x n): softmax(Q (R K)^T / sqrt(d)) (R V)."""
    Q, K, V, R = Q.double(), K.double(), V.double(), R.double()
    Kb, Vb = R @ K, R @ V
    return torch.softmax(Q @ Kb.transpose(-1, -2) / (Q.shape[-1] ** 0.5), dim=-1) @ Vb


def approx_errors(Q, K, V, R, O_kernel=None) -> dict:
    """Errors for one (n, k) over units [..., n, d]:
    - jl_t1: the first theorem's construction P R^T R V against P V, each entry divided
      by ||p_i|| ||v_c|| (the scale of the lemma's guarantee), RMS over entries;
    - rel_lin / jl_lin: the method's output against P V, relative in Frobenius norm and
      normalised as jl_t1;
    - kernel_dev: the library's output against the method in fp64 (relative Frobenius)."""
    P, O = full_attention64(Q, K, V)
    Rd, Vd = R.double(), V.double()
    scale = P.norm(dim=-1, keepdim=True) * Vd.norm(dim=-2, keepdim=True)
    T1 = (P @ Rd.transpose(-1, -2)) @ (Rd @ Vd)
    OL = linformer64(Q, K, V, R)
    out = {"jl_t1": float((((T1 - O) / scale) ** 2).mean().sqrt()),
           "rel_lin": float((OL - O).norm() / O.norm()),
           "jl_lin": float((((OL - O) / scale) ** 2).mean().sqrt())}
    if O_kernel is not None:
        out["kernel_dev"] = float((O_kernel.double() - OL).norm() / OL.norm())
    return out


def approx_error_rows(ns, ks, units=4, device="cuda:0"):
    """One row per (n, k < n): inputs as the workloads draw them (Q, K, V ~ N(0,1),
    one layerwise E = F ~ N(0,1/k), bf16), the library's output in fp32."""
    import rank_linear_complexity_gb300.linformer as lf
    from rank_linear_complexity_gb300.workloads import BF16, LAYERWISE, make_inputs
    rows = []
    for n in ns:
        for k in ks:
            if k >= n:
                continue
            x = make_inputs(1, units, n, 64, k, LAYERWISE, BF16, seed=4321 + n)
            g = {kk: (v.to(device) if v is not None else None) for kk, v in x.items()}
            O = lf.attention(g["Q"], g["K"], g["V"], g["E"], None, None, LAYERWISE, out_fp32=True)
            torch.cuda.synchronize()
            r = approx_errors(g["Q"][0], g["K"][0], g["V"][0], g["E"], O[0])
            rows.append({"n": n, "k": k, **{kk: round(v, 5) for kk, v in r.items()}})
            del g, O
            torch.cuda.empty_cache()
    return rows


def run_approx_error(args):
    rows = approx_error_rows([512, 1024, 2048, 4096], [32, 64, 128, 256])
    print(json.dumps({"experiment": "approx_error", "units": 4, "d": 64,
                      "inputs": "Q, K, V ~ N(0,1), one E = F ~ N(0,1/k), bf16 (workload generator)",
                      "rows": rows}))
    return 0


BWD_SHAPE = dict(b=16, h=12, n=4096, d=64, k=256, share_mode=3)  # LAYERWISE


def bwd_flop(b, h, n, d, k, **_):
    """Algorithmic FLOPs of the backward: eleven n x k x d products per unit (Kbar, Vbar
    recomputed; S, dP, dVbar, dQ, dKbar, dK, dV and the E and F terms), 2 FLOPs each."""
    return 22.0 * b * h * n * k * d


def run_backward(args):
    """fp32 backward (linformer_attn_bwd) at n=4096, k=256, one shared projection."""
    import rank_linear_complexity_gb300.linformer as lf
    from rank_linear_complexity_gb300 import build as libbuild
    from rank_linear_complexity_gb300.workloads import make_inputs, output_gradient
    libbuild.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    c = dict(BWD_SHAPE, b=args.batch) if args.batch else BWD_SHAPE
    b, h, n, d, k, mode = c["b"], c["h"], c["n"], c["d"], c["k"], c["share_mode"]
    x = make_inputs(b, h, n, d, k, mode, 0, seed=77)
    dO_h = output_gradient(b, h, n, d, seed=78)
    g = {kk: (v.to(dev) if v is not None else None) for kk, v in x.items()}
    dO = dO_h.to(dev)
    dQ, dK, dV = torch.empty_like(g["Q"]), torch.empty_like(g["K"]), torch.empty_like(g["V"])
    dE = torch.empty_like(g["E"])
    stream = torch.cuda.current_stream(dev)

    def step():
        st = lf.linformer_attn_bwd(g["Q"], g["K"], g["V"], g["E"], None, g["lengths"], dO, dQ,
                                   dK, dV, dE, None, b, h, n, d, k, mode, 0, stream)
        if st != 0:
            raise lf.LinformerError(st, "linformer_attn_bwd")

    steps = max(1, min(args.steps, 50))
    sampler = ClockSampler(0)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    launches0 = lf.linformer_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    clocks = sampler.summary()
    launches = lf.linformer_launch_count() - launches0
    if lf.linformer_debug_read_device_status(stream) != 0:
        raise RuntimeError("device status set during the timed region")
    ms_step = ev0.elapsed_time(ev1) / steps
    tokens = b * h * n
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    max_mhz = clocks.get("sm_max_mhz") or 2070.0
    fma_peak = sms * 128 * 2 * max_mhz * 1e6 / 1e12  # fp32 FMA lanes x 2 FLOPs x clock
    achieved = bwd_flop(**c) / (ms_step * 1e-3) / 1e12
    # every fp32 product runs as three bf16 tensor-core products (hi.hi + hi.lo + lo.hi)
    tc_achieved, tc_peak = 3.0 * achieved, load_peaks()["bf16_tflops_sustained"]

    # the oracle on a bounded sample of the same workload (units of one batch row)
    from oracle import backward as bw
    units = min(h, 12)
    t0 = time.perf_counter()
    bw.linformer_bwd(x["Q"][:1, :units], x["K"][:1, :units], x["V"][:1, :units], x["E"], None,
                     None, dO_h[:1, :units], mode)
    cpu_s = time.perf_counter() - t0
    line = {
        "experiment": "backward", "metric": "Linformer attn bwd Mtokens/s at n=4096,k=256 fp32",
        "value": tokens / (ms_step * 1e-3) / 1e6, "unit": UNIT, "n_gpus": 1, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"bwd_b{b}_h12_n4096_d64_k256_layerwise", **c,
                   "l2": f"inputs of {4 * b * h * n * d * 4 / 1e6:.0f} MB (Q, K, V, dO)"},
        "roofline": {"kernel": "backward (all launches)", "bound": "tensor",
                     "achieved": tc_achieved, "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": tc_achieved / tc_peak,
                     "peak_source": "measured bf16, sustained (MEASURED_PEAKS.json)",
                     "counts": "three bf16 products per fp32 product (22 n k d FLOPs per unit x 3)"},
        "fp32_equivalent": {"achieved": achieved, "unit": "TFLOP/s",
                            "fma_peak": fma_peak, "frac_of_fma_peak": achieved / fma_peak,
                            "fma_peak_source": f"derived: {sms} SMs x 128 fp32 lanes x 2 x {max_mhz} MHz"},
        "gpu_launches": launches,
        "clocks": {kk: clocks.get(kk) for kk in ("sm_mhz", "sm_max_mhz", "reasons")},
        "cpu_baseline": {"value": units * n / cpu_s / 1e6, "unit": UNIT,
                         "cores": host_cores(), "kind": "oracle",
                         "sample": f"{units} of {b * h} units, fp64 numpy oracle"},
    }
    print(json.dumps(line))
    return 0


# The pages' single-GPU inference table: n in {512, 4096, 65536}, k in {128, 256},
# RoBERTa-base heads (h = 12, d = 64).
TABLE_POINTS = [(512, 128), (512, 256), (4096, 128), (4096, 256), (65536, 128), (65536, 256)]
TABLE_H, TABLE_D = 12, 64
V100_BYTES = 16e9  # the pages' GPU capacity


def time_call(fn, steps, warmup, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def run_inference_table(args):
    """Time and largest batch of Linformer attention against dense softmax attention
    (attention only, one layer, h = 12, d = 64), at the pages' (n, k) points.  Memory per
    sequence = its Q, K, V, O plus the workspace the call draws from the library pool
    (measured high-water mark ÷ sequences); the largest batch is what fits in a capacity
    after E and F; memory saving = ratio of largest batches, as the pages define it."""
    import rank_linear_complexity_gb300.linformer as lf
    from rank_linear_complexity_gb300 import build as libbuild
    from rank_linear_complexity_gb300.workloads import make_inputs
    libbuild.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    hbm = torch.cuda.get_device_properties(dev).total_memory
    h, d = TABLE_H, TABLE_D
    rows = []

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    f32_peak = sms * 128 * 2 * 2070e6 / 1e12  # fp32 FMA lanes x 2 FLOPs x max clock
    bf16_peak = load_peaks()["bf16_tflops"]

    def measure(fn, seqs, io_bytes_per_seq, fixed_bytes, steps, flop_per_seq, peak):
        torch.cuda.synchronize()
        lf.linformer_pool_peak_bytes(reset=True)
        fn()
        torch.cuda.synchronize()
        ws = lf.linformer_pool_peak_bytes()
        ms = time_call(fn, steps, 2, stream)
        per_seq = io_bytes_per_seq + ws / seqs
        tflops = flop_per_seq / (ms / seqs * 1e-3) / 1e12
        return {"ms_per_seq": ms / seqs, "bytes_per_seq": per_seq,
                "tflops": tflops, "frac_of_peak": tflops / peak,
                "max_batch_16GB": int(max(0, V100_BYTES - fixed_bytes) // per_seq),
                "max_batch_hbm": int(max(0, hbm - fixed_bytes) // per_seq)}

    for n, k in TABLE_POINTS:
        row = {"n": n, "k": k}
        # dense fp32: the n x n scores of every unit; one head at n = 65536 (17 GB)
        bd, hd = (16, h) if n <= 512 else ((1, h) if n <= 4096 else (1, 1))
        x = make_inputs(bd, hd, n, d, 1, 0, 0, seed=n)
        Q, K, V = (x[c].to(dev) for c in "QKV")
        O = torch.empty_like(Q)
        seqs = bd * hd / h
        fn = lambda: lf.dense_attention(Q, K, V, out=O)
        row["dense_f32"] = measure(fn, seqs, 4 * h * n * d * 4, 0, 3 if n > 4096 else 10,
                                   4.0 * h * n * n * d, f32_peak)
        del Q, K, V, O, x
        # Linformer, one E = F shared by all heads (layerwise), fp32 and bf16 inputs
        bl = 16 if n <= 4096 else 1
        for name, dt in (("linformer_f32", 0), ("linformer_bf16", 1)):
            x = make_inputs(bl, h, n, d, k, 3, dt, seed=n + k)
            g = {c: (v.to(dev) if v is not None else None) for c, v in x.items()}
            O = torch.empty_like(g["Q"])
            es = 4 if dt == 0 else 2
            fn = lambda: lf.attention(g["Q"], g["K"], g["V"], g["E"], None, None, 3, out=O)
            row[name] = measure(fn, bl, 4 * h * n * d * es, k * n * es, 10, 8.0 * h * n * k * d,
                                f32_peak if dt == 0 else bf16_peak)
            del g, O, x
        for name in ("linformer_f32", "linformer_bf16"):
            row[name]["speedup_vs_dense_f32"] = (row["dense_f32"]["ms_per_seq"] /
                                                 row[name]["ms_per_seq"])
            for cap in ("16GB", "hbm"):
                den = row["dense_f32"][f"max_batch_{cap}"]
                row[name][f"memory_saving_{cap}"] = (row[name][f"max_batch_{cap}"] / den
                                                     if den else None)
        rows.append(row)
        torch.cuda.empty_cache()
    print(json.dumps({"experiment": "inference_table", "h": h, "d": d,
                      "share_mode": "layerwise (one E = F)", "hbm_bytes": hbm,
                      "note": "attention only, one layer; dense keeps the n x n scores of "
                              "every head in device memory; ms per sequence of 12 heads; "
                              "algorithmic FLOPs 4 n^2 d (dense), 8 n k d (Linformer) per "
                              "head; peaks: fp32 derived from SMs x 128 lanes x 2 x 2070 MHz "
                              "(f32 rows), measured bf16 (bf16 rows)",
                      "rows": rows}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=None,
                    help="index into the workload table (default: the n=4096, k=256 case)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the batch size (smaller cases for profiling)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-units", type=int, default=48,
                    help="units of the workload the CPU-baseline oracle pass covers")
    ap.add_argument("--ref-budget-s", type=float, default=90.0,
                    help="--impl reference: seconds for all warm-up + timed steps")
    ap.add_argument("--sustain-s", type=float, default=2.0,
                    help="seconds of back-to-back forwards after the timed steps, for the "
                         "clock record (0: skip)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-flush-pass", action="store_true",
                    help="skip the extra pass timed with L2 flushed before every step")
    ap.add_argument("--approx-error", action="store_true",
                    help="report the method's approximation error over n and k instead")
    ap.add_argument("--backward", action="store_true",
                    help="time the fp32 backward at n=4096, k=256 instead")
    ap.add_argument("--inference-table", action="store_true",
                    help="Linformer against dense attention: time and largest batch")
    args = ap.parse_args()
    if args.approx_error:
        return run_approx_error(args)
    if args.inference_table:
        return run_inference_table(args)
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps, always
    if args.backward:
        return run_backward(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

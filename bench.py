#!/usr/bin/env python3
"""Benchmark of the fused FP8 lightning indexer + exact top-k on GB300.

Metric: indexer+top-k query tokens/s -- query tokens whose top-k key set is produced per second
by dsa_index_topk (plan + run) -- on the DeepSeek-V3.2-shaped prefill: T = N = 8192 tokens,
H = 64 index heads, D = 128, causal windows, top-k 2048, synthetic e4m3 inputs (seed 2).

One step = one pass of the whole hot path over the workload: the planner kernel and the fused
scorer + selector kernel, inputs resident in HBM.  L2 (129 MB) is flushed before every timed step,
outside the timed events: a 256 MB buffer is written, then a second 256 MB buffer is read, so the
step starts with none of its inputs in L2 and no dirty lines left for it to write back (a write
alone leaves ~129 MB of dirty lines whose write-back lands inside the next timed kernel: 13 us on
a 260 MB key stream).  Times are CUDA events on the launching stream.

Also reported on the same JSON line:
  roofline      the fused kernel alone: algorithmic FP8 FLOPs (2 H D x in-window pairs) per
                launch / its mean event time, against the dense FP8 peak (2 x the measured bf16
                burst peak, the nominal fp8 / bf16 ratio);
  phases        the unfused scorer (FP8 TFLOP/s) and the unfused selector (GB/s of algorithmic
                bytes: in-window logits read + indices written + windows read) with their fractions;
  e2e           the same metric through the public API with pinned host inputs copied in and the
                indices copied back inside the timed region;
  configs       dsa_index_topk on the other four named workloads, timed the same way, each with
                its fractions of the FP8 peak and of the HBM peak;
  cpu_baseline  the CPU oracle on every row of the workload (a bounded row sample if that would
                take much longer than 30 s), all host cores;
  clocks        nvidia-smi SM clock samples taken during a sustained loop of the same step just
                before the timed region and during it.

--impl reference times the CPU oracle (the slow reference implementation of the method) on the
whole workload per timed step (a bounded row sample per step when K whole steps would take more
than about 3 minutes) and prints the same JSON line with "impl": "reference".
Multi-GPU (torchrun): the path has no exchange step, so each rank runs an independent replica
of the workload (weak scaling); value = all ranks' tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import csv
import datetime as dt
import hashlib
import io
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

METRIC = "indexer+top-k query tokens/s"
UNIT = "tokens/s"
WORKLOAD = "dsv32"
WORKLOAD_DESC = ("DeepSeek-V3.2-shaped prefill: T=N=8192, H=64, D=128, causal windows (ks=0, ke=t+1), "
                 "top-k 2048, e4m3 q/k per-row scaled, seed 2")
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Evicts L2 (129 MB) before a timed step: writes one buffer larger than L2, then reads a second
    one, so the dirty lines of the write are written back here and not inside the timed kernel."""

    def __init__(self, torch, dev):
        self.wbuf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.rbuf = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.wbuf.zero_()
        self.rbuf.max()
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0  # nominal dense fp8 / bf16 tensor-core ratio (4.5 / 2.25 PFLOP/s)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "index_topk_dsv32_traffic.txt")
KERNEL_SOURCES = ["index_kernel.cuh", "select.cuh", "ptx.cuh", "common.cuh", "types.cuh"]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--workload", default=WORKLOAD, help=argparse.SUPPRESS)
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle CPU baseline leg")
    ap.add_argument("--no-extras", action="store_true", help="skip phases and e2e (profiling runs)")
    ap.add_argument("--phases-only", action="store_true",
                    help="run only the phase kernels (unfused scorer and selector, key quantiser, sparse attention) "
                         "and print their record (profiling runs)")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "sparse_attention_indexer_e4m3_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(key="dram_bytes_per_launch"):
    """Per-launch bytes of the fused kernel from the committed ncu summary (DRAM by default;
    "lts_bytes_per_launch" for the L2), if it was taken on the current kernel source (else None)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    vals = {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha") != kernel_source_hash():
        return None
    try:
        return float(vals[key])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------------------ clocks


class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(1.0)  # let the sampler reach its loop before the timed region

    def mark_start(self):
        self.t0 = dt.datetime.now()

    def mark_end(self):
        self.t1 = dt.datetime.now()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for rec in csv.reader(io.StringIO(out)):
            if len(rec) < 9:
                continue
            try:
                ts = dt.datetime.strptime(rec[0].strip(), "%Y/%m/%d %H:%M:%S.%f")
                sm = float(rec[1].strip().split()[0])
                smax = float(rec[2].strip().split()[0])
            except ValueError:
                continue
            rows.append((ts, sm, smax, [x.strip() for x in rec[4:9]]))
        inside = [r for r in rows if self.t0 and self.t1 and self.t0 <= r[0] <= self.t1]
        note = "samples during a 1.5 s sustained loop of the same step just before the timed region and during it"
        if not inside and rows and self.t0 and self.t1:
            mid = self.t0 + (self.t1 - self.t0) / 2
            inside = sorted(rows, key=lambda r: abs((r[0] - mid).total_seconds()))[:3]
            note = "timed region shorter than the sampling period: nearest samples"
        if not inside:
            return None
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(1, 5) if r[3][i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "note": note}


# ------------------------------------------------------------------------------ helpers


def algorithmic(wl):
    lo = wl.ks.clip(0, wl.N).astype("int64")
    hi = wl.ke.clip(0, wl.N).astype("int64")
    pairs = int((hi - lo).clip(0).sum())
    flops = 2.0 * wl.H * wl.D * pairs
    fused_bytes = (wl.T * wl.H * wl.D + wl.N * wl.D + 4 * wl.N + 4 * wl.T * wl.H + 8 * wl.T + 4 * wl.T * wl.topk)
    select_bytes = 4 * pairs + 4 * wl.T * wl.topk + 8 * wl.T
    score_bytes = fused_bytes - 4 * wl.T * wl.topk + 4 * pairs
    return {"pairs": pairs, "flops": flops, "fused_bytes": float(fused_bytes), "select_bytes": float(select_bytes),
            "score_bytes": float(score_bytes)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def make_max_over_ranks(world, device):
    """max of a float over all ranks (an all-reduce on `device`: a CUDA device under NCCL, the CPU
    under gloo); the identity for one rank."""

    def max_over_ranks(x: float) -> float:
        if world == 1:
            return x
        import torch
        import torch.distributed as tdist

        t = torch.tensor([x], dtype=torch.float64, device=device)
        tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
        return float(t.item())

    return max_over_ranks


def replica_throughput(units_per_rank, local_seconds, world, max_over_ranks):
    """Whole-job throughput of `world` independent replicas that each processed units_per_rank
    units in local_seconds: every rank's units over the slowest rank's time.  Returns
    (value, slowest seconds); identical on every rank."""
    slowest = max_over_ranks(local_seconds)
    return world * units_per_rank / slowest, slowest


def cpu_baseline(wl, seconds=30.0, max_rows=None):
    """The CPU oracle (scores + top-k, as it stands) on all host cores: every query row of the
    workload when that takes at most about `seconds`, else an evenly spaced sample of rows sized
    to about `seconds` of work.  Returns (rows/s, cores, description)."""
    import numpy as np

    import oracle

    cores = oracle.threads()

    def run(rows):
        t = time.perf_counter()
        sc = oracle.index_score(wl.q, wl.w, wl.k, wl.k_scale, wl.ks, wl.ke, rows=rows, nthreads=cores)
        oracle.topk(sc, wl.topk, nthreads=cores)
        return time.perf_counter() - t

    probe = np.linspace(0, wl.T - 1, num=min(wl.T, 2 * cores), dtype=np.int64)
    dt_probe = run(probe)
    rate = len(probe) / max(dt_probe, 1e-6)
    n = int(max(len(probe), min(wl.T, rate * seconds)))
    if max_rows:
        n = min(n, max_rows)
    rows = np.linspace(0, wl.T - 1, num=n, dtype=np.int64)
    elapsed = run(rows)
    if n == wl.T:
        desc = f"all {wl.T} query rows of the workload, oracle scores + top-k, {elapsed:.1f} s"
    else:
        desc = (f"{n} evenly spaced query rows of the {wl.T}-token workload (every ~{wl.T / n:.1f}th row), "
                f"oracle scores + top-k, {elapsed:.1f} s")
    return n / elapsed, cores, desc


def bench_config(wl, world):
    """The JSON line's config object (identical in both arms)."""
    alg = algorithmic(wl)
    return {"workload": WORKLOAD_DESC, "T": wl.T, "N": wl.N, "H": wl.H, "D": wl.D, "topk": wl.topk,
            "pairs": alg["pairs"], "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "flushed before every timed step, outside the events: 256 MB written, then another 256 MB read"}


# ------------------------------------------------------------------------------ reference arm


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    import workloads

    wl = workloads.make_config(args.workload)
    cores = oracle.threads()

    def step(rows):
        t = time.perf_counter()
        sc = oracle.index_score(wl.q, wl.w, wl.k, wl.k_scale, wl.ks, wl.ke, rows=rows, nthreads=cores)
        oracle.topk(sc, wl.topk, nthreads=cores)
        return time.perf_counter() - t

    probe = np.linspace(0, wl.T - 1, num=min(wl.T, 2 * cores), dtype=np.int64)
    rate = len(probe) / max(step(probe), 1e-6)
    # Timed steps take the whole workload when K of them fit the budget (about 3 minutes), else
    # an evenly spaced row sample sized to it; warm-up steps (untimed) take a small sample.
    budget = 180.0
    per_step = max(1, min(wl.T, int(rate * budget / max(1, args.steps))))
    warm_rows = max(1, min(per_step, 2 * cores))
    step_times = []
    for i in range(args.warmup + args.steps):
        n = warm_rows if i < args.warmup else per_step
        if n == wl.T:
            rows = np.arange(wl.T, dtype=np.int64)
        else:
            # evenly spaced rows (the causal row cost grows with the row index), offset per step
            offset = ((i * 0.6180339887) % 1.0) * wl.T / n
            rows = np.unique(np.minimum(wl.T - 1, (np.arange(n) * wl.T / n + offset).astype(np.int64)))
        dt_step = step(rows)
        if i >= args.warmup:
            step_times.append((dt_step, len(rows)))
    total_t = sum(x[0] for x in step_times)
    total_rows = sum(x[1] for x in step_times)
    value = total_rows / total_t
    if per_step == wl.T:
        sample = f"all {wl.T} query rows of the workload per step, oracle scores + top-k on {cores} threads"
    else:
        sample = (f"{per_step} evenly spaced query rows per step (every ~{wl.T / per_step:.1f}th row of the "
                  f"{wl.T}-token workload, offset per step), oracle scores + top-k on {cores} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(wl, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------ GPU arm


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch

    import sparse_attention_indexer_e4m3_gb300 as dsa
    import workloads

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as tdist

        torch.cuda.set_device(local)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dsa.load()

    def barrier():
        if world > 1:
            import torch.distributed as tdist

            tdist.barrier()
        torch.cuda.synchronize()

    max_over_ranks = make_max_over_ranks(world, dev)

    wl = workloads.make_config(args.workload)
    alg = algorithmic(wl)
    host = {n: torch.from_numpy(np.ascontiguousarray(getattr(wl, n))) for n in ("q", "w", "k", "k_scale", "ks", "ke")}
    d = {n: v.to(dev) for n, v in host.items()}
    ws_bytes = dsa.index_topk_workspace_size(wl.T, wl.N, wl.H, wl.D, wl.topk)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    idx = torch.empty((wl.T, wl.topk), dtype=torch.int32, device=dev)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream()

    def plan():
        dsa.index_topk_plan(d["ks"], d["ke"], wl.N, wl.H, wl.D, wl.topk, workspace=ws)

    def run():
        dsa.index_topk_run(d["q"], d["w"], d["k"], d["k_scale"], d["ks"], d["ke"], wl.topk, ws, idx=idx)

    if args.phases_only:
        peaks, _ = load_peaks()
        fp8_peak = FP8_PER_BF16 * float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        print(json.dumps(phases(dsa, torch, wl, d, alg, flush, stream, fp8_peak, hbm_peak, reps=3)), flush=True)
        return 0

    for _ in range(args.warmup):
        flush()
        plan()
        run()
    if dsa.get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(local)
    sampler.start()
    barrier()
    # The clock record covers a sustained loop of the same step (about 1.5 s, untimed) right
    # before the timed region, and the timed region itself: a short timed region falls between
    # two of nvidia-smi's samples.
    sampler.mark_start()
    t_end = time.perf_counter() + 1.5
    while time.perf_counter() < t_end:
        for _ in range(50):
            flush()
            plan()
            run()
        torch.cuda.synchronize()
    barrier()
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        plan()
        ev[i][1].record(stream)
        run()
        ev[i][2].record(stream)
    barrier()
    sampler.mark_end()
    clocks = sampler.stop()
    if dsa.get_device_error() != 0:
        raise RuntimeError("device error in the timed region")
    plan_ms = [e[0].elapsed_time(e[1]) for e in ev]
    run_ms = [e[1].elapsed_time(e[2]) for e in ev]
    step_ms = [a + b for a, b in zip(plan_ms, run_ms)]
    value, total_s = replica_throughput(wl.T * K, sum(step_ms) / 1e3, world, max_over_ranks)

    peaks, peak_src = load_peaks()
    fp8_peak = FP8_PER_BF16 * float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    run_mean_s = statistics.fmean(run_ms) / 1e3
    achieved = alg["flops"] / run_mean_s / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": achieved / fp8_peak, "traffic": committed_traffic(),
                "traffic_l2": committed_traffic("lts_bytes_per_launch"),
                "kernel": "dsa::index_kernel<64,128,true> (fused scorer + selector)",
                "per_launch": {"flops": alg["flops"], "algorithmic_bytes": alg["fused_bytes"],
                               "mean_ms": 1e3 * run_mean_s, "median_ms": statistics.median(run_ms)},
                "peak_source": (f"{peak_src}: 2 x bf16 burst {peaks.get('bf16_tflops')} TFLOP/s "
                                "(nominal fp8/bf16 ratio 2)"),
                "fused_hbm_gbs": alg["fused_bytes"] / run_mean_s / 1e9,
                "fused_hbm_frac": alg["fused_bytes"] / run_mean_s / 1e9 / hbm_peak}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> f32 accumulate, fp32 scores", "data": "synthetic",
        "config": bench_config(wl, world),
        "plan_ms": statistics.fmean(plan_ms), "run_ms": statistics.fmean(run_ms),
        "gpu_launches": 2 * K,
        "roofline": roofline,
        "clocks": clocks,
    }

    if not args.no_extras:
        line["configs"] = other_configs(dsa, torch, dev, flush, stream, fp8_peak, hbm_peak)
        line["phases"] = phases(dsa, torch, wl, d, alg, flush, stream, fp8_peak, hbm_peak)
        line["e2e"] = e2e(dsa, torch, wl, host, dev, stream, args, world, max_over_ranks)
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        rate, cores, sample = cpu_baseline(wl)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as tdist

        tdist.destroy_process_group()
    return 0


OTHER_CONFIGS = {
    "tiny": "256-token prefill: T=N=256, H=4, D=64, causal, top-k 32, seed 0",
    "glm": "GLM-style prefill: T=N=1024, H=32, D=128, causal, top-k 512, seed 1",
    "decode": ("ragged decode: 64 requests x 1 query token, cache lengths uniform in [4096, 65536] packed along N "
               "(realised sum 1,939,851 keys), H=64, D=128, top-k 2048, seed 3"),
    "varlen": ("packed long prefill: documents 2048/6144/8192/16384 packed to T=N=32768, causal within each "
               "document, 1% of keys x8, H=64, D=128, top-k 2048, seed 4, fused only"),
}


def other_configs(dsa, torch, dev, flush, stream, fp8_peak, hbm_peak, reps=20):
    """dsa_index_topk (plan + run) on the other four named workloads, timed like the headline one
    (CUDA events on the launching stream, L2 flushed before every step).  Prefills are graded
    against the FP8 tensor peak, the packed decode against the HBM copy peak."""
    import numpy as np

    import workloads

    out = {}
    for name, desc in OTHER_CONFIGS.items():
        wl = workloads.make_config(name)
        alg = algorithmic(wl)
        d = {n: torch.from_numpy(np.ascontiguousarray(getattr(wl, n))).to(dev)
             for n in ("q", "w", "k", "k_scale", "ks", "ke")}
        ws = torch.empty(max(dsa.index_topk_workspace_size(wl.T, wl.N, wl.H, wl.D, wl.topk), 256),
                         dtype=torch.uint8, device=dev)
        idx = torch.empty((wl.T, wl.topk), dtype=torch.int32, device=dev)

        def step():
            dsa.index_topk_plan(d["ks"], d["ke"], wl.N, wl.H, wl.D, wl.topk, workspace=ws)
            e1.record(stream)
            dsa.index_topk_run(d["q"], d["w"], d["k"], d["k_scale"], d["ks"], d["ke"], wl.topk, ws, idx=idx)

        plan_ms, run_ms = [], []
        for i in range(3 + reps):
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            flush()
            e0.record(stream)
            step()
            e2.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                plan_ms.append(e0.elapsed_time(e1))
                run_ms.append(e1.elapsed_time(e2))
        if dsa.get_device_error() != 0:
            raise RuntimeError(f"device error in workload {name}")
        run_s = statistics.fmean(run_ms) / 1e3
        step_s = run_s + statistics.fmean(plan_ms) / 1e3
        rec = {"workload": desc, "T": wl.T, "N": wl.N, "H": wl.H, "D": wl.D, "topk": wl.topk,
               "pairs": alg["pairs"], "plan_ms": statistics.fmean(plan_ms), "run_ms": 1e3 * run_s,
               "tokens_per_s": wl.T / step_s, "run_tflops": alg["flops"] / run_s / 1e12,
               "run_frac_fp8_peak": alg["flops"] / run_s / 1e12 / fp8_peak,
               "run_hbm_gbs": alg["fused_bytes"] / run_s / 1e9,
               "run_frac_hbm_peak": alg["fused_bytes"] / run_s / 1e9 / hbm_peak,
               "bound": "hbm" if name == "decode" else "tensor"}
        out[name] = rec
        del d, ws, idx
    return out


def phases(dsa, torch, wl, d, alg, flush, stream, fp8_peak, hbm_peak, reps=20):
    """Unfused scorer and selector, each timed alone (L2 flushed before each launch)."""
    logits = torch.empty((wl.T, wl.N), dtype=torch.float32, device=d["q"].device)
    idx = torch.empty((wl.T, wl.topk), dtype=torch.int32, device=d["q"].device)
    for _ in range(3):
        dsa.index_score(d["q"], d["w"], d["k"], d["k_scale"], d["ks"], d["ke"], logits=logits)
        dsa.topk(logits, d["ks"], d["ke"], wl.topk, idx=idx)
    s_ms, t_ms = [], []
    for _ in range(reps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        flush()
        e[0].record(stream)
        dsa.index_score(d["q"], d["w"], d["k"], d["k_scale"], d["ks"], d["ke"], logits=logits)
        e[1].record(stream)
        flush()
        e[2].record(stream)
        dsa.topk(logits, d["ks"], d["ke"], wl.topk, idx=idx)
        e[3].record(stream)
        torch.cuda.synchronize()
        s_ms.append(e[0].elapsed_time(e[1]))
        t_ms.append(e[2].elapsed_time(e[3]))
    s = statistics.fmean(s_ms) / 1e3
    t = statistics.fmean(t_ms) / 1e3
    # the same scores with the key tile resident and the query blocks streamed
    kws = torch.empty(max(256, dsa.index_score_kres_workspace_size(wl.T, wl.N, wl.H, wl.D)), dtype=torch.uint8,
                      device=d["q"].device)
    for _ in range(3):
        dsa.index_score_kres(d["q"], d["w"], d["k"], d["k_scale"], d["ks"], d["ke"], logits=logits, workspace=kws)
    r_ms = []
    for _ in range(reps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        flush()
        e[0].record(stream)
        dsa.index_score_kres(d["q"], d["w"], d["k"], d["k_scale"], d["ks"], d["ke"], logits=logits, workspace=kws)
        e[1].record(stream)
        torch.cuda.synchronize()
        r_ms.append(e[0].elapsed_time(e[1]))
    r = statistics.fmean(r_ms) / 1e3
    del logits, kws
    # key quantiser (bf16 -> e4m3 codes + per-row scales) on a key cache the size of the packed
    # decode workload's (1,939,851 keys), seeded normal values
    nq = 1_939_851
    gen = torch.Generator(device=d["q"].device).manual_seed(7)
    kq = torch.randn((nq, wl.D), generator=gen, device=d["q"].device, dtype=torch.float32).to(torch.bfloat16)
    codes = torch.empty((nq, wl.D), dtype=torch.uint8, device=d["q"].device)
    kscale = torch.empty(nq, dtype=torch.float32, device=d["q"].device)
    for _ in range(3):
        dsa.quantize_k(kq, codes, kscale)
    q_ms = []
    for _ in range(reps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        flush()
        e[0].record(stream)
        dsa.quantize_k(kq, codes, kscale)
        e[1].record(stream)
        torch.cuda.synchronize()
        q_ms.append(e[0].elapsed_time(e[1]))
    qt = statistics.fmean(q_ms) / 1e3
    q_bytes = nq * (3 * wl.D + 4)
    del kq, codes, kscale
    # sparse attention over the selected keys (the selector's output above), 64 heads of
    # D = 512, seeded normal bf16 q / kv, a per-head sink; tensor-core kernel, a few launches
    attn = None
    attn_h128 = None
    attn_bwd = None
    if wl.T <= 8192:
        ha, da = 64, 512
        gen = torch.Generator(device=d["q"].device).manual_seed(8)
        qa = torch.randn((wl.T, ha, da), generator=gen, device=d["q"].device).to(torch.bfloat16)
        kva = torch.randn((wl.N, da), generator=gen, device=d["q"].device).to(torch.bfloat16)
        sink = torch.randn(ha, generator=gen, device=d["q"].device)
        oa = torch.empty((wl.T, ha, da), dtype=torch.bfloat16, device=d["q"].device)
        dsa.sparse_attn(qa, kva, idx, attn_sink=sink, out=oa)
        a_ms = []
        for _ in range(3):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            flush()
            e[0].record(stream)
            dsa.sparse_attn(qa, kva, idx, attn_sink=sink, out=oa)
            e[1].record(stream)
            torch.cuda.synchronize()
            a_ms.append(e[0].elapsed_time(e[1]))
        at = statistics.fmean(a_ms) / 1e3
        pairs = int((idx >= 0).sum().item())
        a_flops = 4.0 * pairs * ha * da  # q.kv and the weighted kv rows, 2 flops per multiply-add
        bf16_peak = fp8_peak / FP8_PER_BF16
        attn = {"kernel": "dsa::sparse_attn_tc_kernel<512> (tcgen05 kind::f16, bf16 weights)", "heads": ha, "dim": da,
                "pairs": pairs, "ms": 1e3 * at, "tflops": a_flops / at / 1e12,
                "frac_bf16_peak": a_flops / at / 1e12 / bf16_peak}
        del qa, sink, oa
        # 128 heads (the head count of the pages' sparse MLA measurements) over the same lists and
        # kv rows: two head groups of 64, one launch each
        hw = 128
        qw = torch.randn((wl.T, hw, da), generator=gen, device=d["q"].device).to(torch.bfloat16)
        sinkw = torch.randn(hw, generator=gen, device=d["q"].device)
        ow = torch.empty((wl.T, hw, da), dtype=torch.bfloat16, device=d["q"].device)
        dsa.sparse_attn(qw, kva, idx, attn_sink=sinkw, out=ow)
        w_ms = []
        for _ in range(3):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            flush()
            e[0].record(stream)
            dsa.sparse_attn(qw, kva, idx, attn_sink=sinkw, out=ow)
            e[1].record(stream)
            torch.cuda.synchronize()
            w_ms.append(e[0].elapsed_time(e[1]))
        wt = statistics.fmean(w_ms) / 1e3
        w_flops = 4.0 * pairs * hw * da
        attn_h128 = {"kernel": "dsa::sparse_attn_tc_kernel<512> x 2 head groups of 64", "heads": hw, "dim": da,
                     "pairs": pairs, "ms": 1e3 * wt, "tflops": w_flops / wt / 1e12,
                     "frac_bf16_peak": w_flops / wt / 1e12 / bf16_peak}
        del qw, sinkw, ow, kva
        # its gradients (the backward kernel takes D <= 256): the same lists, D = 256, 64 heads
        db = 256
        qb = torch.randn((wl.T, ha, db), generator=gen, device=d["q"].device).to(torch.bfloat16)
        kvb = torch.randn((wl.N, db), generator=gen, device=d["q"].device).to(torch.bfloat16)
        dob = torch.randn((wl.T, ha, db), generator=gen, device=d["q"].device).to(torch.bfloat16)
        sinkb = torch.randn(ha, generator=gen, device=d["q"].device)
        lse = torch.empty((wl.T, ha), dtype=torch.float32, device=d["q"].device)
        ob = dsa.sparse_attn(qb, kvb, idx, attn_sink=sinkb, lse=lse)
        gq = torch.empty((wl.T, ha, db), dtype=torch.float32, device=d["q"].device)
        gkv = torch.empty((wl.N, db), dtype=torch.float32, device=d["q"].device)
        gs = torch.empty(ha, dtype=torch.float32, device=d["q"].device)
        dsa.sparse_attn_bwd(qb, kvb, idx, ob, lse, dob, attn_sink=sinkb, dq=gq, dkv=gkv, dsink=gs)
        b_ms = []
        for _ in range(3):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            flush()
            e[0].record(stream)
            dsa.sparse_attn_bwd(qb, kvb, idx, ob, lse, dob, attn_sink=sinkb, dq=gq, dkv=gkv, dsink=gs)
            e[1].record(stream)
            torch.cuda.synchronize()
            b_ms.append(e[0].elapsed_time(e[1]))
        bt = statistics.fmean(b_ms) / 1e3
        b_flops = 10.0 * pairs * ha * db  # five products: S, dP, dQ and dKV's two terms
        attn_bwd = {"kernel": "dsa::sparse_attn_bwd_tc_kernel<256> (tcgen05 kind::f16, atomic dkv)", "heads": ha,
                    "dim": db, "pairs": pairs, "ms": 1e3 * bt, "tflops": b_flops / bt / 1e12,
                    "frac_bf16_peak": b_flops / bt / 1e12 / bf16_peak}
        del qb, kvb, dob, sinkb, lse, ob, gq, gkv, gs
    return {"sparse_attn": attn, "sparse_attn_128_heads": attn_h128, "sparse_attn_bwd": attn_bwd,
            "score": {"kernel": "dsa::index_kernel<64,128,false>", "ms": 1e3 * s, "tflops": alg["flops"] / s / 1e12,
                      "frac_fp8_peak": alg["flops"] / s / 1e12 / fp8_peak,
                      "hbm_gbs": alg["score_bytes"] / s / 1e9},
            "score_k_resident": {"kernel": "dsa::kres_kernel<64,128> (+ window pass)", "ms": 1e3 * r,
                                 "tflops": alg["flops"] / r / 1e12, "frac_fp8_peak": alg["flops"] / r / 1e12 / fp8_peak},
            "quantize_k": {"kernel": "dsa::quantize_rows_kernel", "rows": nq, "ms": 1e3 * qt,
                           "gbs": q_bytes / qt / 1e9, "frac_hbm_peak": q_bytes / qt / 1e9 / hbm_peak},
            "select": {"kernel": ("dsa::topk_rows_stream_kernel" if wl.N <= 8192 else "dsa::topk_rows_kernel"),
                       "ms": 1e3 * t, "gbs": alg["select_bytes"] / t / 1e9,
                       "frac_hbm_peak": alg["select_bytes"] / t / 1e9 / hbm_peak}}


def e2e(dsa, torch, wl, host, dev, stream, args, world, max_over_ranks, reps=None):
    """The public call with pinned host inputs: every step copies its inputs host -> device, runs
    dsa_index_topk and copies its indices device -> host.  Steps are pipelined the way a serving
    loop would run them: copies on their own streams, two sets of device buffers, so step i's
    compute overlaps step i+1's input copy and step i-1's result copy (each step still moves all
    of its own bytes).  The same steps run back to back on one stream are reported beside it."""
    reps = reps or max(5, min(50, args.steps))
    pinned = {n: v.pin_memory() for n, v in host.items()}
    bufs = [{n: torch.empty_like(v, device=dev) for n, v in host.items()} for _ in range(2)]
    outs = [torch.empty((wl.T, wl.topk), dtype=torch.int32).pin_memory() for _ in range(2)]
    idxs = [torch.empty((wl.T, wl.topk), dtype=torch.int32, device=dev) for _ in range(2)]
    ws = torch.empty(max(dsa.index_topk_workspace_size(wl.T, wl.N, wl.H, wl.D, wl.topk), 256), dtype=torch.uint8,
                     device=dev)
    s_in, s_run, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    run_done = [None, None]
    out_done = [None, None]

    def step(i, pipelined):
        b = i % 2 if pipelined else 0
        si, sr, so = (s_in, s_run, s_out) if pipelined else (stream, stream, stream)
        d = bufs[b]
        with torch.cuda.stream(si):
            if run_done[b] is not None:
                si.wait_event(run_done[b])  # step i-2 has finished reading these inputs
            for n in pinned:
                d[n].copy_(pinned[n], non_blocking=True)
            in_done = torch.cuda.Event()
            in_done.record(si)
        with torch.cuda.stream(sr):
            sr.wait_event(in_done)
            if out_done[b] is not None:
                sr.wait_event(out_done[b])  # step i-2's indices have left the device
            dsa.index_topk(d["q"], d["w"], d["k"], d["k_scale"], d["ks"], d["ke"], wl.topk, idx=idxs[b],
                           workspace=ws, stream=sr)
            run_done[b] = torch.cuda.Event()
            run_done[b].record(sr)
        with torch.cuda.stream(so):
            so.wait_event(run_done[b])
            outs[b].copy_(idxs[b], non_blocking=True)
            out_done[b] = torch.cuda.Event()
            out_done[b].record(so)

    def timed(pipelined):
        for i in range(3):
            step(i, pipelined)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(reps):
            step(i, pipelined)
        torch.cuda.synchronize()
        return time.perf_counter() - t0

    seq_s = max_over_ranks(timed(False))
    pipe_s = max_over_ranks(timed(True))
    value, total_s = replica_throughput(wl.T * reps, pipe_s, world, lambda x: x)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(wl.T * wl.topk * 4), "ms_per_step": 1e3 * total_s / reps, "steps": reps,
            "pipelined": "H2D / compute / D2H on three streams, double-buffered; host wall clock over all steps",
            "sequential_ms_per_step": 1e3 * seq_s / reps}


if __name__ == "__main__":
    sys.exit(main())

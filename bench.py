"""Benchmark of the gradient all-reduce over N virtual ranks on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one all-reduce of the workload: 16 virtual ranks, each a 192 MiB
fp32 gradient (50,331,648 values, N(0, 1e-3^2), seed 0), summed in ring order
by the fused single pass (bit-identical to the step-by-step ring). The timed
region holds K steps on one stream, bracketed by a barrier and a device
synchronise. Each step reads 16 x 192 MiB and writes 16 x 192 MiB (6 GiB of
traffic), far more than the 126 MB L2, so no flush is needed between steps.
Inputs are kept pristine (out of place) so every step reduces the same data.

Reported (one JSON line from rank 0):
  value      algbw = per-rank buffer bytes x steps x GPUs / time (GB/s, 1e9)
  busbw      algbw x 2(N-1)/N (the nccl-tests convention)
  roofline   the fused kernel's algorithmic bytes (2 N S) per launch / its
             CUDA-event launch time, against the measured HBM copy bandwidth
  executors  the step-by-step ring and Rabenseifner on the same workload,
             each against its own byte count, 5(N-1) S; and the blockwise
             INT8 compressed all-reduce with error feedback (fused pass, and
             compressor + reducer), each against its own byte count
  latency    small messages: the 16-rank ring and Rabenseifner at 1 KiB per
             rank, bound once and replayed (ar_execute_bound); both run
             every step in one CTA
  e2e        the same all-reduce from pinned host buffers through
             ar_execute_host, copies included
  cpu_baseline  the CPU oracle (step-by-step ring simulation) on a bounded
             sample of the same workload: one process per host core (value,
             cores) and one core alone (value_one_core)

With --gpus N > 1 (torchrun, one process per GPU) every GPU all-reduces its
own copy of the workload (weak scaling, no collective on the data path); the
timing is the maximum over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "all-reduce algbw/busbw GB/s (N virtual ranks, 1 GB300) and % of HBM roofline"
UNIT = "GB/s"
PROFILE = os.path.join(ROOT, "profiles", "fused_ring_n16_192mib.md")
KERNEL_SOURCES = ["gradient_sync_gb300/csrc/fused.cu", "gradient_sync_gb300/csrc/common.cuh"]
# From internal.h only what the fused kernel compiles from: its parameter
# block and the block size (other declarations there do not change it).
KERNEL_HEADER = "gradient_sync_gb300/csrc/internal.h"


# ------------------------------------------------------------------ helpers


def kernel_sources_hash() -> str:
    """Hash of the fused kernel's sources: fused.cu, common.cuh, and from
    internal.h the FusedParams struct and the kThreads constant."""
    import re

    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    with open(os.path.join(ROOT, KERNEL_HEADER)) as f:
        text = f.read()
    for pattern in (r"struct FusedParams \{.*?\n\};", r"constexpr int kThreads = \d+;"):
        m = re.search(pattern, text, flags=re.S)
        h.update((m.group(0) if m else "").encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the fused kernel from the committed ncu summary,
    if it was taken on the current kernel sources; else None."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, _, v = line.strip()[2:].partition(":")
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("sources_sha256") != kernel_sources_hash():
        return None
    try:
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks, power and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        for line in self.out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [r for r in rows if r["power"] > 300.0] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": sorted(reasons),
                "samples": len(loaded), "power_w_max": max(r["power"] for r in rows)}


def _oracle_sample(win: int):
    """The cpu_baseline sample: one `win`-element window per chunk of every
    rank of the 16 x 192 MiB workload, and the element indices it covers."""
    import numpy as np

    import workloads

    spec = workloads.RING_N16_192MIB
    N, L = spec.n_ranks, spec.count
    idx = np.concatenate([np.arange((c * L) // N, (c * L) // N + win) for c in range(N)]).astype(np.int64)
    x = np.stack([np.concatenate([workloads.rank_buffer(spec, r, (c * L) // N, (c * L) // N + win, threads=1)
                                  for c in range(N)]) for r in range(N)])
    return x, idx, L


def _oracle_loop(args):
    """Run the oracle's step-by-step ring on the sample for `seconds`; returns
    (repetitions, elapsed seconds, sampled bytes per rank)."""
    x, idx, L, seconds = args
    from oracle import schedules

    reps, t0 = 0, time.perf_counter()
    while True:
        schedules.ring_allreduce(x, idx=idx, L=L)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return reps, el, idx.size * 4


def cpu_baseline(seconds: float = 10.0):
    """The oracle (step-by-step ring simulation in numpy) on a bounded sample of
    the workload, one 16 Ki-element window per chunk of every rank: on one core,
    then as one process per host core, each running the same sample (elements
    are independent, so cores multiply the throughput)."""
    import multiprocessing as mp

    win = 16 * 1024
    x, idx, L = _oracle_sample(win)
    reps, el, per_rank = _oracle_loop((x, idx, L, seconds))
    one = per_rank * reps / el / 1e9
    procs = max(1, os.cpu_count() or 1)
    ctx = mp.get_context("spawn")  # this process has initialised CUDA: no fork
    with ctx.Pool(procs) as pool:
        res = pool.map(_oracle_loop, [(x, idx, L, seconds)] * procs)
    wall = max(e for _, e, _ in res)
    many = sum(r * b for r, _, b in res) / wall / 1e9
    return {"value": round(many, 6), "unit": UNIT, "cores": procs, "kind": "oracle",
            "value_one_core": round(one, 6),
            "sample": f"16 ranks x {idx.size} fp32 elements ({win} per chunk, all 16 chunks) of the 192 MiB "
                      f"workload, step-by-step ring simulation; {procs} processes each repeating it for "
                      f"{seconds:.0f} s (one core alone: {reps} repetitions in {el:.1f} s); algbw = sampled "
                      f"per-rank bytes / time"}


# ------------------------------------------------------------------ distributed harness


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str, timeout_s: float | None = None):
    """The process group of a multi-GPU run (None for one process). With
    `timeout_s`, a collective that waits longer (a rank that never arrives)
    raises instead of blocking."""
    if world <= 1:
        return None
    import datetime

    import torch.distributed as dist

    if not dist.is_initialized():
        kw = {} if timeout_s is None else {"timeout": datetime.timedelta(seconds=timeout_s)}
        dist.init_process_group(backend=backend, **kw)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def timed(dist, step, sync, n_steps: int, n_warmup: int, device=None, event_timer=None):
    """Run n_warmup untimed steps, then time n_steps bracketed by a barrier and a
    sync on both sides; returns the max over ranks of the per-rank time (ms)."""
    for _ in range(n_warmup):
        step()
    sync()
    barrier(dist, device)
    sync()
    if event_timer is not None:
        ms = event_timer(step, n_steps)
    else:
        t0 = time.perf_counter()
        for _ in range(n_steps):
            step()
        sync()
        ms = (time.perf_counter() - t0) * 1e3
    sync()
    barrier(dist, device)
    return max_over_ranks(dist, ms, device)


# ------------------------------------------------------------------ arms


def run_ours(args):
    import numpy as np
    import torch

    import gradient_sync_gb300 as g
    import workloads
    from gradient_sync_gb300 import build

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    build.build()

    spec = workloads.RING_N16_192MIB
    N, L = spec.n_ranks, spec.count
    S = L * 4
    stream = torch.cuda.Stream(device=dev)

    host = [workloads.rank_buffer(spec, r) for r in range(N)]
    bufs = [torch.from_numpy(h).to(dev) for h in host]
    outs = [torch.empty_like(b) for b in bufs]
    torch.cuda.synchronize(dev)

    def event_timer(step, n):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            step()
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b)

    def sync():
        torch.cuda.synchronize(dev)

    def make_step(plan, ws=None):
        handle = int(stream.cuda_stream)
        return lambda: g.ar_execute(plan, bufs, outs=outs, workspace=ws, stream=handle)

    fused = g.ar_plan(N, L, "f32", "fused", order="ring")
    st = fused.stats
    with ClockSampler(local) as clocks:
        ms_total = timed(dist, make_step(fused), sync, args.steps, args.warmup, local if dist else None,
                         event_timer)
    ms = ms_total / args.steps
    hbm_peak, peak_kind = measured_peaks()
    achieved = st["hbm_bytes"] / (ms * 1e-3) / 1e9
    algbw = S / (ms * 1e-3) / 1e9
    value = algbw * world

    executors = {}
    for algo in ("ring", "rabenseifner"):
        plan = g.ar_plan(N, L, "f32", algo)
        k = max(5, args.steps // 20)
        ms_e = timed(dist, make_step(plan), sync, k, args.warmup, local if dist else None, event_timer) / k
        pst = plan.stats
        bw = pst["hbm_bytes"] / (ms_e * 1e-3) / 1e9
        executors[algo] = {"ms": round(ms_e, 4), "algbw": round(S / (ms_e * 1e-3) / 1e9, 2),
                           "busbw": round(S / (ms_e * 1e-3) / 1e9 * 2 * (N - 1) / N, 2),
                           "steps": pst["steps"], "launches": pst["launches"],
                           "hbm_bytes": pst["hbm_bytes"], "achieved_gbs": round(bw, 1),
                           "frac_of_hbm": round(bw / hbm_peak, 4)}

    # blockwise INT8 compressed all-reduce with error feedback (block 128, sum
    # scaled by 1/N) on the same gradients: the fused pass and the two calls
    from gradient_sync_gb300.cases import compressed_hbm_bytes

    block = 128
    res = [torch.zeros(L, dtype=torch.float32, device=dev) for _ in range(N)]
    n_sc, _ = g.ar_compress_sizes(L, block)
    codes = [torch.empty(L, dtype=torch.int8, device=dev) for _ in range(N)]
    scales = [torch.empty(n_sc, dtype=torch.float32, device=dev) for _ in range(N)]
    handle = int(stream.cuda_stream)

    def comp_fused():
        g.ar_compressed_allreduce(bufs, block, residuals=res, scale=1.0 / N, outs=outs, stream=handle)

    def comp_two():
        g.ar_compress(bufs, codes, scales, block, residuals=res, stream=handle)
        g.ar_compressed_reduce(codes, scales, outs, block, scale=1.0 / N, stream=handle)

    for name, fn, path, launches in (("compressed_int8_fused", comp_fused, "fused", 1),
                                     ("compressed_int8_two_calls", comp_two, "two", 2)):
        k = max(5, args.steps // 20)
        ms_c = timed(dist, fn, sync, k, args.warmup, local if dist else None, event_timer) / k
        hb = compressed_hbm_bytes(N, L, "f32", block, path, True)
        bw = hb / (ms_c * 1e-3) / 1e9
        executors[name] = {"ms": round(ms_c, 4), "algbw": round(S / (ms_c * 1e-3) / 1e9, 2), "block": block,
                           "error_feedback": True, "launches": launches, "hbm_bytes": hb,
                           "achieved_gbs": round(bw, 1), "frac_of_hbm": round(bw / hbm_peak, 4)}
    del res, codes, scales
    torch.cuda.empty_cache()

    # small messages: per-call time of a bound plan, back to back from Python
    from gradient_sync_gb300.cases import time_case

    latency = {"workload": "16 ranks x 1 KiB fp32, ar_bind once, ar_execute_bound per call, back to back"}
    for algo in ("ring", "rabenseifner"):
        r = time_case(16, 256, algo=algo, iters=30, warmup=5, reps=100, bound=True)
        latency[algo] = {"us_per_call": r["us"], "steps": r["steps"], "launches": r["launches"]}

    # end to end: pinned host buffers in and out through ar_execute_host
    host_in = [torch.from_numpy(h).pin_memory() for h in host]
    host_out = [torch.empty(L, dtype=torch.float32).pin_memory() for _ in range(N)]
    del host
    handle = int(stream.cuda_stream)

    def e2e_step():
        g.ar_execute_host(fused, host_in, host_out, outs, stream=handle)

    k_e2e = max(3, min(10, args.steps // 100))
    ms_e2e = timed(dist, e2e_step, sync, k_e2e, 1, local if dist else None) / k_e2e
    got = host_out[3][: 1 << 16].numpy()
    assert np.isfinite(got).all()

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": spec.name + ", fused single pass in ring order (bit-identical to the "
                   "step-by-step ring), out of place", "n_ranks": N, "count_per_rank": L,
                   "bytes_per_rank": S, "algo": "fused", "order": "ring",
                   "l2": "no flush: each step moves 6 GiB, > 40x the L2",
                   "parallelism": f"replicas x{world} (one workload per GPU)"},
        "busbw": round(value * 2 * (N - 1) / N, 2),
        "hbm_frac": round(achieved / hbm_peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": profiled_traffic(),
                     "kernel": "fused_flat_kernel<fp32, seq>", "peak_kind": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": st["hbm_bytes"]},
        "executors": executors,
        "latency": latency,
        "e2e": {"value": round(S * world / (ms_e2e * 1e-3) / 1e9, 2), "unit": UNIT,
                "h2d_bytes_per_step": N * S, "d2h_bytes_per_step": N * S, "ms_per_step": round(ms_e2e, 3),
                "api": "ar_execute_host: pinned host buffers read and written by the kernel over NVLink-C2C"},
        "gpu_launches": args.steps * st["launches"],
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier(device_ids=[local])
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle timed as the reference arm: each step is the
    step-by-step ring simulation on a bounded sample of the same workload."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np

    import workloads
    from oracle import schedules

    spec = workloads.RING_N16_192MIB
    N, L = spec.n_ranks, spec.count
    win = 256
    idx = np.concatenate([np.arange((c * L) // N, (c * L) // N + win) for c in range(N)]).astype(np.int64)
    x = np.stack([np.concatenate([workloads.rank_buffer(spec, r, (c * L) // N, (c * L) // N + win, threads=1)
                                  for c in range(N)]) for r in range(N)])

    def step():
        schedules.ring_allreduce(x, idx=idx, L=L)

    ms_total = timed(None, step, lambda: None, args.steps, args.warmup)
    ms = ms_total / args.steps
    per_rank = idx.size * 4
    value = per_rank / (ms * 1e-3) / 1e9
    sample = (f"{N} ranks x {idx.size} fp32 elements ({win} per chunk, all {N} chunks) of the 192 MiB "
              "workload per step; step-by-step ring simulation")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": spec.name + ", ring all-reduce (CPU oracle on a sample)", "n_ranks": N,
                       "count_per_rank": L, "bytes_per_rank": L * 4, "algo": "ring", "order": "ring"},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the ~10 s oracle timing")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, _, _ = dist_env()
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}; launch N>1 with torchrun")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

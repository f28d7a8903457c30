"""Benchmark of the gradient all-reduce over N virtual ranks on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one all-reduce of the headline workload: 16 virtual ranks, each a
192 MiB fp32 gradient (50,331,648 values, N(0, 1e-3^2), seed 0), summed in
ring order by the fused single pass (bit-identical to the step-by-step ring).
The timed region holds K steps on one stream, bracketed by a barrier and a
device synchronise. Each step reads 16 x 192 MiB and writes 16 x 192 MiB
(6 GiB of traffic), far more than the 126 MB L2, so no flush is needed
between steps. Inputs are kept pristine (out of place) so every step reduces
the same data.

Reported (one JSON line from rank 0):
  value      algbw = per-rank buffer bytes x steps x GPUs / time (GB/s, 1e9)
  busbw      algbw x 2(N-1)/N (the nccl-tests convention)
  roofline   the fused kernel's algorithmic bytes (2 N S) per launch / its
             CUDA-event launch time, against the measured HBM copy bandwidth
  executors  on the headline workload: the step-by-step ring and Rabenseifner,
             each against its own byte count, 5(N-1) S; and the blockwise
             INT8 compressed all-reduce with error feedback (fused pass, and
             compressor + reducer), each against its own byte count
  workloads  the other workloads, each path against its own algorithmic bytes,
             each with the CPU oracle running the same algorithm beside it:
               ring_n4_int       4 ranks x 1,048,576 integer-valued fp32
               hier_2x8_bf16     16 ranks as 2 groups of 8, 96 Mi bf16 each
                                 (and the INT8 compressed all-reduce of the
                                 same gradients without error feedback)
               buckets_n8_transformer  8 ranks, 16-layer transformer bf16
                                 gradients in 25 MiB buckets, x1/8, bf16 out
               sm_budget_n16_192mib  the headline's fused pass held to 32
                                 and 64 SMs (sm_budget)
               overlap_8192_tokens_32_sms  the bucketed sync of the 8-rank
                                 transformer behind a synthetic backward
                                 (exposed time, hidden fraction)
               sweep             2, 16 and 64 ranks x 1 GiB fp32, and
                                 16 ranks x 1 KiB (per-call latency)
  latency    small messages: the 16-rank ring and Rabenseifner at 1 KiB per
             rank, bound once and replayed (ar_execute_bound)
  e2e        the headline all-reduce from pinned host buffers through
             ar_execute_host, copies included
  cpu_baseline  the CPU oracle (step-by-step ring simulation) on a bounded
             sample of the headline workload: one process per host core
             (value, cores) and one core alone (value_one_core)

With --gpus N > 1 (torchrun, one process per GPU) every GPU all-reduces its
own copy of the workload (weak scaling, no collective on the data path); the
timing is the maximum over ranks.

Single measurements (for tables and profiles; not part of the contract):

    python bench.py --case --algo fused --order ring --n 16 --count 8388608 --iters 3
    python bench.py --sweep > sweep.jsonl
    python bench.py --buckets fused|pack --iters 5
    python bench.py --overlap --n 8 --tokens 4096 --sm-budget 32 --iters 5
    python bench.py --compressed fused|two --n 16 --count 50331648 --block 128

Each prints one JSON line per case: time per call (median of CUDA-event
timings on the launching stream, after warm-up), algbw = S/T, busbw, and the
achieved algorithmic HBM bandwidth (ar_plan_stats.hbm_bytes / T). Their
inputs are device-filled random data (timing does not depend on values).
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
KiB, MiB, GiB = 1 << 10, 1 << 20, 1 << 30


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


def profiled_traffic(launch_bytes: int):
    """DRAM bytes per launch of the fused kernel, from the committed ncu
    summary, if it was taken on the current kernel sources; else None. The
    summary records the traffic of a smaller case of the same kernel and the
    algorithmic bytes of that case; DRAM traffic of this streaming kernel
    grows in proportion to the elements processed, so it is scaled by the
    ratio of algorithmic bytes to a full launch."""
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
        traffic = int(fields["traffic_bytes_per_launch"])
        case_bytes = int(fields["algorithmic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None
    return int(round(traffic * launch_bytes / case_bytes))


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


# ------------------------------------------------------------------ CPU oracle baselines
#
# Each baseline runs the oracle's simulation of the same algorithm the GPU
# path runs, on a bounded sample of the workload: windows of consecutive
# elements (elements never interact, so a window computes exactly what the
# full run computes there). algbw is the sampled bytes per rank over the
# time, the same definition as the GPU figure.


def _headline_sample(win: int):
    """One `win`-element window per chunk of every rank of the 16 x 192 MiB
    workload (the workload's own seeded values) and the indices it covers."""
    import numpy as np

    import workloads

    spec = workloads.RING_N16_192MIB
    N, L = spec.n_ranks, spec.count
    idx = np.concatenate([np.arange((c * L) // N, (c * L) // N + win) for c in range(N)]).astype(np.int64)
    x = np.stack([np.concatenate([workloads.rank_buffer(spec, r, (c * L) // N, (c * L) // N + win, threads=1)
                                  for c in range(N)]) for r in range(N)])
    return x, idx, L


def _chunk_windows(L: int, n_chunks: int, win: int):
    import numpy as np

    return np.concatenate([np.arange((c * L) // n_chunks, min((c * L) // n_chunks + win, L))
                           for c in range(n_chunks)]).astype(np.int64)


def _sample_values(kind: str, n: int, k: int, seed: int = 0):
    """[n, k] sample values with a workload's distribution ("normal" N(0, 1e-3^2),
    "uniform" [-1, 1], both rounded to fp32; "normal_bf16" further rounded to
    bf16 bits). Drawn for the baseline sample only: the oracle's time does
    not depend on the values."""
    import numpy as np

    rng = np.random.default_rng(seed)
    if kind == "uniform":
        return rng.uniform(-1.0, 1.0, (n, k)).astype(np.float32)
    x = (rng.standard_normal((n, k)) * 1e-3).astype(np.float32)
    if kind == "normal_bf16":
        import workloads

        return workloads.f32_to_bf16_bits_torch(x.reshape(-1)).reshape(n, k)
    return x


def _oracle_call(task):
    """One call of the oracle on a sample; returns the sampled bytes per rank."""
    from oracle import buckets, numerics, schedules

    kind = task["kind"]
    if kind == "ring":
        schedules.ring_allreduce(task["x"], idx=task.get("idx"), L=task.get("L"))
    elif kind == "rabenseifner":
        schedules.rabenseifner_allreduce(task["x"], idx=task.get("idx"), L=task.get("L"))
    elif kind == "hier_bf16":
        xf = numerics.bf16_to_f32(task["x"])
        schedules.hierarchical_allreduce(xf, task["group_size"], idx=task["idx"], L=task["L"],
                                         finish=schedules.finish_bf16())
    elif kind == "buckets":
        for bucket, grads, windows in task["buckets"]:
            buckets.sync_bucket(grads, bucket, task["counts"], task["scale"], windows=windows)
    else:
        raise ValueError(kind)
    return task["bytes_per_rank"]


def _oracle_loop(args):
    """Repeat the oracle call on the sample for `seconds`; returns
    (repetitions, elapsed seconds, sampled bytes per rank)."""
    task, seconds = args
    reps, t0 = 0, time.perf_counter()
    while True:
        per_rank = _oracle_call(task)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return reps, el, per_rank


def _headline_task(win: int):
    x, idx, L = _headline_sample(win)
    return {"kind": "ring", "x": x, "idx": idx, "L": L, "bytes_per_rank": idx.size * 4}


def _ring_n4_task():
    import workloads

    spec = workloads.RING_N4_INT
    x = workloads.all_ranks(spec)
    return {"kind": "ring", "x": x, "bytes_per_rank": spec.count * 4}, \
        "the whole workload (4 ranks x 1,048,576 values, seeded as the GPU's inputs), step-by-step ring simulation"


def _hier_task(win: int = 8192):
    import workloads

    spec = workloads.HIER_2X8_BF16
    N, L = spec.n_ranks, spec.count
    idx = _chunk_windows(L, N, win)  # the 16 sub-chunks of the 8 slices x 2 groups
    x = _sample_values("normal_bf16", N, idx.size)
    return ({"kind": "hier_bf16", "x": x, "idx": idx, "L": L, "group_size": spec.group_size,
             "bytes_per_rank": idx.size * 2},
            f"16 ranks x {idx.size} bf16 elements ({win} at the start of each of the 16 sub-chunks), "
            "hierarchical simulation (8-rank ring reduce-scatter, 2-rank ring all-reduce of each slice, "
            "8-rank all-gather) with fp32 partials and one bf16 rounding")


def _bucket_task(win: int = 2048):
    """A sample of the bucketed sync: one window at the start of every ring
    chunk of four buckets, one of each shape (a lone FFN matrix, the
    norm2+Wo+Wv+Wk bucket, the Wq+norm1 bucket, and the embedding)."""
    import numpy as np

    import workloads
    from oracle import buckets as ob

    spec = workloads.BUCKETED_N8
    N = spec.n_ranks
    counts = [c for _, c in workloads.transformer_tensors()]
    plan = ob.bucket_plan(counts, 2, spec.extra["cap_bytes"])
    chosen, seen = [], set()
    for b in plan:
        shape = tuple(counts[t] for t in b)
        if shape not in seen:
            seen.add(shape)
            chosen.append(b)
    parts, n_el = [], 0
    seed = 0
    for b in chosen:
        offs = ob.bucket_offsets(b, counts)
        Lb = sum(counts[t] for t in b)
        windows = []
        for c in range(N):
            p = (c * Lb) // N
            t = max((t for t in b if offs[t] <= p), key=lambda t: offs[t])
            lo = p - offs[t]
            windows.append((t, lo, min(counts[t], lo + win)))
        k = sum(hi - lo for _, lo, hi in windows)
        vals = _sample_values("normal_bf16", N, k, seed)
        seed += 1
        grads = []
        for r in range(N):
            d, pos = {}, 0
            for t, lo, hi in windows:
                d[(t, lo)] = np.ascontiguousarray(vals[r, pos:pos + hi - lo])
                pos += hi - lo
            grads.append(d)
        parts.append((b, grads, windows))
        n_el += k
    return ({"kind": "buckets", "buckets": parts, "counts": counts, "scale": 1.0 / N, "bytes_per_rank": n_el * 2},
            f"8 ranks x {n_el} bf16 elements: {win} at the start of every ring chunk of {len(chosen)} buckets "
            "(one of each shape), bucketed sync simulation (widen, 8-rank ring in fp32, x1/8, bf16)")


def _sweep_task(n: int, count: int, algo: str = "ring"):
    win = max(1024, 65536 // n)
    if count <= win * n:
        idx, k = None, count
    else:
        idx = _chunk_windows(count, n, win)
        k = idx.size
    x = _sample_values("uniform", n, k)
    task = {"kind": algo, "x": x, "idx": idx, "L": None if idx is None else count, "bytes_per_rank": k * 4}
    what = "the whole buffers" if idx is None else f"{win} elements at the start of each of the {n} chunks"
    return task, f"{n} ranks x {k} fp32 elements ({what}), step-by-step {algo} simulation"


def cpu_baselines(tasks, seconds, pool_size):
    """Time each (name, task, sample text) on `pool_size` spawned processes, every
    process repeating the task's oracle call for `seconds`; returns
    {name: cpu_baseline dict}."""
    import multiprocessing as mp

    out = {}
    ctx = mp.get_context("spawn")  # this process has initialised CUDA: no fork
    with ctx.Pool(pool_size) as pool:
        for name, task, sample in tasks:
            res = pool.map(_oracle_loop, [(task, seconds)] * pool_size)
            wall = max(e for _, e, _ in res)
            value = sum(r * b for r, _, b in res) / wall / 1e9
            reps = sum(r for r, _, _ in res)
            out[name] = {"value": round(value, 6), "unit": UNIT, "cores": pool_size, "kind": "oracle",
                         "sample": f"{sample}; {pool_size} processes each repeating it for {seconds:.0f} s "
                                   f"({reps} calls in all); algbw = sampled per-rank bytes / time"}
    return out


def cpu_baseline(seconds: float = 10.0):
    """The oracle (step-by-step ring simulation in numpy) on a bounded sample of
    the headline workload, one 16 Ki-element window per chunk of every rank:
    on one core, then as one process per host core, each running the same
    sample (elements are independent, so cores multiply the throughput)."""
    win = 16 * 1024
    task = _headline_task(win)
    reps, el, per_rank = _oracle_loop((task, seconds))
    one = per_rank * reps / el / 1e9
    procs = max(1, os.cpu_count() or 1)
    res = cpu_baselines([("headline", task, "")], seconds, procs)["headline"]
    res["value_one_core"] = round(one, 6)
    res["sample"] = (f"16 ranks x {task['idx'].size} fp32 elements ({win} per chunk, all 16 chunks) of the "
                     f"192 MiB workload, step-by-step ring simulation; {procs} processes each repeating it for "
                     f"{seconds:.0f} s (one core alone: {reps} repetitions in {el:.1f} s); algbw = sampled "
                     f"per-rank bytes / time")
    return res


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


# ------------------------------------------------------------------ GPU timing of one case


def event_ms(fn, stream, iters: int, warmup: int, reps: int = 1) -> float:
    """Median over `iters` timings of `reps` back-to-back calls of `fn`, in ms
    per call: CUDA events recorded on `stream` (the stream `fn` launches on),
    after `warmup` untimed calls and a device synchronise."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b) / reps)
    times.sort()
    return times[len(times) // 2]


def l2_bytes() -> int:
    import torch

    return torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size


def figures(ms: float, n: int, bytes_per_rank: int, hbm_bytes: int, peak: float, collective="allreduce",
            **extra) -> dict:
    """The reported numbers of one timed path: time, algbw = S/T, busbw (the
    nccl-tests factor: 2(N-1)/N for all-reduce, (N-1)/N for its halves), the
    algorithmic HBM bytes per call and the bandwidth they imply, and the
    fraction of the HBM peak -- only when the traffic is well above the L2
    size (4x); smaller cases are latency and are read in microseconds."""
    algbw = bytes_per_rank / (ms * 1e-3) / 1e9
    factor = 2 * (n - 1) / n if collective == "allreduce" else (n - 1) / n
    achieved = hbm_bytes / (ms * 1e-3) / 1e9
    resident = hbm_bytes <= 4 * l2_bytes()
    out = {"us" if ms < 0.1 else "ms": round(ms * 1e3, 2) if ms < 0.1 else round(ms, 4),
           "algbw": round(algbw, 2), "busbw": round(algbw * factor, 2), "hbm_bytes": int(hbm_bytes),
           "achieved_gbs": round(achieved, 1),
           "frac_of_hbm": None if resident else round(achieved / peak, 4)}
    if resident:
        out["note"] = "traffic within 4x the L2: latency, read in us"
    out.update(extra)
    return out


def time_case(n, count, dtype="f32", algo="fused", order="ring", group_size=0, iters=20, warmup=5,
              reps=None, graph=False, collective="allreduce", sm_budget=0, kernel="auto", torus_dims=(0, 0, 0),
              bound=False, bufs=None):
    """Time one plan on device-filled (or given) buffers, out of place."""
    import torch

    import gradient_sync_gb300 as g

    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    esz = 4 if dtype == "f32" else 2
    if bufs is None:
        bufs = [torch.rand(count, device="cuda").to(tdt) for _ in range(n)]
    outs = [torch.empty_like(b) for b in bufs]
    plan = g.ar_plan(n, count, dtype, algo, group_size=group_size, order=order, collective=collective,
                     sm_budget=sm_budget, kernel=kernel, torus_dims=torus_dims)
    ws = g.workspace_for(plan)
    st = plan.stats
    nbytes = n * count * esz
    if reps is None:  # calls per timing: enough work to resolve the time of small cases, and
        # at least 3 back to back, so that one call's launch from Python is not timed alone
        reps = max(3, min(1000, (256 * MiB) // max(1, 2 * nbytes), 4000 // max(1, st["launches"])))
    stream = torch.cuda.current_stream()
    handle = int(stream.cuda_stream)

    def call():
        g.ar_execute(plan, bufs, outs=outs, workspace=ws, stream=handle)

    fn = call
    if bound:  # a persistent collective: bound once, replayed from Python with one call each
        bnd = g.ar_bind(plan, bufs, outs=outs, workspace=ws)

        def fn():
            g.ar_execute_bound(bnd, stream=handle)
    if graph:  # the reps calls captured once into a CUDA graph: device time without host launch cost
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            cg.capture_begin()
            for _ in range(reps):
                g.ar_execute(plan, bufs, outs=outs, workspace=ws, stream=side)
            cg.capture_end()
        stream.wait_stream(side)
        ms = event_ms(cg.replay, stream, iters, 1) / reps
    else:
        ms = event_ms(fn, stream, iters, warmup, reps)
    S = count * esz
    res = {"n": n, "collective": collective, "sm_budget": sm_budget, "kernel": kernel, "bytes_per_rank": S,
           "dtype": dtype, "algo": algo, "order": order if algo == "fused" else None,
           "timing": "cuda graph" if graph else ("bound, replayed from python" if bound else "launched from python"),
           "group_size": group_size or None, "torus_dims": list(torus_dims) if algo == "torus" else None,
           "us": round(ms * 1e3, 2), "steps": st["steps"], "launches": st["launches"]}
    hbm = st["hbm_bytes"]
    if algo != "fused" and collective == "allgather" and n > 1:  # out of place: each rank's own chunk
        hbm += count * esz * (2 if st["launches"] == 1 else 1)  # also goes to its output (ar.h)
    f = figures(ms, n, S, hbm, measured_peaks()[0], collective)
    res.update({k: v for k, v in f.items() if k not in ("ms", "us")})
    res["hbm_frac"] = res.pop("frac_of_hbm")
    del bufs, outs, ws
    torch.cuda.empty_cache()
    return res


def bucket_ranges(counts, cap_bytes=25 * MiB):
    """(first tensor, end tensor, elements) of every bucket, in sync order."""
    import gradient_sync_gb300 as g

    of, nb = g.ar_bucket_plan(counts, 2, cap_bytes)
    ranges = []
    for b in range(nb):
        ts = [t for t in range(len(counts)) if of[t] == b]
        ranges.append((min(ts), max(ts) + 1, sum(counts[t] for t in ts)))
    return ranges


def bucket_sync(grads, counts, n, path, stream_handle, cap_bytes=25 * MiB):
    """The bucketed gradient sync of `grads` ([rank][tensor] bf16, in place,
    sum x 1/n) as one callable: every bucket either packed, ring all-reduced
    in fp32 and unpacked ("pack"), or all-reduced in one fused pass over the
    gradients ("fused"). Returns (sync, algorithmic HBM bytes, launches,
    buckets, state to keep alive)."""
    import torch

    import gradient_sync_gb300 as g

    ranges = bucket_ranges(counts, cap_bytes)
    table = g.TensorTable(grads, counts)  # marshalled once, as a DDP reducer builds its buckets once
    scale = 1.0 / n
    if path == "pack":
        max_lb = max(lb for _, _, lb in ranges)
        bucket_t = [torch.empty(max_lb, dtype=torch.float32, device="cuda") for _ in range(n)]
        bucket = g._ptrs(bucket_t)
        plans = {lb: g.ar_plan(n, lb, "f32", "ring") for _, _, lb in ranges}
        hbm = sum(n * lb * (2 + 4) * 2 + plans[lb].stats["hbm_bytes"] for _, _, lb in ranges)
        launches = sum(plans[lb].stats["launches"] + 2 for _, _, lb in ranges)

        def sync():
            for lo, hi, lb in ranges:
                g.ar_bucket_pack(table, None, lo, hi, "bf16", bucket, stream=stream_handle)
                g.ar_execute(plans[lb], bucket_t, stream=stream_handle)
                g.ar_bucket_unpack(bucket, scale, "bf16", table, None, lo, hi, stream=stream_handle)
        keep = (table, bucket_t, bucket, plans)
    else:
        hbm = 2 * n * sum(counts) * 2
        launches = len(ranges)

        def sync():
            for lo, hi, _ in ranges:
                g.ar_bucket_allreduce(table, None, lo, hi, "bf16", scale, stream=stream_handle)
        keep = (table,)
    return sync, hbm, launches, len(ranges), keep


def time_buckets(n=8, path="fused", iters=5, warmup=2, cap_bytes=25 * MiB, layers=16):
    """Time one bucketed gradient sync of the transformer (16 layers unless
    `layers`; hidden 2048, FFN 8192, vocab 32000; bf16 gradients; 25 MiB
    buckets in reverse layer order; sum scaled by 1/n) on device-filled
    gradients."""
    import torch

    import workloads

    counts = [c for _, c in workloads.transformer_tensors(layers=layers)]
    grads = [[torch.randn(c, device="cuda").to(torch.bfloat16) for c in counts] for _ in range(n)]
    stream = torch.cuda.current_stream()
    sync, hbm, launches, nb, keep = bucket_sync(grads, counts, n, path, int(stream.cuda_stream), cap_bytes)
    ms = event_ms(sync, stream, iters, warmup, 2)
    S = sum(counts) * 2
    res = {"workload": f"bucketed {layers}-layer transformer", "n": n, "path": path, "buckets": nb,
           "bytes_per_rank": S, "launches": launches}
    res.update(figures(ms, n, S, hbm, measured_peaks()[0]))
    del grads, keep
    torch.cuda.empty_cache()
    return res


def compressed_hbm_bytes(n, count, dtype="f32", block=128, path="fused", ef=True):
    """Algorithmic HBM bytes of one compressed all-reduce: every element and
    scale read or written counted once per access at its storage width. Fused:
    gradients read, results written to every rank, residuals read and
    rewritten. Two calls: the compressor reads gradients (and residuals) and
    writes codes, scales (and residuals); the reducer reads codes and scales
    and writes every rank's result."""
    esz = 4 if dtype == "f32" else 2
    nb = (count + block - 1) // block
    res = 8 * n * count if ef else 0
    if path == "fused":
        return n * count * 2 * esz + res
    return n * count * (esz + 1) + 4 * n * nb + res + n * count + 4 * n * nb + n * count * esz


def compressed_call(grads, outs, block, dtype, res, n, path, stream_handle, codes=None, scales=None):
    """One blockwise INT8 compressed all-reduce (sum x 1/n) as a callable: the
    fused pass, or the compressor and the reducer as two calls with the
    messages in HBM between them."""
    import gradient_sync_gb300 as g

    if path == "two":
        def call():
            g.ar_compress(grads, codes, scales, block, dtype=dtype, residuals=res, stream=stream_handle)
            g.ar_compressed_reduce(codes, scales, outs, block, scale=1.0 / n, out_dtype=dtype,
                                   stream=stream_handle)
    else:
        def call():
            g.ar_compressed_allreduce(grads, block, dtype=dtype, residuals=res, scale=1.0 / n, outs=outs,
                                      stream=stream_handle)
    return call


def time_compressed(n=16, count=50_331_648, dtype="f32", block=128, path="fused", ef=True, iters=10, warmup=3):
    """Time the blockwise INT8 compressed all-reduce (error feedback on when
    ``ef``) on device-filled gradients."""
    import torch

    import gradient_sync_gb300 as g

    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    grads = [torch.randn(count, device="cuda").mul_(1e-3).to(tdt) for _ in range(n)]
    outs = [torch.empty_like(t) for t in grads]
    res = [torch.zeros(count, device="cuda") for _ in range(n)] if ef else None
    nb, _ = g.ar_compress_sizes(count, block)
    codes = scales = None
    if path == "two":
        codes = [torch.empty(count, dtype=torch.int8, device="cuda") for _ in range(n)]
        scales = [torch.empty(nb, dtype=torch.float32, device="cuda") for _ in range(n)]
    stream = torch.cuda.current_stream()
    call = compressed_call(grads, outs, block, dtype, res, n, path, int(stream.cuda_stream), codes, scales)
    hbm = compressed_hbm_bytes(n, count, dtype, block, path, ef)
    reps = max(3, min(200, (256 * MiB) // max(1, hbm)))
    ms = event_ms(call, stream, iters, warmup, reps)
    S = count * (4 if dtype == "f32" else 2)
    out = {"workload": "blockwise INT8 compressed all-reduce", "n": n, "count": count, "dtype": dtype,
           "block": block, "path": path, "error_feedback": ef, "launches": 1 if path == "fused" else 2,
           "us": round(ms * 1e3, 2)}
    f = figures(ms, n, S, hbm, measured_peaks()[0])
    out.update({k: v for k, v in f.items() if k not in ("ms", "us")})
    out["hbm_frac"] = out.pop("frac_of_hbm")
    del grads, outs, res
    torch.cuda.empty_cache()
    return out


def sweep(out=sys.stdout, max_total=64 * GiB, graph=False):
    """The size/algorithm sweep: N in {2,4,8,16,64} x 1 KiB..1 GiB per rank
    (powers of 4, N*S <= 64 GiB), fused (ring and rank order), ring and
    Rabenseifner, fp32."""
    for n in (2, 4, 8, 16, 64):
        for k in range(11):
            S = KiB * 4 ** k
            if n * S > max_total:
                continue
            for algo, order in (("fused", "ring"), ("fused", "rank"), ("ring", "ring"), ("rabenseifner", "ring")):
                iters = 10 if n * S < GiB else 5
                res = time_case(n, S // 4, "f32", algo, order, iters=iters, warmup=3, graph=graph)
                print(json.dumps(res), file=out, flush=True)


# ------------------------------------------------------------------ the other workloads


def device_normal_bf16(count: int, seed: int, dev):
    """N(0, 1e-3^2) values drawn on the device (torch's generator, seeded),
    rounded to bf16 (round to nearest even)."""
    import torch

    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    return torch.randn(count, generator=gen, device=dev).mul_(1e-3).to(torch.bfloat16)


def device_uniform(count: int, seed: int, dev):
    """uniform [-1, 1) fp32 values drawn on the device (torch's generator, seeded)."""
    import torch

    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    return torch.rand(count, generator=gen, device=dev).mul_(2.0).sub_(1.0)


def run_workloads(dev, stream, peak, k_big: int, warmup: int):
    """Time every path of the other workloads on `stream`; returns
    ({workload: entry}, [(name, oracle task, sample text)])."""
    import numpy as np
    import torch

    import gradient_sync_gb300 as g
    import workloads

    handle = int(stream.cuda_stream)
    out, tasks = {}, []

    def plan_path(plan, bufs, outs, n, S, iters, reps=3, ws=None, **extra):
        ws = g.workspace_for(plan) if ws is None else ws
        st = plan.stats
        ms = event_ms(lambda: g.ar_execute(plan, bufs, outs=outs, workspace=ws, stream=handle), stream,
                      iters, warmup, reps)
        return figures(ms, n, S, st["hbm_bytes"], peak, steps=st["steps"], launches=st["launches"], **extra)

    # 4 ranks x 1,048,576 integer-valued fp32 (16 MiB in all: L2-resident, latency-bound)
    spec = workloads.RING_N4_INT
    N, L = spec.n_ranks, spec.count
    bufs = [torch.from_numpy(workloads.rank_buffer(spec, r)).to(dev) for r in range(N)]
    outs = [torch.empty_like(b) for b in bufs]
    out["ring_n4_int"] = {
        "workload": spec.name, "n_ranks": N, "count_per_rank": L, "bytes_per_rank": L * 4,
        "inputs": "seeded host values (the tests' recipe), copied to the device once",
        "timing": "100 back-to-back calls launched from Python per timing, median of 10",
        "paths": {
            "ring_steps": plan_path(g.ar_plan(N, L, "f32", "ring"), bufs, outs, N, L * 4, 10, 100),
            "fused_ring_order": plan_path(g.ar_plan(N, L, "f32", "fused", order="ring"), bufs, outs, N, L * 4,
                                          10, 100)}}
    task, sample = _ring_n4_task()
    tasks.append(("ring_n4_int", task, sample))
    del bufs, outs

    # 16 ranks as 2 groups of 8, 96 Mi bf16 each: hierarchical steps (fp32
    # partials in the workspace) and the fused pass in two orders
    spec = workloads.HIER_2X8_BF16
    N, L, G = spec.n_ranks, spec.count, spec.group_size
    bufs = [device_normal_bf16(L, r, dev) for r in range(N)]
    outs = [torch.empty_like(b) for b in bufs]
    S = L * 2
    out["hier_2x8_bf16"] = {
        "workload": spec.name, "n_ranks": N, "group_size": G, "count_per_rank": L, "bytes_per_rank": S,
        "inputs": "device-filled: torch.randn on the GPU (seed = rank) x 1e-3, rounded to bf16",
        "timing": f"median of {k_big} timings of 3 calls back to back, after {warmup} warm-ups, out of place; "
                  "traffic > 40x the L2",
        "paths": {
            "hier_steps": plan_path(g.ar_plan(N, L, "bf16", "hier", group_size=G), bufs, outs, N, S, k_big),
            "fused_hier_order": plan_path(g.ar_plan(N, L, "bf16", "fused", group_size=G, order="hier"), bufs,
                                          outs, N, S, k_big),
            "fused_rank_order": plan_path(g.ar_plan(N, L, "bf16", "fused", order="rank"), bufs, outs, N, S,
                                          k_big)}}
    # the blockwise INT8 compressed all-reduce of the same bf16 gradients,
    # without error feedback (block 128, sum x 1/16): fused pass and two calls
    block = 128
    n_sc, _ = g.ar_compress_sizes(L, block)
    codes = [torch.empty(L, dtype=torch.int8, device=dev) for _ in range(N)]
    scales = [torch.empty(n_sc, dtype=torch.float32, device=dev) for _ in range(N)]
    for name, path in (("compressed_int8_fused", "fused"), ("compressed_int8_two_calls", "two")):
        fn = compressed_call(bufs, outs, block, "bf16", None, N, path, handle, codes, scales)
        ms = event_ms(fn, stream, k_big, warmup, 3)
        out["hier_2x8_bf16"]["paths"][name] = figures(
            ms, N, S, compressed_hbm_bytes(N, L, "bf16", block, path, False), peak, block=block,
            error_feedback=False, launches=1 if path == "fused" else 2)
    del codes, scales
    task, sample = _hier_task()
    tasks.append(("hier_2x8_bf16", task, sample))
    del bufs, outs
    torch.cuda.empty_cache()

    # 8 ranks, the 16-layer transformer's bf16 gradients in 25 MiB buckets
    spec = workloads.BUCKETED_N8
    N = spec.n_ranks
    counts = [c for _, c in workloads.transformer_tensors()]
    grads = [[device_normal_bf16(c, 1000 * r + t, dev) for t, c in enumerate(counts)] for r in range(N)]
    S = sum(counts) * 2
    paths = {}
    for path in ("fused", "pack"):
        sync, hbm, launches, nb, keep = bucket_sync(grads, counts, N, path, handle)
        ms = event_ms(sync, stream, max(3, k_big // 2), min(warmup, 3), 2)
        paths["fused_no_pack" if path == "fused" else "pack_ring_unpack"] = figures(
            ms, N, S, hbm, peak, buckets=nb, launches=launches)
        del keep
    out["buckets_n8_transformer"] = {
        "workload": spec.name, "n_ranks": N, "tensors": len(counts), "count_per_rank": sum(counts),
        "bytes_per_rank": S,
        "inputs": "device-filled: torch.randn on the GPU (one seed per rank and tensor) x 1e-3, rounded to bf16",
        "timing": f"median of {max(3, k_big // 2)} timings of 2 whole syncs back to back (every bucket, in "
                  "place) after warm-up",
        "paths": paths}
    task, sample = _bucket_task()
    tasks.append(("buckets_n8_transformer", task, sample))
    del grads
    torch.cuda.empty_cache()

    # a launch held to a few SMs (sm_budget, what the overlap uses): the
    # fused ring-order pass of the headline's size on 32 and 64 SMs' worth of
    # CTAs, then the bucketed sync behind a synthetic backward (8 ranks, the
    # 16-layer model's bf16 gradients, 8192 tokens, 32 SMs)
    n, L = 16, 50_331_648
    bufs = [device_uniform(L, r, dev) for r in range(n)]
    outs = [torch.empty_like(b) for b in bufs]
    k = max(3, k_big // 2)
    paths = {}
    for b in (32, 64):
        plan = g.ar_plan(n, L, "f32", "fused", order="ring", sm_budget=b)
        paths[f"fused_ring_order_{b}_sms"] = plan_path(plan, bufs, outs, n, L * 4, k, sm_budget=b)
    out["sm_budget_n16_192mib"] = {
        "workload": "fused ring-order all-reduce, 16 ranks x 192 MiB fp32, held to an SM budget", "n_ranks": n,
        "count_per_rank": L, "bytes_per_rank": L * 4,
        "inputs": "device-filled: torch.rand on the GPU (seed = rank), mapped to [-1, 1)",
        "timing": f"median of {k} timings of 3 calls back to back", "paths": paths}
    del bufs, outs
    torch.cuda.empty_cache()
    from gradient_sync_gb300.overlap import time_overlap

    with torch.cuda.stream(stream):
        ovl = time_overlap(n_ranks=8, tokens=8192, sm_budget=32, iters=5)
    out["overlap_8192_tokens_32_sms"] = {
        **ovl, "timing": "median of 5 timings each: the backward alone, the sync alone, both in sequence, "
                         "both overlapped (sync on a second stream)"}
    torch.cuda.empty_cache()

    # the sweep's corners: 2, 16 and 64 ranks x 1 GiB fp32 (bandwidth) and
    # 16 ranks x 1 KiB (latency)
    sweep_out = {}
    for n in (2, 16, 64):
        L = GiB // 4
        bufs = [device_uniform(L, r, dev) for r in range(n)]
        outs = [torch.empty_like(b) for b in bufs]
        k = max(3, k_big // 4)
        paths = {}
        for name, plan in (("fused_ring_order", g.ar_plan(n, L, "f32", "fused", order="ring")),
                           ("fused_rank_order", g.ar_plan(n, L, "f32", "fused", order="rank")),
                           ("ring_steps", g.ar_plan(n, L, "f32", "ring")),
                           ("rabenseifner_steps", g.ar_plan(n, L, "f32", "rabenseifner"))):
            paths[name] = plan_path(plan, bufs, outs, n, GiB, k)
        sweep_out[f"n{n}_1gib"] = {"n_ranks": n, "bytes_per_rank": GiB,
                                   "timing": f"median of {k} timings of 3 calls back to back",
                                   "paths": paths}
        task, sample = _sweep_task(n, L)
        tasks.append((f"sweep_n{n}_1gib", task, sample))
        del bufs, outs
        torch.cuda.empty_cache()
    n, L = 16, 256
    bufs = [device_uniform(L, r, dev) for r in range(n)]
    outs = [torch.empty_like(b) for b in bufs]
    paths = {}
    for name, algo in (("fused_ring_order", "fused"), ("ring_steps", "ring"), ("rabenseifner_steps", "rabenseifner")):
        plan = g.ar_plan(n, L, "f32", algo)
        bnd = g.ar_bind(plan, bufs, outs=outs)
        ms = event_ms(lambda: g.ar_execute_bound(bnd, stream=handle), stream, 10, 5, 100)
        paths[name] = figures(ms, n, KiB, plan.stats["hbm_bytes"], peak, steps=plan.stats["steps"],
                              launches=plan.stats["launches"])
        del bnd
    sweep_out["n16_1kib"] = {"n_ranks": n, "bytes_per_rank": KiB,
                             "timing": "bound once (ar_bind), 100 ar_execute_bound calls back to back per "
                                       "timing, median of 10", "paths": paths}
    task, sample = _sweep_task(n, L)
    tasks.append(("sweep_n16_1kib", task, sample))
    del bufs, outs
    out["sweep"] = {"workload": "size/algorithm sweep corners, fp32 uniform [-1, 1]",
                    "inputs": "device-filled: torch.rand on the GPU (seed = rank), mapped to [-1, 1)",
                    "points": sweep_out}
    torch.cuda.empty_cache()
    return out, tasks


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
    block = 128
    res = [torch.zeros(L, dtype=torch.float32, device=dev) for _ in range(N)]
    n_sc, _ = g.ar_compress_sizes(L, block)
    codes = [torch.empty(L, dtype=torch.int8, device=dev) for _ in range(N)]
    scales = [torch.empty(n_sc, dtype=torch.float32, device=dev) for _ in range(N)]
    handle = int(stream.cuda_stream)
    for name, path, launches in (("compressed_int8_fused", "fused", 1), ("compressed_int8_two_calls", "two", 2)):
        fn = compressed_call(bufs, outs, block, "f32", res, N, path, handle, codes, scales)
        k = max(5, args.steps // 20)
        ms_c = timed(dist, fn, sync, k, args.warmup, local if dist else None, event_timer) / k
        hb = compressed_hbm_bytes(N, L, "f32", block, path, True)
        bw = hb / (ms_c * 1e-3) / 1e9
        executors[name] = {"ms": round(ms_c, 4), "algbw": round(S / (ms_c * 1e-3) / 1e9, 2), "block": block,
                           "error_feedback": True, "launches": launches, "hbm_bytes": hb,
                           "achieved_gbs": round(bw, 1), "frac_of_hbm": round(bw / hbm_peak, 4)}
    del res, codes, scales
    torch.cuda.empty_cache()

    # end to end: pinned host buffers in and out through ar_execute_host
    host_in = [torch.from_numpy(h).pin_memory() for h in host]
    host_out = [torch.empty(L, dtype=torch.float32).pin_memory() for _ in range(N)]
    del host

    def e2e_step():
        g.ar_execute_host(fused, host_in, host_out, outs, stream=handle)

    k_e2e = max(3, min(10, args.steps // 100))
    ms_e2e = timed(dist, e2e_step, sync, k_e2e, 1, local if dist else None) / k_e2e
    got = host_out[3][: 1 << 16].numpy()
    assert np.isfinite(got).all()
    del host_in, host_out, bufs, outs
    torch.cuda.empty_cache()

    # the other workloads, each against its own algorithmic bytes
    others, tasks = run_workloads(dev, stream, hbm_peak, max(5, min(20, args.steps // 20)), args.warmup)
    latency = {"workload": "16 ranks x 1 KiB fp32, ar_bind once, ar_execute_bound per call, back to back"}
    for algo in ("ring", "rabenseifner"):
        p = others["sweep"]["points"]["n16_1kib"]["paths"][f"{algo}_steps"]
        latency[algo] = {"us_per_call": p["us"], "steps": p["steps"], "launches": p["launches"]}

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
                     "frac": round(achieved / hbm_peak, 4), "traffic": profiled_traffic(st["hbm_bytes"]),
                     "kernel": "fused_flat_kernel<fp32, seq>", "peak_kind": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": st["hbm_bytes"]},
        "executors": executors,
        "workloads": others,
        "latency": latency,
        "e2e": {"value": round(S * world / (ms_e2e * 1e-3) / 1e9, 2), "unit": UNIT,
                "h2d_bytes_per_step": N * S, "d2h_bytes_per_step": N * S, "ms_per_step": round(ms_e2e, 3),
                "api": "ar_execute_host: pinned host buffers read and written by the kernel over NVLink-C2C"},
        "gpu_launches": args.steps * st["launches"],
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
        procs = max(1, os.cpu_count() or 1)
        for name, base in cpu_baselines(tasks, 3.0, procs).items():
            if name.startswith("sweep_"):
                others["sweep"]["points"][name[len("sweep_"):]]["cpu_baseline"] = base
            else:
                others[name]["cpu_baseline"] = base
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


def run_single(a):
    """The single-measurement modes (--case, --sweep, --buckets, --overlap, --compressed)."""
    from gradient_sync_gb300 import build

    build.build()
    if a.sweep:
        sweep(graph=a.graph)
    elif a.compressed:
        print(json.dumps(time_compressed(a.n, a.count, a.dtype, a.block, a.compressed, not a.no_ef,
                                         a.iters, a.warmup)))
    elif a.buckets:
        print(json.dumps(time_buckets(path=a.buckets, iters=a.iters, warmup=min(a.warmup, 3), layers=a.layers)))
    elif a.overlap:
        from gradient_sync_gb300.overlap import time_overlap

        print(json.dumps(time_overlap(n_ranks=a.n, tokens=a.tokens, sm_budget=a.sm_budget, iters=a.iters,
                                      warmup=min(a.warmup, 3), kernel=a.kernel)))
    else:
        print(json.dumps(time_case(a.n, a.count, a.dtype, a.algo, a.order, a.group_size, a.iters, a.warmup,
                                   a.reps, graph=a.graph, collective=a.collective, sm_budget=a.sm_budget,
                                   kernel=a.kernel, torus_dims=tuple(int(v) for v in a.dims.split(",")),
                                   bound=a.bound)))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=None, help="warm-up steps (default 10; 5 for single cases)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timings")
    single = ap.add_argument_group("single measurements")
    single.add_argument("--case", action="store_true", help="time one plan (--algo, --n, --count, ...)")
    single.add_argument("--sweep", action="store_true", help="the size/algorithm sweep, one line per case")
    single.add_argument("--buckets", choices=["fused", "pack"], default=None)
    single.add_argument("--overlap", action="store_true", help="bucketed sync overlapped with a synthetic backward")
    single.add_argument("--compressed", choices=["fused", "two"], default=None,
                        help="blockwise INT8 compressed all-reduce (fused pass or compressor + reducer)")
    single.add_argument("--algo", default="fused")
    single.add_argument("--order", default="ring")
    single.add_argument("--n", type=int, default=16)
    single.add_argument("--count", type=int, default=8 * MiB)
    single.add_argument("--dtype", default="f32")
    single.add_argument("--group-size", type=int, default=0)
    single.add_argument("--collective", default="allreduce", choices=["allreduce", "reduce_scatter", "allgather"])
    single.add_argument("--iters", type=int, default=20)
    single.add_argument("--reps", type=int, default=None)
    single.add_argument("--graph", action="store_true", help="replay the timed calls from a CUDA graph")
    single.add_argument("--bound", action="store_true", help="bind the plan once (ar_bind) and time ar_execute_bound")
    single.add_argument("--tokens", type=int, default=4096)
    single.add_argument("--layers", type=int, default=16, help="transformer layers for --buckets")
    single.add_argument("--sm-budget", type=int, default=0)
    single.add_argument("--kernel", default="auto", choices=["auto", "loads", "bulk"])
    single.add_argument("--dims", default="0,0,0", help="torus dimensions X,Y[,Z] for --algo torus")
    single.add_argument("--block", type=int, default=128)
    single.add_argument("--no-ef", action="store_true", help="compressed all-reduce without error feedback")
    args = ap.parse_args(argv)
    if args.case or args.sweep or args.buckets or args.overlap or args.compressed:
        args.warmup = 5 if args.warmup is None else args.warmup
        run_single(args)
        return
    args.warmup = 10 if args.warmup is None else args.warmup
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

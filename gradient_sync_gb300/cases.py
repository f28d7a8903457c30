"""Run and time one all-reduce case, or the size/algorithm sweep, on the GPU.

    python -m gradient_sync_gb300.cases --algo fused --order ring --n 16 --count 8388608 --iters 3
    python -m gradient_sync_gb300.cases --sweep > sweep.jsonl
    python -m gradient_sync_gb300.cases --buckets fused|pack --iters 5
    python -m gradient_sync_gb300.cases --overlap --n 8 --tokens 4096 --sm-budget 32 --iters 5
    python -m gradient_sync_gb300.cases --compressed fused|two --n 16 --count 50331648 --block 128

Each timed case prints one JSON line: time per call (median of CUDA-event
timings on the launching stream, after warm-up), algbw = S/T, busbw =
algbw * 2(N-1)/N, and the achieved algorithmic HBM bandwidth of the plan
(ar_plan_stats.hbm_bytes / T). Inputs are random device data (timing does not
depend on values); buffers are out of place so every call reduces the same
data. Small cases run many calls per timing so that the per-call time is
resolved; %HBM is only meaningful when N*S is well above the L2 size.
"""

from __future__ import annotations

import argparse
import json
import os
import sys

import torch

import gradient_sync_gb300 as g

KiB, MiB, GiB = 1 << 10, 1 << 20, 1 << 30


def hbm_peak():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    try:
        with open(os.path.join(root, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"])
    except (OSError, KeyError, ValueError):
        return 6800.0


def time_case(n, count, dtype="f32", algo="fused", order="ring", group_size=0, iters=20, warmup=5,
              reps=None, graph=False, collective="allreduce", sm_budget=0, kernel="auto", torus_dims=(0, 0, 0),
              bound=False):
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    esz = 4 if dtype == "f32" else 2
    bufs = [torch.rand(count, device="cuda").to(tdt) for _ in range(n)]
    outs = [torch.empty_like(b) for b in bufs]
    plan = g.ar_plan(n, count, dtype, algo, group_size=group_size, order=order, collective=collective,
                     sm_budget=sm_budget, kernel=kernel, torus_dims=torus_dims)
    ws = g.workspace_for(plan)
    st = plan.stats
    nbytes = n * count * esz
    if reps is None:  # calls per timing: enough work to resolve the time of small cases
        reps = max(1, min(1000, (256 * MiB) // max(1, 2 * nbytes), 4000 // max(1, st["launches"])))
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        g.ar_execute(plan, bufs, outs=outs, workspace=ws)
    torch.cuda.synchronize()
    run = None
    if bound:  # a persistent collective: bound once, replayed from Python with one call each
        bnd = g.ar_bind(plan, bufs, outs=outs, workspace=ws)
        handle = int(stream.cuda_stream)

        def run():
            for _ in range(reps):
                g.ar_execute_bound(bnd, stream=handle)
        run()
        torch.cuda.synchronize()
    if graph:  # the reps calls captured once into a CUDA graph: device time without host launch cost
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            cg.capture_begin()
            for _ in range(reps):
                g.ar_execute(plan, bufs, outs=outs, workspace=ws, stream=side)
            cg.capture_end()
        stream.wait_stream(side)
        cg.replay()
        torch.cuda.synchronize()
        run = cg.replay
    times = []
    for _ in range(iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        if run is not None:
            run()
        else:
            for _ in range(reps):
                g.ar_execute(plan, bufs, outs=outs, workspace=ws)
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b) / reps)
    times.sort()
    ms = times[len(times) // 2]
    S = count * esz
    algbw = S / (ms * 1e-3) / 1e9
    hbm = st["hbm_bytes"] / (ms * 1e-3) / 1e9
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    factor = 2 * (n - 1) / n if collective == "allreduce" else (n - 1) / n  # busbw (primer §4.8)
    res = {"n": n, "collective": collective, "sm_budget": sm_budget, "kernel": kernel, "bytes_per_rank": S, "dtype": dtype, "algo": algo,
           "order": order if algo == "fused" else None,
           "timing": "cuda graph" if graph else ("bound, replayed from python" if bound else "launched from python"),
           "group_size": group_size or None, "torus_dims": list(torus_dims) if algo == "torus" else None,
           "us": round(ms * 1e3, 2), "algbw": round(algbw, 2),
           "busbw": round(algbw * factor, 2), "steps": st["steps"], "launches": st["launches"],
           "hbm_bytes": st["hbm_bytes"], "hbm_gbs": round(hbm, 1),
           "hbm_frac": round(hbm / hbm_peak(), 4) if nbytes > 4 * l2 else None}
    del bufs, outs, ws
    torch.cuda.empty_cache()
    return res


def time_buckets(n=8, path="fused", iters=5, warmup=2, cap_bytes=25 * MiB):
    """Time one bucketed gradient sync of the 16-layer transformer (hidden 2048,
    FFN 8192, vocab 32000; bf16 gradients; 25 MiB buckets in reverse layer
    order; sum scaled by 1/n): every bucket either packed, ring all-reduced in
    fp32 and unpacked ("pack"), or all-reduced in one fused pass over the
    gradients in place ("fused")."""
    import workloads

    counts = [c for _, c in workloads.transformer_tensors()]
    of, nb = g.ar_bucket_plan(counts, 2, cap_bytes)
    ranges = []
    for b in range(nb):
        ts = [t for t in range(len(counts)) if of[t] == b]
        ranges.append((min(ts), max(ts) + 1, sum(counts[t] for t in ts)))
    grads = [[torch.randn(c, device="cuda").to(torch.bfloat16) for c in counts] for _ in range(n)]
    table = g.TensorTable(grads, counts)  # marshalled once, as a DDP reducer builds its buckets once
    stream = int(torch.cuda.current_stream().cuda_stream)
    scale = 1.0 / n
    total = sum(counts)
    if path == "pack":
        max_lb = max(lb for _, _, lb in ranges)
        bucket_t = [torch.empty(max_lb, dtype=torch.float32, device="cuda") for _ in range(n)]
        bucket = g._ptrs(bucket_t)
        plans = {lb: g.ar_plan(n, lb, "f32", "ring") for _, _, lb in ranges}
        hbm = sum(n * lb * (2 + 4) * 2 + plans[lb].stats["hbm_bytes"] for _, _, lb in ranges)
        launches = sum(plans[lb].stats["launches"] + 2 for _, _, lb in ranges)

        def sync():
            for lo, hi, lb in ranges:
                g.ar_bucket_pack(table, None, lo, hi, "bf16", bucket, stream=stream)
                g.ar_execute(plans[lb], bucket_t, stream=stream)
                g.ar_bucket_unpack(bucket, scale, "bf16", table, None, lo, hi, stream=stream)
    else:
        hbm = 2 * n * total * 2
        launches = nb

        def sync():
            for lo, hi, _ in ranges:
                g.ar_bucket_allreduce(table, None, lo, hi, "bf16", scale, stream=stream)
    cur = torch.cuda.current_stream()
    for _ in range(warmup):
        sync()
    torch.cuda.synchronize()
    times = []
    for _ in range(iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        sync()
        b.record(cur)
        b.synchronize()
        times.append(a.elapsed_time(b))
    times.sort()
    ms = times[len(times) // 2]
    S = total * 2
    res = {"workload": "bucketed 16-layer transformer", "n": n, "path": path, "buckets": nb,
           "bytes_per_rank": S, "ms": round(ms, 4), "algbw": round(S / (ms * 1e-3) / 1e9, 2),
           "busbw": round(S / (ms * 1e-3) / 1e9 * 2 * (n - 1) / n, 2), "launches": launches,
           "hbm_bytes": hbm, "hbm_gbs": round(hbm / (ms * 1e-3) / 1e9, 1),
           "hbm_frac": round(hbm / (ms * 1e-3) / 1e9 / hbm_peak(), 4)}
    del grads, table
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


def time_compressed(n=16, count=50_331_648, dtype="f32", block=128, path="fused", ef=True, iters=10, warmup=3):
    """Time the blockwise INT8 compressed all-reduce (error feedback on when
    ``ef``; sum scaled by 1/n): the fused single pass, or the compressor and
    the reducer as two calls with the messages in HBM between them."""
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    grads = [torch.randn(count, device="cuda").mul_(1e-3).to(tdt) for _ in range(n)]
    outs = [torch.empty_like(t) for t in grads]
    res = [torch.zeros(count, device="cuda") for _ in range(n)] if ef else None
    nb, _ = g.ar_compress_sizes(count, block)
    if path == "two":
        codes = [torch.empty(count, dtype=torch.int8, device="cuda") for _ in range(n)]
        scales = [torch.empty(nb, dtype=torch.float32, device="cuda") for _ in range(n)]
        launches = 2

        def call():
            g.ar_compress(grads, codes, scales, block, dtype=dtype, residuals=res)
            g.ar_compressed_reduce(codes, scales, outs, block, scale=1.0 / n, out_dtype=dtype)
    else:
        launches = 1

        def call():
            g.ar_compressed_allreduce(grads, block, dtype=dtype, residuals=res, scale=1.0 / n, outs=outs)
    hbm = compressed_hbm_bytes(n, count, dtype, block, path, ef)
    reps = max(1, min(200, (256 * MiB) // max(1, hbm)))
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    times = []
    for _ in range(iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            call()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b) / reps)
    times.sort()
    ms = times[len(times) // 2]
    S = count * (4 if dtype == "f32" else 2)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    bw = hbm / (ms * 1e-3) / 1e9
    out = {"workload": "blockwise INT8 compressed all-reduce", "n": n, "count": count, "dtype": dtype,
           "block": block, "path": path, "error_feedback": ef, "us": round(ms * 1e3, 2),
           "algbw": round(S / (ms * 1e-3) / 1e9, 2), "launches": launches, "hbm_bytes": hbm,
           "hbm_gbs": round(bw, 1), "hbm_frac": round(bw / hbm_peak(), 4) if hbm > 8 * l2 else None}
    del grads, outs, res
    torch.cuda.empty_cache()
    return out


def sweep(out=sys.stdout, max_total=64 * GiB, graph=False):
    for n in (2, 4, 8, 16, 64):
        for k in range(11):
            S = KiB * 4 ** k
            if n * S > max_total:
                continue
            for algo, order in (("fused", "ring"), ("fused", "rank"), ("ring", "ring"), ("rabenseifner", "ring")):
                iters = 10 if n * S < GiB else 5
                res = time_case(n, S // 4, "f32", algo, order, iters=iters, warmup=3, graph=graph)
                print(json.dumps(res), file=out, flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--algo", default="fused")
    ap.add_argument("--order", default="ring")
    ap.add_argument("--n", type=int, default=16)
    ap.add_argument("--count", type=int, default=8 * MiB)
    ap.add_argument("--dtype", default="f32")
    ap.add_argument("--group-size", type=int, default=0)
    ap.add_argument("--collective", default="allreduce", choices=["allreduce", "reduce_scatter", "allgather"])
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--reps", type=int, default=None)
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--graph", action="store_true", help="replay the timed calls from a CUDA graph")
    ap.add_argument("--bound", action="store_true", help="bind the plan once (ar_bind) and time ar_execute_bound")
    ap.add_argument("--buckets", choices=["fused", "pack"], default=None)
    ap.add_argument("--overlap", action="store_true", help="bucketed sync overlapped with a synthetic backward")
    ap.add_argument("--tokens", type=int, default=4096)
    ap.add_argument("--sm-budget", type=int, default=0)
    ap.add_argument("--kernel", default="auto", choices=["auto", "loads", "bulk"])
    ap.add_argument("--dims", default="0,0,0", help="torus dimensions X,Y[,Z] for --algo torus")
    ap.add_argument("--compressed", choices=["fused", "two"], default=None,
                    help="blockwise INT8 compressed all-reduce (fused pass or compressor + reducer)")
    ap.add_argument("--block", type=int, default=128)
    ap.add_argument("--no-ef", action="store_true", help="compressed all-reduce without error feedback")
    a = ap.parse_args(argv)
    from gradient_sync_gb300 import build

    build.build()
    if a.sweep:
        sweep(graph=a.graph)
        return
    if a.compressed:
        print(json.dumps(time_compressed(a.n, a.count, a.dtype, a.block, a.compressed, not a.no_ef,
                                         a.iters, a.warmup)))
        return
    if a.buckets:
        print(json.dumps(time_buckets(path=a.buckets, iters=a.iters, warmup=min(a.warmup, 3))))
        return
    if a.overlap:
        from gradient_sync_gb300.overlap import time_overlap

        print(json.dumps(time_overlap(n_ranks=a.n, tokens=a.tokens, sm_budget=a.sm_budget, iters=a.iters,
                                      warmup=min(a.warmup, 3), kernel=a.kernel)))
        return
    print(json.dumps(time_case(a.n, a.count, a.dtype, a.algo, a.order, a.group_size, a.iters, a.warmup, a.reps,
                               graph=a.graph, collective=a.collective, sm_budget=a.sm_budget,
                               kernel=a.kernel, torus_dims=tuple(int(v) for v in a.dims.split(",")),
                               bound=a.bound)))


if __name__ == "__main__":
    main()

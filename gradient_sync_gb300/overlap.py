"""Overlap of the bucketed gradient all-reduce with the backward computation.

Scaling ML Systems ("Collective communication", sections on layer-wise overlap
and bucket fusion) and the AI Infra Book (ch. 7, §7.6.1-§7.6.2) describe the
mechanism: backward produces parameter gradients in reverse layer order; a
bucket's all-reduce starts as soon as its last gradient exists, on a
communication stream, while the computation of earlier layers goes on; the
optimizer step waits for both. What the computation does not hide is exposed.

Here the N ranks are virtual: their gradients live in this GPU's memory, and
the "communication" is the library's fused bucket all-reduce. It competes with
the computation for the same SMs and HBM, so `sm_budget` caps the SMs it may
take, as a NCCL channel occupies one SM (primer §4.5).

The synthetic backward emulates one rank's weight- and input-gradient GEMMs of
the 16-layer transformer (bf16, `tokens` tokens per step, cuBLAS through
torch); it writes scratch buffers, so the gradients being reduced are the
caller's and the result is the same with or without overlap.
"""

from __future__ import annotations

import torch

import gradient_sync_gb300 as g

MiB = 1 << 20


class BucketedReducer:
    """DDP-style reducer over N virtual ranks' gradients.

    grads[r][t]: rank r's gradient of parameter t (forward order), all of the
    same dtype. Buckets follow ar_bucket_plan (reverse order, capped). Call
    ready(t) when gradient t has been produced on the current stream, and
    finish() before using the results.
    """

    def __init__(self, grads, counts=None, cap_bytes=25 * MiB, scale=None, comm_stream=None, sm_budget=0,
                 kernel="auto"):
        self.dtype = "bf16" if grads[0][0].dtype == torch.bfloat16 else "f32"
        self.n = len(grads)
        self.table = g.TensorTable(grads, counts)
        counts = self.table.counts
        of, nb = g.ar_bucket_plan(counts, 2 if self.dtype == "bf16" else 4, cap_bytes)
        self.bucket_of = of
        self.buckets = []
        for b in range(nb):
            ts = [t for t in range(len(counts)) if of[t] == b]
            self.buckets.append((min(ts), max(ts) + 1, len(ts)))
        self.scale = 1.0 / self.n if scale is None else scale
        self.comm = comm_stream or torch.cuda.Stream()
        self.comm_handle = int(self.comm.cuda_stream)
        self.sm_budget = sm_budget
        self.kernel = kernel
        self._remaining = [k for _, _, k in self.buckets]

    def launch(self, b):
        lo, hi, _ = self.buckets[b]
        g.ar_bucket_allreduce(self.table, None, lo, hi, self.dtype, self.scale, stream=self.comm_handle,
                              sm_budget=self.sm_budget, kernel=self.kernel)

    def ready(self, t):
        """Gradient t is complete on the current stream."""
        b = self.bucket_of[t]
        self._remaining[b] -= 1
        if self._remaining[b] == 0:
            self.comm.wait_stream(torch.cuda.current_stream())
            self.launch(b)

    def finish(self):
        """Make the current stream wait for every bucket's all-reduce."""
        torch.cuda.current_stream().wait_stream(self.comm)
        self._remaining = [k for _, _, k in self.buckets]

    def sync_all(self):
        """Every bucket, one after another, on the current stream (no overlap)."""
        cur = int(torch.cuda.current_stream().cuda_stream)
        for lo, hi, _ in self.buckets:
            g.ar_bucket_allreduce(self.table, None, lo, hi, self.dtype, self.scale, stream=cur,
                                  sm_budget=self.sm_budget, kernel=self.kernel)


class SyntheticBackward:
    """One rank's backward GEMMs for the transformer's parameters, in reverse
    forward order: for a weight of shape (out, in), dW = dY^T X and dX = dY W
    (2 * 2 * tokens * in * out flop); for a norm, a weighted sum over tokens;
    for the embedding, an index_add of the tokens' rows."""

    def __init__(self, tensors, tokens=4096, hidden=2048):
        dev = "cuda"
        self.tensors = tensors  # (name, count) in forward order
        self.tokens = tokens
        self.work = []
        shapes = {}
        for name, count in tensors:
            if name == "embedding":
                shape = ("embedding", count // hidden, hidden)
            elif name.endswith(("norm1", "norm2")):
                shape = ("norm", count)
            else:
                k = name.rsplit(".", 1)[-1]
                out_f, in_f = {"wq": (hidden, hidden), "wk": (hidden, hidden), "wv": (hidden, hidden),
                               "wo": (hidden, hidden), "w1": (count // hidden, hidden),
                               "w3": (count // hidden, hidden), "w2": (hidden, count // hidden)}[k]
                shape = ("linear", out_f, in_f)
            self.work.append(shape)
            shapes[shape] = None
        bf = torch.bfloat16
        self.buf = {}
        for shape in shapes:
            if shape[0] == "linear":
                _, o, i = shape
                self.buf[shape] = dict(x=torch.randn(tokens, i, device=dev, dtype=bf),
                                       dy=torch.randn(tokens, o, device=dev, dtype=bf),
                                       w=torch.randn(o, i, device=dev, dtype=bf),
                                       dw=torch.empty(o, i, device=dev, dtype=bf),
                                       dx=torch.empty(tokens, i, device=dev, dtype=bf))
            elif shape[0] == "norm":
                n = shape[1]
                self.buf[shape] = dict(x=torch.randn(tokens, n, device=dev, dtype=bf),
                                       dy=torch.randn(tokens, n, device=dev, dtype=bf))
            else:
                _, rows, h = shape
                self.buf[shape] = dict(idx=torch.randint(0, rows, (tokens,), device=dev),
                                       dy=torch.randn(tokens, h, device=dev, dtype=bf),
                                       dw=torch.zeros(rows, h, device=dev, dtype=bf))

    def flops(self):
        total = 0
        for shape in self.work:
            if shape[0] == "linear":
                total += 4 * self.tokens * shape[1] * shape[2]
        return total

    def run(self, on_ready=None):
        for t in reversed(range(len(self.work))):
            shape = self.work[t]
            b = self.buf[shape]
            if shape[0] == "linear":
                torch.matmul(b["dy"].t(), b["x"], out=b["dw"])
                torch.matmul(b["dy"], b["w"], out=b["dx"])
            elif shape[0] == "norm":
                (b["x"] * b["dy"]).sum(0)
            else:
                b["dw"].index_add_(0, b["idx"], b["dy"])
            if on_ready is not None:
                on_ready(t)


def critical_path(ready, durations, compute_end):
    """End of a step whose buckets' collectives run one after another on one
    stream: bucket b starts at max(its readiness, the previous bucket's end);
    the step ends when both the computation and the last collective have."""
    end = 0.0
    for r, d in zip(ready, durations):
        end = max(r, end) + d
    return max(compute_end, end)


def _time(fn, stream, iters):
    times = []
    for _ in range(iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    times.sort()
    return times[len(times) // 2]


def time_overlap(n_ranks=8, tokens=4096, sm_budget=0, iters=5, warmup=2, layers=16, kernel="auto"):
    """Milliseconds of: the backward alone, the gradient sync alone, the two in
    sequence, and overlapped; plus the exposed communication and what the
    critical-path model predicts from the measured bucket readiness and
    durations."""
    import workloads

    tensors = workloads.transformer_tensors(layers=layers)
    counts = [c for _, c in tensors]
    grads = [[torch.randn(c, device="cuda").to(torch.bfloat16) for c in counts] for _ in range(n_ranks)]
    red = BucketedReducer(grads, counts, sm_budget=sm_budget, kernel=kernel)
    bwd = SyntheticBackward(tensors, tokens=tokens)
    main = torch.cuda.current_stream()

    def overlapped():
        bwd.run(red.ready)
        red.finish()

    def sequential():
        bwd.run()
        red.sync_all()

    for _ in range(warmup):
        overlapped()
        sequential()
    torch.cuda.synchronize()
    t_compute = _time(lambda: bwd.run(), main, iters)
    t_comm = _time(red.sync_all, main, iters)
    t_seq = _time(sequential, main, iters)
    t_ovl = _time(overlapped, main, iters)
    # readiness of each bucket inside the backward, and each bucket's duration alone
    marks = {}
    start = torch.cuda.Event(enable_timing=True)
    start.record(main)

    def mark(t):
        b = red.bucket_of[t]
        if t == red.buckets[b][0]:  # the lowest id is produced last
            e = torch.cuda.Event(enable_timing=True)
            e.record(main)
            marks[b] = e

    bwd.run(mark)
    end = torch.cuda.Event(enable_timing=True)
    end.record(main)
    end.synchronize()
    ready = [start.elapsed_time(marks[b]) for b in range(len(red.buckets))]
    durations = []
    handle = int(main.cuda_stream)
    for lo, hi, _ in red.buckets:
        durations.append(_time(lambda: g.ar_bucket_allreduce(red.table, None, lo, hi, red.dtype, red.scale,
                                                             stream=handle, sm_budget=sm_budget,
                                                             kernel=kernel), main, 3))
    predicted = critical_path(ready, durations, start.elapsed_time(end))
    del grads
    torch.cuda.empty_cache()
    return {"workload": f"{layers}-layer transformer backward, {tokens} tokens, bucketed sync of {n_ranks} ranks",
            "n_ranks": n_ranks, "tokens": tokens, "sm_budget": sm_budget, "kernel": kernel,
            "buckets": len(red.buckets),
            "backward_tflop": round(bwd.flops() / 1e12, 3),
            "ms_compute": round(t_compute, 3), "ms_comm": round(t_comm, 3), "ms_sequential": round(t_seq, 3),
            "ms_overlapped": round(t_ovl, 3), "ms_exposed": round(t_ovl - t_compute, 3),
            "hidden_fraction": round(1 - (t_ovl - t_compute) / t_comm, 3) if t_comm > 0 else None,
            "ms_model_no_contention": round(predicted, 3)}

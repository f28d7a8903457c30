"""GB300 gradient all-reduce over N virtual ranks held in one GPU's memory.

A thin Python binding of libar_gb300.so: the functions below carry the C
ABI's names (include/ar.h) and only marshal arguments -- torch tensors or raw
integer device pointers in, status codes out as exceptions. Every step of the
all-reduce runs in the library's CUDA kernels; there is no Python or CPU
fallback, and importing a function whose library is missing raises.
"""

from __future__ import annotations

import ctypes

from . import _lib

# ---- enums of include/ar.h
AR_OK, AR_EINVAL, AR_EUNSUPPORTED, AR_ENOMEM, AR_ECUDA, AR_ETIMEOUT = range(6)
AR_F32, AR_BF16 = 0, 1
AR_RING, AR_RABENSEIFNER, AR_HIER, AR_FUSED, AR_AUTO = 0, 1, 2, 3, 4
AR_ORDER_RING, AR_ORDER_RANK, AR_ORDER_TREE, AR_ORDER_HIER = 0, 1, 2, 3
AR_ALLREDUCE, AR_REDUCE_SCATTER, AR_ALLGATHER = 0, 1, 2
AR_KERNEL_AUTO, AR_KERNEL_LOADS, AR_KERNEL_BULK = 0, 1, 2
AR_MAX_RANKS = 64
AR_MAX_BUCKET_TENSORS = 32

AR_RECDOUBLING, AR_DBTREE, AR_TORUS = 5, 6, 7
ALGOS = {"ring": AR_RING, "rabenseifner": AR_RABENSEIFNER, "hier": AR_HIER, "fused": AR_FUSED, "auto": AR_AUTO,
         "recdoubling": AR_RECDOUBLING, "dbtree": AR_DBTREE, "torus": AR_TORUS}
ALGO_NAMES = {v: k for k, v in ALGOS.items()}
AR_DEVICE_ALPHA_S, AR_DEVICE_BW, AR_DEVICE_CTA_STEP_S, AR_DEVICE_CTA_STEP_MEM_S = 1.5e-6, 6.0e12, 0.28e-6, 0.75e-6
ORDERS = {"ring": AR_ORDER_RING, "rank": AR_ORDER_RANK, "tree": AR_ORDER_TREE, "hier": AR_ORDER_HIER}
DTYPES = {"f32": AR_F32, "bf16": AR_BF16}
COLLECTIVES = {"allreduce": AR_ALLREDUCE, "reduce_scatter": AR_REDUCE_SCATTER, "allgather": AR_ALLGATHER}
KERNELS = {"auto": AR_KERNEL_AUTO, "loads": AR_KERNEL_LOADS, "bulk": AR_KERNEL_BULK}
KERNEL_NAMES = {v: k for k, v in KERNELS.items()}


class ArError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {ar_status_string(status)}" if what else ar_status_string(status))


def _check(status: int, what: str):
    if status != AR_OK:
        raise ArError(status, what)


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _ptrs(xs):
    return _lib.ptr_array([_ptr(x) for x in xs])


def _stream(stream) -> int:
    if stream is None:
        import torch

        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


# ---------------------------------------------------------------- plans


class Plan:
    """An ar_plan_t*; destroyed with the object."""

    def __init__(self, handle: int, desc: dict):
        self.handle = handle
        self.desc = desc

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h:
            try:
                _lib.load().ar_plan_destroy(h)
            except Exception:
                pass

    @property
    def stats(self) -> dict:
        return ar_plan_stats(self)


def ar_plan(n_ranks: int, count: int, dtype="f32", algo="fused", group_size: int = 0, order="ring",
            scale: float = 1.0, collective="allreduce", sm_budget: int = 0, kernel="auto",
            torus_dims=(0, 0, 0)) -> Plan:
    """Validate the descriptor and build the schedule (host only)."""
    dims = (list(torus_dims) + [0, 0, 0])[:3]
    d = _lib.ArDesc(int(n_ranks), int(count), DTYPES.get(dtype, dtype), ALGOS.get(algo, algo),
                    int(group_size), ORDERS.get(order, order), float(scale),
                    COLLECTIVES.get(collective, collective), int(sm_budget), KERNELS.get(kernel, kernel),
                    (_lib.c_int * 3)(*[int(v) for v in dims]))
    h = _lib.c_void_p()
    _check(_lib.load().ar_plan(d, h), "ar_plan")
    return Plan(h.value, dict(n_ranks=n_ranks, count=count, dtype=dtype, algo=algo, group_size=group_size,
                              order=order, scale=scale, collective=collective, sm_budget=sm_budget,
                              kernel=kernel, torus_dims=tuple(dims)))


def ar_plan_desc(plan: Plan) -> dict:
    """The plan's descriptor as the library holds it (AR_AUTO resolved)."""
    d = _lib.ArDesc()
    _check(_lib.load().ar_plan_desc(plan.handle, d), "ar_plan_desc")
    return {"n_ranks": d.n_ranks, "count": d.count, "dtype": d.dtype, "algo": ALGO_NAMES.get(d.algo, d.algo),
            "group_size": d.group_size, "order": d.order, "scale": d.scale, "collective": d.collective,
            "sm_budget": d.sm_budget, "kernel": KERNEL_NAMES.get(d.kernel, d.kernel),
            "torus_dims": tuple(d.torus_dims)}


def fabric(alpha, bw_local, bw_net=None, ranks_per_server=0, in_network=False, shared_memory=False):
    """An ar_fabric: seconds per round, bytes/s inside and between servers."""
    return _lib.ArFabric(float(alpha), float(bw_local), float(bw_net if bw_net is not None else bw_local),
                         int(ranks_per_server), int(bool(in_network)), int(bool(shared_memory)))


def ar_plan_predict(plan: Plan, fab) -> float:
    """Predicted seconds of one ar_execute of the plan on a fabric (round model)."""
    t = ctypes.c_double()
    _check(_lib.load().ar_plan_predict(plan.handle, fab, t), "ar_plan_predict")
    return t.value


def ar_select(n_ranks, count, fab, dtype="f32", order="ring", scale=1.0, collective="allreduce"):
    """(algorithm name, group size, predicted seconds) of the fastest algorithm on a fabric."""
    d = _lib.ArDesc(int(n_ranks), int(count), DTYPES.get(dtype, dtype), AR_FUSED, 0, ORDERS.get(order, order),
                    float(scale), COLLECTIVES.get(collective, collective), 0)
    a, gs, t = _lib.c_int(), _lib.c_int(), ctypes.c_double()
    _check(_lib.load().ar_select(d, fab, a, gs, t), "ar_select")
    return ALGO_NAMES[a.value], gs.value, t.value


def ar_plan_stats(plan: Plan) -> dict:
    s = _lib.ArStats()
    _check(_lib.load().ar_plan_stats(plan.handle, s), "ar_plan_stats")
    return {f: getattr(s, f) for f, _ in _lib.ArStats._fields_}


def ar_plan_transfers(plan: Plan, step: int):
    """(op, [(src, dst, first, end), ...]) of one step of a step plan."""
    lib = _lib.load()
    op, n = _lib.c_int(), _lib.c_int()
    _check(lib.ar_plan_transfers(plan.handle, step, op, n, None, 0), "ar_plan_transfers")
    buf = (ctypes.c_int64 * max(1, 4 * n.value))()
    _check(lib.ar_plan_transfers(plan.handle, step, op, n, buf, n.value), "ar_plan_transfers")
    rows = [tuple(buf[4 * i: 4 * i + 4]) for i in range(n.value)]
    return ("reduce" if op.value == 0 else "copy"), rows


def ar_execute(plan: Plan, bufs, outs=None, workspace=None, stream=None):
    """Enqueue the all-reduce of the N device buffers ``bufs`` (in place unless ``outs``)."""
    o = _ptrs(outs) if outs is not None else None
    _check(_lib.load().ar_execute(plan.handle, _ptrs(bufs), o, _ptr(workspace), _stream(stream)),
           "ar_execute")


def ar_execute_host(plan: Plan, host_in, host_out, dev_bufs, workspace=None, stream=None):
    """All-reduce host buffers through device staging buffers; returns when done."""
    _check(_lib.load().ar_execute_host(plan.handle, _ptrs(host_in), _ptrs(host_out), _ptrs(dev_bufs),
                                       _ptr(workspace), _stream(stream)), "ar_execute_host")


AR_STATIC_WORKSPACE_BYTES = 64 << 20


def ar_execute_noalloc(plan: Plan, bufs, outs=None, stream=None):
    """ar_execute for callers that cannot allocate device memory: the workspace
    comes from a fixed array inside the library (AR_STATIC_WORKSPACE_BYTES).
    Calls share that array, so calls that overlap on the GPU race."""
    o = _ptrs(outs) if outs is not None else None
    _check(_lib.load().ar_execute_noalloc(plan.handle, _ptrs(bufs), o, _stream(stream)), "ar_execute_noalloc")


class Bound:
    """An ar_bound_t*: a plan bound to its buffers (a persistent collective).
    Keeps the buffers alive; destroyed with the object."""

    def __init__(self, handle: int, keep):
        self.handle = handle
        self._keep = keep

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h:
            try:
                _lib.load().ar_bound_destroy(h)
            except Exception:
                pass

    def execute(self, stream=None):
        ar_execute_bound(self, stream)


def ar_bind(plan: Plan, bufs, outs=None, workspace=None) -> Bound:
    """Validate the buffers once and record the plan's launches (see include/ar.h)."""
    o = _ptrs(outs) if outs is not None else None
    h = _lib.c_void_p()
    _check(_lib.load().ar_bind(plan.handle, _ptrs(bufs), o, _ptr(workspace), h), "ar_bind")
    return Bound(h.value, (list(bufs), None if outs is None else list(outs), workspace))


def ar_execute_bound(bound: Bound, stream=None):
    """Replay a bound all-reduce on ``stream`` (an int handle skips the torch lookup)."""
    _check(_lib.load().ar_execute_bound(bound.handle, _stream(stream)), "ar_execute_bound")


# ---------------------------------------------------------------- buckets


def _counts(counts):
    return (_lib.c_size_t * len(counts))(*[int(c) for c in counts])


def ar_bucket_plan(counts, elem_bytes: int, cap_bytes: int):
    """Returns (bucket_of_tensor list, n_buckets)."""
    n = len(counts)
    out = (_lib.c_int * n)()
    nb = _lib.c_int()
    _check(_lib.load().ar_bucket_plan(_counts(counts), n, int(elem_bytes), int(cap_bytes), out, nb),
           "ar_bucket_plan")
    return list(out), nb.value


class TensorTable:
    """The [rank][tensor] pointer table and element counts of the bucket calls,
    marshalled once. Pass it in place of the nested tensor list when the same
    gradients are synchronised again and again (as DDP does every step): the
    per-call cost is then independent of the number of tensors."""

    def __init__(self, tensors, counts=None):
        self.n_ranks = len(tensors)
        self.n_tensors = len(tensors[0])
        if counts is None:
            counts = [t.numel() for t in tensors[0]]
        self.counts = list(counts)
        self.c_ptrs = _lib.ptr_array([_ptr(t) for row in tensors for t in row])
        self.c_counts = _counts(self.counts)


def _marshal(tensors, counts):
    if isinstance(tensors, TensorTable):
        return tensors.n_ranks, tensors.c_ptrs, tensors.c_counts, tensors.n_tensors
    return len(tensors), _lib.ptr_array([_ptr(t) for row in tensors for t in row]), _counts(counts), len(counts)


def _buckets(bucket):
    """Bucket buffers: a list of tensors/pointers, or an already marshalled pointer array."""
    return bucket if isinstance(bucket, ctypes.Array) else _ptrs(bucket)


def ar_bucket_pack(tensors, counts, t_begin: int, t_end: int, in_dtype, bucket, stream=None):
    n, ptrs, cnt, nt = _marshal(tensors, counts)
    _check(_lib.load().ar_bucket_pack(n, ptrs, cnt, nt, t_begin, t_end, DTYPES.get(in_dtype, in_dtype),
                                      _buckets(bucket), _stream(stream)), "ar_bucket_pack")


def ar_bucket_unpack(bucket, scale: float, out_dtype, tensors, counts, t_begin: int, t_end: int,
                     stream=None):
    n, ptrs, cnt, nt = _marshal(tensors, counts)
    _check(_lib.load().ar_bucket_unpack(n, _buckets(bucket), float(scale), DTYPES.get(out_dtype, out_dtype),
                                        ptrs, cnt, nt, t_begin, t_end, _stream(stream)), "ar_bucket_unpack")


def ar_bucket_allreduce(tensors, counts, t_begin: int, t_end: int, dtype, scale: float, stream=None,
                        sm_budget: int = 0, kernel="auto"):
    n, ptrs, cnt, nt = _marshal(tensors, counts)
    _check(_lib.load().ar_bucket_allreduce(n, ptrs, cnt, nt, t_begin, t_end, DTYPES.get(dtype, dtype),
                                           float(scale), int(sm_budget), KERNELS.get(kernel, kernel),
                                           _stream(stream)), "ar_bucket_allreduce")


# ---------------------------------------------------------------- compression

AR_COMPRESS_MIN_BLOCK, AR_COMPRESS_MAX_BLOCK = 16, 1024


def ar_compress_sizes(count: int, block: int):
    """(number of scales, message bytes) of one rank's compressed message."""
    ns, mb = _lib.c_size_t(), _lib.c_size_t()
    _check(_lib.load().ar_compress_sizes(int(count), int(block), ns, mb), "ar_compress_sizes")
    return ns.value, mb.value


def ar_compress(grads, codes, scales, block: int, dtype="f32", residuals=None, count=None, stream=None):
    """Blockwise INT8 compression of every rank's gradient (with error feedback
    when ``residuals`` is given: read as e, overwritten with the new residual)."""
    n = len(grads)
    count = grads[0].numel() if count is None else count
    res = _ptrs(residuals) if residuals is not None else None
    _check(_lib.load().ar_compress(n, int(count), int(block), DTYPES.get(dtype, dtype), _ptrs(grads), res,
                                   _ptrs(codes), _ptrs(scales), _stream(stream)), "ar_compress")


def ar_compressed_reduce(codes, scales, outs, block: int, scale: float = 1.0, out_dtype="f32", count=None,
                         stream=None):
    """Sum the ranks' compressed messages in rank order into every ``outs[r]``."""
    n = len(codes)
    count = codes[0].numel() if count is None else count
    _check(_lib.load().ar_compressed_reduce(n, int(count), int(block), _ptrs(codes), _ptrs(scales), float(scale),
                                            DTYPES.get(out_dtype, out_dtype), _ptrs(outs), _stream(stream)),
           "ar_compressed_reduce")


def ar_compressed_allreduce(grads, block: int, dtype="f32", residuals=None, scale: float = 1.0, outs=None,
                            count=None, stream=None):
    """Compression and reduction in one pass (in place unless ``outs``)."""
    n = len(grads)
    count = grads[0].numel() if count is None else count
    res = _ptrs(residuals) if residuals is not None else None
    o = _ptrs(outs) if outs is not None else None
    _check(_lib.load().ar_compressed_allreduce(n, int(count), int(block), DTYPES.get(dtype, dtype), _ptrs(grads),
                                               res, float(scale), o, _stream(stream)), "ar_compressed_allreduce")


# ---------------------------------------------------------------- status


def ar_device_status(clear: bool = True) -> int:
    return _lib.load().ar_device_status(1 if clear else 0)


def ar_plan_query(plan: Plan) -> int:
    """The plan's sticky asynchronous status (AR_OK or AR_ETIMEOUT), read
    without synchronising; see include/ar.h."""
    return _lib.load().ar_plan_query(plan.handle)


def ar_selftest_wait_timeout(polls: int = 1000, stream=None):
    """Run the bounded-wait self-test kernel (see include/ar.h)."""
    _check(_lib.load().ar_selftest_wait_timeout(int(polls), _stream(stream)), "ar_selftest_wait_timeout")


def ar_selftest_scale_quotient() -> int:
    """Mismatches of the division-free block scale against the IEEE division
    over every non-negative float (see include/ar.h)."""
    n = ctypes.c_ulonglong(0)
    _check(_lib.load().ar_selftest_scale_quotient(ctypes.byref(n)), "ar_selftest_scale_quotient")
    return n.value


def ar_status_string(status: int) -> str:
    return _lib.load().ar_status_string(int(status)).decode()


def ar_version() -> int:
    return _lib.load().ar_version()


# ---------------------------------------------------------------- convenience


def workspace_for(plan: Plan, device=None):
    """A torch byte tensor of the plan's workspace size (None when it needs none)."""
    nbytes = plan.stats["workspace_bytes"]
    if nbytes == 0:
        return None
    import torch

    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")

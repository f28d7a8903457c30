"""Out-of-bounds checks without a sanitizer: red zones around every buffer.

Every device buffer a call touches is carved out of one larger allocation,
with a guard region of 0xFF bytes before and after it (0xFF bytes are a NaN
in fp32 and in bf16). After the call:
- every guard byte must still be 0xFF: a write outside a buffer changes one;
- every result must equal the oracle's bit for bit: a read outside a buffer
  brings a NaN into a sum or a maximum and shows as a mismatch.
The element counts are ragged (no multiple of any vector, tile or chunk), so
every kernel's tail path runs next to a guard region. Buffers are carved at
16-byte alignment that is not 32-byte alignment, and at 256-byte alignment,
so both the 16-byte and the 32-byte vector paths run."""

import numpy as np
import pytest
import torch

import workloads
from _gpu import assert_bits_equal, expected, to_host, widened
from oracle import compress as C
from oracle import numerics, schedules
from oracle.chunks import chunk_bounds

pytestmark = pytest.mark.gpu

RZ = 4096  # guard bytes on each side of every buffer
TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "i8": torch.int8, "u8": torch.uint8}
SIZE = {"f32": 4, "bf16": 2, "i8": 1, "u8": 1}


@pytest.fixture(scope="module")
def g():
    from gradient_sync_gb300 import build

    build.build()
    import gradient_sync_gb300 as g

    return g


class Arena:
    """Buffers of the given (elements, dtype) carved from one allocation, each
    between two guard regions. align16: every buffer starts 16 bytes past a
    multiple of 32; else on a multiple of 256."""

    def __init__(self, shapes, align16: bool):
        self.spans, pos = [], RZ
        for n, dt in shapes:
            pos = (pos + 255) // 256 * 256 + (16 if align16 else 0)
            nbytes = max(n, 1) * SIZE[dt]
            self.spans.append((pos, nbytes, dt, n))
            pos += nbytes + RZ
        self.mem = torch.full((pos + 256,), 0xFF, dtype=torch.uint8, device="cuda")
        shift = (-self.mem.data_ptr()) % 256  # the allocation's base on a 256-byte boundary
        self.spans = [(o + shift, nb, dt, n) for o, nb, dt, n in self.spans]
        self.views = [self.mem[o:o + nb].view(TORCH[dt])[:n] for o, nb, dt, n in self.spans]

    def __getitem__(self, i):
        return self.views[i]

    def check_guards(self, what=""):
        torch.cuda.synchronize()
        host = self.mem.cpu().numpy()
        inside = np.zeros(host.size, bool)
        for o, nb, _, _ in self.spans:
            inside[o:o + nb] = True
        bad = np.nonzero((host != 0xFF) & ~inside)[0]
        assert bad.size == 0, f"{what}: {bad.size} guard bytes written, first at byte offsets {bad[:8].tolist()}"


def _fill(view, arr, dtype):
    host = np.ascontiguousarray(arr)
    src = torch.from_numpy(host.view(np.int16) if dtype == "bf16" else host).cuda()
    view.copy_(src.view(view.dtype))


ALLREDUCE = [("ring", "ring", 0, None), ("rabenseifner", "ring", 0, None), ("hier", "ring", 4, None),
             ("recdoubling", "ring", 0, None), ("dbtree", "ring", 0, None), ("torus", "ring", 0, (2, 4)),
             ("fused", "ring", 0, None), ("fused", "rank", 0, None), ("fused", "tree", 0, None),
             ("fused", "hier", 4, None)]


@pytest.mark.parametrize("align16", [True, False])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo,order,G,dims", ALLREDUCE)
def test_allreduce_stays_inside_its_buffers(g, algo, order, G, dims, dtype, align16):
    N = 8
    # the fused pass: register pipeline, bulk copies, and held to a few SMs
    kernels = [("loads", 0), ("bulk", 0), ("loads", 7)] if algo == "fused" else [("auto", 0)]
    for L in (4099, 37):
        x = workloads.all_ranks(workloads.small_spec(N, L, dtype, "normal", seed=L + 11 * N))
        scale = 0.5 if L % 2 else 1.0
        want = expected(algo, order, x, dtype, group_size=G, scale=scale, torus_dims=dims)
        for kernel, sm_budget in kernels:
            for out_of_place in (False, True):
                plan = g.ar_plan(N, L, dtype, algo, group_size=G, order=order, scale=scale, kernel=kernel,
                                 torus_dims=dims or (0, 0, 0), sm_budget=sm_budget)
                ws_bytes = plan.stats["workspace_bytes"]
                shapes = [(L, dtype)] * N + ([(L, dtype)] * N if out_of_place else [])
                shapes += [(ws_bytes, "u8")] if ws_bytes else []
                a = Arena(shapes, align16)
                for r in range(N):
                    _fill(a[r], x[r], dtype)
                outs = [a[N + r] for r in range(N)] if out_of_place else None
                ws = a[len(shapes) - 1] if ws_bytes else None
                g.ar_execute(plan, [a[r] for r in range(N)], outs=outs, workspace=ws)
                what = (f"{algo}/{order} {kernel} sm_budget={sm_budget} L={L} "
                        f"{'out of place' if out_of_place else 'in place'}")
                a.check_guards(what)
                for r in range(N):
                    got = to_host(outs[r] if out_of_place else a[r], dtype)
                    assert_bits_equal(got, want, f"{what} rank {r}")


@pytest.mark.parametrize("align16", [True, False])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo,coll,kernel,sm_budget,out_of_place",
                         [("ring", "reduce_scatter", "auto", 0, False), ("fused", "reduce_scatter", "auto", 0, False),
                          ("fused", "reduce_scatter", "loads", 5, False), ("ring", "allgather", "auto", 0, False),
                          ("ring", "allgather", "auto", 0, True), ("fused", "allgather", "loads", 0, False),
                          ("fused", "allgather", "bulk", 0, False), ("fused", "allgather", "bulk", 0, True)])
@pytest.mark.parametrize("L", [20011, 20010])
def test_collectives_stay_inside_their_buffers(g, algo, coll, kernel, sm_budget, out_of_place, dtype, align16, L):
    """Out of place the ring all-gather's first step also writes each sent
    chunk to the sender's output; held to a few SMs the reduce-scatter runs
    the kernel that loads ahead across tiles; with even chunk bounds (L =
    20010) bf16 copy steps move fp32 pairs."""
    N = 5
    x = workloads.all_ranks(workloads.small_spec(N, L, dtype, "uniform", seed=3 + L))
    xf = widened(x, dtype)
    b = chunk_bounds(L, N)
    if coll == "allgather":
        want, _ = schedules.ring_allgather(x)
    elif algo == "ring":
        finish = schedules.finish_bf16(1.0) if dtype == "bf16" else schedules.finish_scale(1.0)
        out, _ = schedules.ring_reduce_scatter(xf, finish=finish)
        want = [numerics.f32_to_bf16_rne(out[r]) if dtype == "bf16" else out[r] for r in range(N)]
    else:
        s = numerics.fused_sum(xf, "ring_rs")
        want = [numerics.f32_to_bf16_rne(s) if dtype == "bf16" else s] * N
    plan = g.ar_plan(N, L, dtype, algo, collective=coll, kernel=kernel, sm_budget=sm_budget)
    ws_bytes = plan.stats["workspace_bytes"]
    shapes = [(L, dtype)] * N + ([(L, dtype)] * N if out_of_place else [])
    a = Arena(shapes + ([(ws_bytes, "u8")] if ws_bytes else []), align16)
    for r in range(N):
        _fill(a[r], x[r], dtype)
    outs = [a[N + r] for r in range(N)] if out_of_place else None
    g.ar_execute(plan, [a[r] for r in range(N)], outs=outs, workspace=a[len(shapes)] if ws_bytes else None)
    a.check_guards(f"{algo} {coll} {kernel} sm_budget={sm_budget} out_of_place={out_of_place}")
    for r in range(N):
        got = to_host(outs[r] if out_of_place else a[r], dtype)
        if out_of_place:
            np.testing.assert_array_equal(to_host(a[r], dtype), x[r])
        if coll == "allgather":
            assert_bits_equal(got, want[r], f"rank {r}")
        else:
            seg = slice(b[r], b[r + 1])
            assert_bits_equal(got[seg], want[r][seg], f"rank {r}")


@pytest.mark.parametrize("align16", [True, False])
def test_bucket_calls_stay_inside_their_buffers(g, align16):
    from oracle import buckets as ob

    N = 6
    counts = [5, 1000, 37, 4099, 9, 2051, 3]
    scale = 1.0 / N
    rng = np.random.default_rng(17)
    grads = [[numerics.f32_to_bf16_rne((rng.standard_normal(c) * 1e-3).astype(np.float32)) for c in counts]
             for _ in range(N)]
    nt = len(counts)
    for b in ob.bucket_plan(counts, 2, 2 * 4200):
        lo, hi = min(b), max(b) + 1
        Lb = sum(counts[t] for t in b)
        want = ob.sync_bucket(grads, b, counts, scale)
        for path in ("pack", "fused_loads", "fused_bulk", "fused_loads_budget"):
            shapes = [(counts[t], "bf16") for r in range(N) for t in range(nt)]
            shapes += [(Lb, "f32")] * N if path == "pack" else []
            a = Arena(shapes, align16)
            tensors = [[a[r * nt + t] for t in range(nt)] for r in range(N)]
            for r in range(N):
                for t in range(nt):
                    _fill(tensors[r][t], grads[r][t], "bf16")
            if path == "pack":
                bucket = [a[N * nt + r] for r in range(N)]
                g.ar_bucket_pack(tensors, counts, lo, hi, "bf16", bucket)
                g.ar_execute(g.ar_plan(N, Lb, "f32", "ring"), bucket)
                g.ar_bucket_unpack(bucket, scale, "bf16", tensors, counts, lo, hi)
            else:  # the budgeted launch runs the kernel that loads ahead across tiles
                g.ar_bucket_allreduce(tensors, counts, lo, hi, "bf16", scale, kernel=path.split("_")[1],
                                      sm_budget=5 if path.endswith("budget") else 0)
            a.check_guards(f"bucket {lo}..{hi} {path}")
            for r in range(N):
                for t in range(nt):
                    want_t = want[(t, 0)][r] if t in b else grads[r][t]
                    assert_bits_equal(to_host(tensors[r][t], "bf16"), want_t, f"{path} t={t} r={r}")


@pytest.mark.parametrize("align16", [True, False])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ef", [False, True])
@pytest.mark.parametrize("block", [64, 512, 1024])
def test_compression_stays_inside_its_buffers(g, dtype, ef, block, align16):
    """Blocks of 512 and 1024 run the kernels for blocks that span warps."""
    N = 5
    for L in (4103, 23):
        rng = np.random.default_rng(L + 7)
        xf = (rng.standard_normal((N, L)) * 1e-2).astype(np.float32)
        x = numerics.f32_to_bf16_rne(xf) if dtype == "bf16" else xf
        e = (rng.standard_normal((N, L)) * 1e-5).astype(np.float32) if ef else None
        nb, _ = g.ar_compress_sizes(L, block)
        # compressor and reducer: gradients, residuals, codes, scales, outputs
        shapes = [(L, dtype)] * N + ([(L, "f32")] * N if ef else []) + [(L, "i8")] * N + [(nb, "f32")] * N
        shapes += [(L, dtype)] * N
        a = Arena(shapes, align16)
        k = 0
        grads = [a[k + r] for r in range(N)]
        k += N
        res = None
        if ef:
            res = [a[k + r] for r in range(N)]
            k += N
        codes = [a[k + r] for r in range(N)]
        scales = [a[k + N + r] for r in range(N)]
        outs = [a[k + 2 * N + r] for r in range(N)]
        for r in range(N):
            _fill(grads[r], x[r], dtype)
            if ef:
                _fill(res[r], e[r], "f32")
        g.ar_compress(grads, codes, scales, block, dtype=dtype, residuals=res, count=L)
        g.ar_compressed_reduce(codes, scales, outs, block, scale=0.25, out_dtype=dtype, count=L)
        a.check_guards(f"compress + reduce L={L}")
        qs, ss, es = [], [], []
        for r in range(N):
            q, s, en = C.compress_rank(widened(x, dtype)[r], None if e is None else e[r], block)
            qs.append(q)
            ss.append(s)
            es.append(en)
            np.testing.assert_array_equal(codes[r].cpu().numpy(), q, err_msg=f"codes rank {r}")
            assert_bits_equal(scales[r].cpu().numpy(), s, f"scales rank {r}")
            if ef:
                assert_bits_equal(to_host(res[r], "f32"), en, f"residual rank {r}")
        want = C.dequant_allreduce(qs, ss, block, scale=0.25, out_dtype=dtype)
        for r in range(N):
            assert_bits_equal(to_host(outs[r], dtype), want, f"reduced rank {r}")
        # the fused pass, in place
        b2 = Arena([(L, dtype)] * N + ([(L, "f32")] * N if ef else []), align16)
        for r in range(N):
            _fill(b2[r], x[r], dtype)
            if ef:
                _fill(b2[N + r], e[r], "f32")
        g.ar_compressed_allreduce([b2[r] for r in range(N)], block, dtype=dtype,
                                  residuals=[b2[N + r] for r in range(N)] if ef else None, scale=0.25, count=L)
        b2.check_guards(f"fused compressed L={L}")
        want_f, want_e, _, _ = C.compressed_allreduce(widened(x, dtype), e, block, scale=0.25, out_dtype=dtype)
        for r in range(N):
            assert_bits_equal(to_host(b2[r], dtype), want_f, f"fused rank {r}")
            if ef:
                assert_bits_equal(to_host(b2[N + r], "f32"), want_e[r], f"fused residual rank {r}")

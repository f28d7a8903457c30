"""GPU parity of the blockwise INT8 compression with error feedback and the
compressed all-reduce against the oracle, bit for bit, through the C ABI.

The oracle computes every step in fp32 in the page's order, as the kernels do,
so codes, scales, residuals and sums must match exactly. The reducer is fed the
oracle's own messages, so its check does not depend on the GPU compressor."""

import numpy as np
import pytest
import torch

import workloads
from _gpu import assert_bits_equal, to_device, to_host, widened
from oracle import compress as C
from oracle import numerics

pytestmark = pytest.mark.gpu

F32 = np.float32
BLOCKS = [16, 32, 64, 128, 256, 512, 1024]


@pytest.fixture(scope="module")
def g():
    from gradient_sync_gb300 import build

    build.build()
    import gradient_sync_gb300 as g

    assert torch.cuda.is_available()
    return g


def _inputs(N, L, dtype, seed, dist="normal"):
    spec = workloads.small_spec(N, L, dtype, dist, seed=seed)
    x = workloads.all_ranks(spec)
    e = np.stack([workloads.residual_buffer(spec, r) for r in range(N)]) if N else None
    return x, e


def _heavy_tailed(N, L, seed):
    """Normal gradients with a heavy tail, whole zero blocks and values so
    small that a block's scale underflows."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, L)) * 1e-3
    hot = rng.random((N, L)) < 0.005
    x[hot] *= rng.uniform(50, 500, hot.sum())
    if L >= 64:
        x[:, 16:32] = 0.0
        x[:, 32:48] = rng.choice([1e-44, -3e-45, 0.0], (N, 16))
    return x.astype(F32)


def _dev(arrs, dtype):
    return [to_device(a, dtype) for a in arrs]


def _oracle_messages(xf, e, block):
    qs, ss, es = [], [], []
    for r in range(xf.shape[0]):
        q, s, en = C.compress_rank(xf[r], None if e is None else e[r], block)
        qs.append(q)
        ss.append(s)
        es.append(en)
    return qs, ss, es


def _compress_on_gpu(g, x, e, dtype, block):
    N, L = x.shape
    grads = _dev(x, dtype)
    res = _dev(e, "f32") if e is not None else None
    nb, _ = g.ar_compress_sizes(L, block)
    codes = [torch.full((max(L, 1),), 77, dtype=torch.int8, device="cuda") for _ in range(N)]
    scales = [torch.full((max(nb, 1),), -1.0, dtype=torch.float32, device="cuda") for _ in range(N)]
    g.ar_compress(grads, codes, scales, block, dtype=dtype, residuals=res, count=L)
    torch.cuda.synchronize()
    for r in range(N):  # the gradients are read only
        np.testing.assert_array_equal(to_host(grads[r], dtype), x[r])
    return ([c[:L].cpu().numpy() for c in codes], [s[:nb].cpu().numpy() for s in scales],
            None if res is None else [to_host(t, "f32") for t in res])


def _check_messages(got, want, ef):
    gq, gs, ge = got
    wq, ws, we = want
    for r in range(len(wq)):
        np.testing.assert_array_equal(gq[r], wq[r], err_msg=f"codes rank {r}")
        assert_bits_equal(gs[r], ws[r], f"scales rank {r}")
        if ef:
            assert_bits_equal(ge[r], we[r], f"residual rank {r}")


SIZES = [1, 7, 16, 100, 1000, 4103, 20011, (1 << 17) + 5]


@pytest.mark.parametrize("ef", [False, True])
@pytest.mark.parametrize("block", BLOCKS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_compress_matches_oracle(g, dtype, block, ef):
    for i, L in enumerate(SIZES):
        N = (1, 2, 3, 5)[i % 4]
        x, e = _inputs(N, L, dtype, seed=block + 7 * i)
        e = e if ef else None
        got = _compress_on_gpu(g, x, e, dtype, block)
        _check_messages(got, _oracle_messages(widened(x, dtype), e, block), ef)


@pytest.mark.parametrize("block", [16, 64, 128, 1024])
def test_compress_heavy_tails_zero_and_underflowing_blocks(g, block):
    x = _heavy_tailed(4, 5003, block)
    e = (np.random.default_rng(block).standard_normal(x.shape) * 1e-5).astype(F32)
    for ee in (None, e):
        got = _compress_on_gpu(g, x, ee, "f32", block)
        _check_messages(got, _oracle_messages(x, ee, block), ee is not None)
    gq, gs, _ = _compress_on_gpu(g, x, None, "f32", block)
    if block == 16:  # the zero block and the underflowing block have scale 0 and codes 0
        assert gs[0][1] == 0 and gs[0][2] == 0 and not gq[0][16:48].any()


def test_compress_exact_grid_and_ties(g):
    """Grid values k * 2^j with |k| = 127 in each block: the scale is 2^j and
    the codes are k; half-way values (k + 1/2) * 2^j round to the even
    integer, as the oracle reads the page's round()."""
    rng = np.random.default_rng(11)
    b, nb = 64, 300
    k = rng.integers(-127, 128, b * nb)
    k[::b] = 127 * rng.choice([-1, 1], nb)
    j = np.repeat(rng.integers(-40, 20, nb), b)
    x = (k * np.exp2(j)).astype(F32)
    half = np.arange(x.size) % b == 5
    x[half] = ((rng.integers(-126, 126, half.sum()) + 0.5) * np.exp2(j[half])).astype(F32)
    got = _compress_on_gpu(g, x[None], None, "f32", b)
    want = _oracle_messages(x[None], None, b)
    _check_messages(got, want, False)
    np.testing.assert_array_equal(got[1][0], np.exp2(j[::b]).astype(F32))
    assert np.all(got[0][0][half].astype(int) % 2 == 0)


@pytest.mark.parametrize("block", [16, 128, 1024])
def test_compress_near_ties_with_arbitrary_scales(g, block):
    """Values a few ulps either side of (k + 1/2) * s for scales that are not
    powers of two: the quotients x / s fall next to half-integers, where only
    the correctly rounded quotient decides the code."""
    rng = np.random.default_rng(block + 1)
    nb = 64
    m = (rng.uniform(0.5, 2.0, nb) * np.exp2(rng.integers(-30, 10, nb))).astype(F32)
    s = (m / F32(127)).astype(F32)
    k = rng.integers(-126, 126, (nb, block)) + 0.5
    x = (k * s[:, None].astype(np.float64)).astype(F32)  # the fp32 nearest to (k + 1/2) * s
    step = rng.integers(-2, 3, x.shape)  # then 0, 1 or 2 ulps up or down
    for _ in range(2):
        x = np.where(step > 0, np.nextafter(x, F32(np.inf)), np.where(step < 0, np.nextafter(x, F32(-np.inf)), x))
        step = step - np.sign(step)
    x = x.astype(F32)
    x[:, 0] = m * rng.choice([-1, 1], nb)
    x = x.reshape(1, -1)
    got = _compress_on_gpu(g, x, None, "f32", block)
    _check_messages(got, _oracle_messages(x, None, block), False)
    e = (rng.standard_normal(x.shape) * 1e-9).astype(F32)
    got = _compress_on_gpu(g, x, e, "f32", block)
    _check_messages(got, _oracle_messages(x, e, block), True)


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("block", [16, 128, 1024])
@pytest.mark.parametrize("N", [1, 2, 5, 8, 16, 64])
def test_compressed_reduce_matches_oracle(g, N, block, out_dtype):
    """The receiving side, fed the oracle's own messages."""
    for L, scale in ((4099, 1.0), (20011, 0.125), (33, 1 / 3)):
        if N == 64 and L > 4099:
            continue
        x, e = _inputs(N, L, "f32", seed=N * 31 + block + L)
        qs, ss, _ = _oracle_messages(x, e, block)
        codes = [torch.from_numpy(q).cuda() for q in qs]
        scales = [torch.from_numpy(s).cuda() for s in ss]
        tdt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
        outs = [torch.full((L,), 3.0, dtype=tdt, device="cuda") for _ in range(N)]
        g.ar_compressed_reduce(codes, scales, outs, block, scale=scale, out_dtype=out_dtype, count=L)
        torch.cuda.synchronize()
        want = C.dequant_allreduce(qs, ss, block, scale=scale, out_dtype=out_dtype)
        for r in range(N):
            assert_bits_equal(to_host(outs[r], out_dtype), want, f"N={N} L={L} rank {r}")


@pytest.mark.parametrize("ef", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("block", BLOCKS)
def test_compressed_allreduce_matches_oracle(g, block, dtype, ef):
    for i, (N, L) in enumerate([(1, 1000), (2, 7), (3, 4103), (8, 20011), (16, 1 << 15), (64, 1029)]):
        x, e = _inputs(N, L, dtype, seed=3 * block + i)
        e = e if ef else None
        scale = (1.0, 1 / N, 0.3)[i % 3]
        grads = _dev(x, dtype)
        res = _dev(e, "f32") if ef else None
        in_place = i % 2 == 1
        outs = None if in_place else [torch.empty_like(t) for t in grads]
        g.ar_compressed_allreduce(grads, block, dtype=dtype, residuals=res, scale=scale, outs=outs, count=L)
        torch.cuda.synchronize()
        want, want_e, _, _ = C.compressed_allreduce(widened(x, dtype), e, block, scale=scale, out_dtype=dtype)
        got = grads if in_place else outs
        for r in range(N):
            assert_bits_equal(to_host(got[r], dtype), want, f"N={N} L={L} rank {r}")
            if not in_place:
                np.testing.assert_array_equal(to_host(grads[r], dtype), x[r])
            if ef:
                assert_bits_equal(to_host(res[r], "f32"), want_e[r], f"residual N={N} L={L} rank {r}")


def _bf16_near_tie_blocks(block, nb, seed):
    """[nb * block] bf16 bit patterns: block k holds its maximum +-m_k first,
    then the bf16 values x whose quotients x / s_k (s_k = RN(m_k / 127)) lie
    closest to a half-integer (within 2^-13, exact ties included), both
    signs. Every m_k is a bf16 value, so s_k is the scale the kernels and the
    oracle compute for the block."""
    rng = np.random.default_rng(seed)
    out = np.zeros((nb, block), np.uint16)
    for k in range(nb):
        exp = int(rng.integers(110, 140))
        if k % 4 == 0:  # m = 127 * 2^j: s is a power of two and ties are exact
            mbits = int(numerics.f32_to_bf16_rne(np.array([127.0 * 2.0 ** (exp - 127)], F32))[0])
        else:
            mbits = (exp << 7) | int(rng.integers(0, 128))
        m = numerics.bf16_to_f32(np.array([mbits], np.uint16))[0]
        s = np.float64(F32(m) / F32(127))
        cand = np.arange(1, mbits, dtype=np.uint16)  # every positive bf16 value below m
        q = numerics.bf16_to_f32(cand).astype(np.float64) / s
        dist = np.abs(q - (np.floor(q) + 0.5))
        near = cand[dist < 2.0 ** -13]
        if near.size == 0:
            near = cand[np.argsort(dist)[:8]]
        vals = np.resize(near, block - 1)
        signs = rng.integers(0, 2, block - 1).astype(np.uint16) << 15
        out[k, 0] = mbits | (np.uint16(rng.integers(0, 2)) << 15)
        out[k, 1:] = vals | signs
        rng.shuffle(out[k, 1:])
    return out.reshape(-1)


@pytest.mark.parametrize("block", [16, 128, 1024])
@pytest.mark.parametrize("N", [2, 3, 4])
def test_compressed_allreduce_bf16_near_ties(g, N, block):
    """bf16 without feedback on quotients next to half-integers and on exact
    ties: the code of every element must be the one the correctly rounded
    quotient gives, so the result is the oracle's bit for bit (even N runs the
    packed kernel, odd N the generic one)."""
    nb = max(8, 4096 // block)
    x = np.stack([_bf16_near_tie_blocks(block, nb, seed=100 * N + block + r) for r in range(N)])
    L = x.shape[1] - 3  # a ragged end as well
    x = np.ascontiguousarray(x[:, :L])
    grads = _dev(x, "bf16")
    outs = [torch.empty_like(t) for t in grads]
    g.ar_compressed_allreduce(grads, block, dtype="bf16", scale=1.0 / N, outs=outs, count=L)
    torch.cuda.synchronize()
    want, _, _, _ = C.compressed_allreduce(widened(x, "bf16"), None, block, scale=1.0 / N, out_dtype="bf16")
    for r in range(N):
        assert_bits_equal(to_host(outs[r], "bf16"), want, f"N={N} rank {r}")


def test_compressed_allreduce_bf16_full_size(g):
    """16 ranks x 96 Mi bf16 without feedback, block 128, x1/16, out of place:
    the packed kernel in the benchmark's launch configuration. The oracle
    checks block-aligned windows (blocks are independent); every rank's result
    is bitwise identical on the whole buffer."""
    spec = workloads.HIER_2X8_BF16
    N, L, block = spec.n_ranks, spec.count, 128
    rng = np.random.default_rng(1)
    starts = np.unique(np.concatenate([[0, L - 4 * block], rng.integers(0, L // block - 8, 48) * block]))
    idx = np.concatenate([np.arange(s, s + 4 * block) for s in starts]).astype(np.int64)
    grads, xs = [], []
    for r in range(N):
        h = workloads.rank_buffer(spec, r)
        grads.append(to_device(h, "bf16"))
        xs.append(h[idx])
        del h
    xs = np.stack(xs)
    outs = [torch.empty_like(t) for t in grads]
    g.ar_compressed_allreduce(grads, block, dtype="bf16", scale=1 / N, outs=outs)
    torch.cuda.synchronize()
    want, _, _, _ = C.compressed_allreduce(widened(xs, "bf16"), None, block, scale=1 / N, out_dtype="bf16")
    didx = torch.from_numpy(idx).cuda()
    for r in range(N):
        assert_bits_equal(outs[r][didx].view(torch.int16).cpu().numpy().view(np.uint16), want, f"rank {r}")
        if r:
            assert torch.equal(outs[r].view(torch.int16), outs[0].view(torch.int16))
    del grads, outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_two_calls_equal_the_fused_pass(g, dtype):
    """ar_compress + ar_compressed_reduce against the oracle, and the fused pass
    bit-identical to them (results and residuals), with error feedback."""
    N, L, block = 6, 50_001, 128
    x, e = _inputs(N, L, dtype, seed=99)
    grads = _dev(x, dtype)
    res_a, res_b = _dev(e, "f32"), _dev(e, "f32")
    nb, _ = g.ar_compress_sizes(L, block)
    codes = [torch.empty(L, dtype=torch.int8, device="cuda") for _ in range(N)]
    scales = [torch.empty(nb, dtype=torch.float32, device="cuda") for _ in range(N)]
    outs_a = [torch.empty_like(t) for t in grads]
    outs_b = [torch.empty_like(t) for t in grads]
    g.ar_compress(grads, codes, scales, block, dtype=dtype, residuals=res_a)
    g.ar_compressed_reduce(codes, scales, outs_a, block, scale=0.5, out_dtype=dtype)
    g.ar_compressed_allreduce(grads, block, dtype=dtype, residuals=res_b, scale=0.5, outs=outs_b)
    torch.cuda.synchronize()
    want, want_e, _, _ = C.compressed_allreduce(widened(x, dtype), e, block, scale=0.5, out_dtype=dtype)
    for r in range(N):
        assert_bits_equal(to_host(outs_a[r], dtype), want, f"two calls rank {r}")
        assert_bits_equal(to_host(outs_b[r], dtype), want, f"fused rank {r}")
        assert_bits_equal(to_host(res_a[r], "f32"), want_e[r], f"residual (two calls) rank {r}")
        assert torch.equal(res_a[r], res_b[r])


def test_error_feedback_over_steps(g):
    """Three training steps with the residuals carried on the device: each
    step's result and residuals equal the oracle's chain, and what was sent
    over the steps plus the last residual equals the sum of the gradients plus
    the first residual (the page's telescoping sum), up to fp32 rounding."""
    N, L, block = 4, 9000, 64
    spec0 = workloads.small_spec(N, L, "f32", "normal", seed=0)
    e0 = np.stack([workloads.residual_buffer(spec0, r) for r in range(N)])
    res = _dev(e0, "f32")
    e = e0.copy()
    sent = np.zeros((N, L))
    gsum = np.zeros((N, L))
    for step in range(3):
        x = workloads.all_ranks(workloads.small_spec(N, L, "f32", "normal", seed=100 + step))
        grads = _dev(x, "f32")
        outs = [torch.empty_like(t) for t in grads]
        g.ar_compressed_allreduce(grads, block, residuals=res, outs=outs)
        torch.cuda.synchronize()
        want, e_new, qs, ss = C.compressed_allreduce(x, e, block)
        for r in range(N):
            assert_bits_equal(to_host(outs[r], "f32"), want, f"step {step} rank {r}")
            assert_bits_equal(to_host(res[r], "f32"), e_new[r], f"residual step {step} rank {r}")
            sent[r] += C.dequantize(qs[r], ss[r], block)
            gsum[r] += x[r]
        e = e_new
    assert np.allclose(sent + e, gsum + e0, rtol=0, atol=1e-9)


def test_compressed_allreduce_of_exact_values_is_the_exact_sum(g):
    """Grid inputs compress losslessly: the result is the exact sum and every
    residual is zero (closed form, independent of the oracle)."""
    rng = np.random.default_rng(5)
    N, b, L = 6, 32, 32 * 300 + 5
    k = rng.integers(-127, 128, (N, L))
    k[:, ::b] = 127
    x = (k * 2.0 ** -10).astype(F32)
    grads = _dev(x, "f32")
    res = [torch.zeros(L, dtype=torch.float32, device="cuda") for _ in range(N)]
    g.ar_compressed_allreduce(grads, b, residuals=res)
    torch.cuda.synchronize()
    want = numerics.reference_sum_f64(x).astype(F32)
    for r in range(N):
        assert_bits_equal(to_host(grads[r], "f32"), want, f"rank {r}")
        assert not res[r].any().item()


def test_compressed_allreduce_full_size(g):
    """16 ranks x 192 MiB fp32 (the all-reduce workload) with error feedback,
    block 128, in the benchmark's launch configuration: the oracle checks
    block-aligned windows (blocks are independent), every rank's result is
    bitwise identical on the whole buffer, and the two-call path equals the
    fused pass on the whole buffer."""
    spec = workloads.RING_N16_192MIB
    N, L, block = spec.n_ranks, spec.count, 128
    rng = np.random.default_rng(0)
    starts = np.unique(np.concatenate([[0, L - 4 * block], rng.integers(0, L // block - 8, 48) * block]))
    idx = np.concatenate([np.arange(s, s + 4 * block) for s in starts]).astype(np.int64)
    grads, res, xs, es = [], [], [], []
    for r in range(N):
        h = workloads.rank_buffer(spec, r)
        grads.append(torch.from_numpy(h).cuda())
        xs.append(h[idx])
        del h
        he = workloads.residual_buffer(spec, r)
        res.append(torch.from_numpy(he).cuda())
        es.append(he[idx])
        del he
    xs, es = np.stack(xs), np.stack(es)
    res_b = [t.clone() for t in res]
    outs = [torch.empty_like(t) for t in grads]
    g.ar_compressed_allreduce(grads, block, residuals=res, scale=1 / N, outs=outs)
    torch.cuda.synchronize()
    want, want_e, _, _ = C.compressed_allreduce(xs, es, block, scale=1 / N)
    for r in range(N):
        assert_bits_equal(outs[r][torch.from_numpy(idx).cuda()].cpu().numpy(), want, f"rank {r}")
        assert_bits_equal(res[r][torch.from_numpy(idx).cuda()].cpu().numpy(), want_e[r], f"residual rank {r}")
        if r:
            assert torch.equal(outs[r].view(torch.int32), outs[0].view(torch.int32))
    nb, _ = g.ar_compress_sizes(L, block)
    codes = [torch.empty(L, dtype=torch.int8, device="cuda") for _ in range(N)]
    scales = [torch.empty(nb, dtype=torch.float32, device="cuda") for _ in range(N)]
    g.ar_compress(grads, codes, scales, block, residuals=res_b)
    outs_b = [torch.empty_like(t) for t in grads]
    g.ar_compressed_reduce(codes, scales, outs_b, block, scale=1 / N)
    torch.cuda.synchronize()
    for r in range(N):
        assert torch.equal(outs_b[r].view(torch.int32), outs[0].view(torch.int32)), r
        assert torch.equal(res_b[r].view(torch.int32), res[r].view(torch.int32)), r
    del grads, res, res_b, outs, outs_b, codes, scales
    torch.cuda.empty_cache()


def test_division_free_scale_equals_the_ieee_quotient_for_every_float(g):
    """The kernels compute the block scale max|x| / 127 without a division;
    over every non-negative float bit pattern it must equal the IEEE
    division's result (NaN for NaN)."""
    assert g.ar_selftest_scale_quotient() == 0


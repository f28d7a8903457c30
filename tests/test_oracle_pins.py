"""The oracle against the values the pages print (worked examples, figures, tables).

Every fixture under tests/golden/ carries its citation.
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import chunks, numerics, schedules

MiB = 1 << 20


def _popcount_grid(w):
    """Contribution count of every (rank, chunk) cell when rank r's input is 2^r
    and each chunk holds one element: the set bits of the fp32 sum."""
    return [[bin(int(v)).count("1") for v in w.x[r]] for r in range(w.N)]


def _provenance_inputs(N):
    return np.array([[float(1 << r)] * N for r in range(N)], dtype=np.float32)


def test_ring_trace_4gpu(golden):
    rows = dict(golden("ring_trace_4gpu.txt"))
    x = np.array([[float(v) for v in rows[f"rank{r}"].split()] for r in range(4)], dtype=np.float32)
    want = np.array([float(v) for v in rows["sum"].split()], dtype=np.float32)
    out, st = schedules.ring_allreduce(x)
    for r in range(4):
        np.testing.assert_array_equal(out[r], want)
    np.testing.assert_array_equal(numerics.reference_sum_f64(x), want)
    np.testing.assert_array_equal(numerics.fused_sum(x, "ring"), want)
    assert st.steps == 2 * (4 - 1)


def test_ring_send_table_fig_4_2(golden):
    N = 4
    _, st = schedules.ring_allreduce(np.zeros((N, N), np.float32))
    table = {}
    for step, src, dst, lo, hi in st.sends:
        assert hi - lo == 1  # one element per chunk, so the element is the chunk
        table.setdefault((src, dst), []).append(lo)
    for key, val in golden("ring_send_table_n4.txt"):
        src, dst = (int(t[1:]) for t in key.split("->"))
        rs, ag = val.split("|")
        want = [int(t[1:]) for t in rs.split()] + [int(t[1:]) for t in ag.split()]
        assert table[(src, dst)] == want, key
    # in every step the N sends carry N different chunks (Fig. 4.2: no chunk twice in a column)
    for s in range(2 * (N - 1)):
        assert sorted(lo for step, _, _, lo, _ in st.sends if step == s) == list(range(N))


def test_ring_grids_fig_4_3(golden):
    N = 4
    rows = golden("ring_grids_n4.txt")
    want = {}
    for key, val in rows:
        fields = dict(f.split("=") for f in val.split())
        want[key] = fields
    x = _provenance_inputs(N)
    start = [[1] * N for _ in range(N)]
    sent_log = []

    def trace(w):
        sent_log.append(int(w.stats.elements_sent[0]))
        return _popcount_grid(w)

    out, st = schedules.ring_allreduce(x, trace=trace)
    names = ["reduce-scatter 1", "reduce-scatter 2", "reduce-scatter 3",
             "all-gather 1", "all-gather 2", "all-gather 3"]
    snapshots = [("start", start)] + [(n, g) for n, (_, g) in zip(names, st.trace)]
    sent = [0] + sent_log
    for (name, grid), s in zip(snapshots, sent):
        w = want[name]
        for r in range(N):
            assert "".join(str(v) for v in grid[r]) == w[f"R{r}"], (name, r)
        assert s == int(w["sent"]), name
        # every rank sends the same number of chunks
    assert len(set(st.elements_sent.tolist())) == 1
    owner = want["owner"]
    for r in range(N):
        lo, hi = st.owned[r]
        assert (lo, hi) == (int(owner[f"R{r}"]), int(owner[f"R{r}"]) + 1)
    # the contributor sets, not only their sizes: after the reduce-scatter the
    # owned chunk holds all four ranks' inputs, and in the end everything does
    np.testing.assert_array_equal(out, np.full((N, N), 15.0, np.float32))


def test_ring_provenance_or_matches_counts():
    """Provenance with bitwise OR on integers gives the same contributor sets as fp32 sums of 2^r."""
    N = 6
    xi = np.array([[1 << r] * N for r in range(N)], dtype=np.uint64)
    out_i, st_i = schedules.ring_allreduce(xi, combine=np.bitwise_or,
                                           trace=lambda w: w.x.copy())
    out_f, st_f = schedules.ring_allreduce(_provenance_inputs(N), trace=lambda w: w.x.copy())
    for (_, gi), (_, gf) in zip(st_i.trace, st_f.trace):
        np.testing.assert_array_equal(gi, gf.astype(np.uint64))
    assert np.all(out_i == (1 << N) - 1)


def test_rabenseifner_fig_4_5(golden):
    rows = golden("rabenseifner_n8.txt")
    N = 8
    x = _provenance_inputs(N)
    held = []

    def trace(w):
        return w.x.copy()

    out, st = schedules.rabenseifner_allreduce(x, trace=trace)
    assert st.steps == 2 * 3
    pairs_by_step = {}
    for step, src, dst, lo, hi in st.sends:
        pairs_by_step.setdefault(step, set()).add(tuple(sorted((src, dst))))
    sends_by_step = {}
    for step, src, dst, lo, hi in st.sends:
        if src == 0:
            sends_by_step[step] = hi - lo
    d = dict((k, v) for k, v in rows if not k.startswith("pairs"))
    for key, val in rows:
        if key.startswith("pairs"):
            k = int(key.split()[1])
            want = {tuple(int(t) for t in p.split("-")) for p in val.split()}
            assert pairs_by_step[k - 1] == want
    # contribution counts: after reduce-scatter step k every element a rank
    # keeps has 2^k contributions; the all-gather only copies
    counts = [int(v) for v in d["contributions"].split()]
    assert counts[0] == 1
    ranges = [(0, N)] * N
    for k in range(1, 4):
        snap = st.trace[k - 1][1]
        new = []
        for i in range(N):
            lo, hi = ranges[i]
            mid = (lo + hi) // 2
            keep = (lo, mid) if ((i >> (k - 1)) & 1) == 0 else (mid, hi)
            new.append(keep)
            vals = snap[i, keep[0]:keep[1]]
            assert all(bin(int(v)).count("1") == counts[k] for v in vals)
        ranges = new
    # bytes per reduce-scatter step and in total, as fractions of S
    halving = [Fraction(v) for v in d["halving sends"].split()]
    assert [Fraction(sends_by_step[s], N) for s in range(3)] == halving
    assert sum(halving) == Fraction(d["halving total"])
    owner = dict(f.split("=") for f in d["owner"].split())
    for r in range(N):
        lo, hi = st.owned[r]
        assert hi - lo == 1 and chr(ord("A") + lo) == owner[f"R{r}"]
        # and the same rule for every N: bit reversal of i
    np.testing.assert_array_equal(out, np.full((N, N), 255.0, np.float32))


@pytest.mark.parametrize("N", [2, 4, 16, 32, 64])
def test_rabenseifner_owner_is_bit_reversal(N):
    _, st = schedules.rabenseifner_allreduce(np.zeros((N, 0), np.float32), idx=np.zeros(0), L=N)
    bits = N.bit_length() - 1
    for i in range(N):
        rev = int(format(i, f"0{bits}b")[::-1], 2) if bits else 0
        assert st.owned[i] == (rev, rev + 1)


def _accounting_run(fn, N, L, **kw):
    return fn(np.zeros((N, 0), np.float32), idx=np.zeros(0, np.int64), L=L, **kw)[1]


def test_192mib_16_ranks_accounting(golden):
    d = dict(golden("allreduce_192mib_16ranks.txt"))
    S = int(d["gradient_bytes"])
    N = int(d["ranks"])
    L = S // 4
    # continuous ring: ranks 0-7 on server A, 8-15 on server B
    st = _accounting_run(schedules.ring_allreduce, N, L, server_of=[i // 8 for i in range(N)])
    assert st.steps == int(d["ring_rounds"])
    assert all(int(e) * 4 == int(d["ring_sent_per_rank_mib"]) * MiB for e in st.elements_sent)
    assert int(st.elements_sent.sum()) * 4 == int(d["ring_sent_total_mib"]) * MiB
    assert {hi - lo for _, _, _, lo, hi in st.sends} == {int(d["ring_edge_round_mib"]) * MiB // 4}
    assert st.cross_elements * 4 == int(d["continuous_ring_cross_mib"]) * MiB
    # interleaved ring 0, 8, 1, 9, ...: ring position i is GPU (i // 2) + 8 * (i % 2)
    gpu = [(i // 2) + 8 * (i % 2) for i in range(N)]
    st = _accounting_run(schedules.ring_allreduce, N, L, server_of=[g // 8 for g in gpu])
    assert st.cross_elements * 4 == int(d["interleaved_ring_cross_mib"]) * MiB
    assert int(st.elements_sent.sum()) * 4 == int(d["ring_sent_total_mib"]) * MiB
    # hierarchical, 2 groups of 8
    st = _accounting_run(schedules.hierarchical_allreduce, N, L, group_size=8,
                         server_of=[i // 8 for i in range(N)])
    assert st.steps == int(d["hier_rounds"])
    assert st.cross_elements * 4 == int(d["hierarchical_cross_mib"]) * MiB
    first = [hi - lo for step, _, _, lo, hi in st.sends if step == 0]
    assert set(first) == {int(d["hier_slice_mib"]) * MiB // 4}
    pair = sum(hi - lo for _, src, dst, lo, hi in st.sends if {src, dst} == {3, 11})
    assert pair * 4 == int(d["hier_pair_mib"]) * MiB
    for r in range(N):
        local = sum(hi - lo for _, src, dst, lo, hi in st.sends if src == r and dst // 8 == r // 8)
        assert local * 4 == int(d["hier_local_per_rank_mib"]) * MiB


@pytest.mark.parametrize("G,M", [(8, 2), (4, 2), (2, 4), (8, 4), (4, 4), (1, 8), (8, 1)])
def test_hierarchical_bytes_formula(G, M):
    """Primer §4.4, Animation 4.3: (G-1)/G*S per GPU on the local links in each of
    phases 1 and 3, and 2(M-1)/M*S/G on the network."""
    N = G * M
    L = 64 * N * N  # divisible by every cut
    st = _accounting_run(schedules.hierarchical_allreduce, N, L, group_size=G,
                         server_of=[i // G for i in range(N)])
    assert st.steps == 2 * (G - 1) + 2 * (M - 1)
    for r in range(N):
        local = sum(hi - lo for _, s, d, lo, hi in st.sends if s == r and d // G == r // G)
        net = sum(hi - lo for _, s, d, lo, hi in st.sends if s == r and d // G != r // G)
        assert Fraction(local, L) == 2 * Fraction(G - 1, G)
        assert Fraction(net, L) == 2 * Fraction(M - 1, M) / G


@pytest.mark.parametrize("N", [2, 3, 4, 5, 7, 8, 16, 64])
def test_ring_bytes_and_steps_closed_form(N):
    """Primer §4.2: 2(N-1) steps and 2(N-1)/N*S bytes per rank, which equals the
    lower bound of (N-1)/N*S each way (Scaling ML Systems, "The bandwidth-optimal
    lower bound")."""
    L = 12 * N
    st = _accounting_run(schedules.ring_allreduce, N, L)
    assert st.steps == 2 * (N - 1)
    assert all(Fraction(int(e), L) == Fraction(2 * (N - 1), N) for e in st.elements_sent)
    # the reduce-scatter half alone meets the one-way lower bound
    rs = [sum(hi - lo for step, s, _, lo, hi in st.sends if s == r and step < N - 1) for r in range(N)]
    assert all(Fraction(v, L) == Fraction(N - 1, N) for v in rs)


@pytest.mark.parametrize("N", [2, 4, 8, 64, 1024])
def test_rabenseifner_bytes_and_steps_closed_form(N):
    """Primer §4.3: 2 log2 N steps with the ring's 2(N-1)/N*S bytes."""
    L = N
    st = _accounting_run(schedules.rabenseifner_allreduce, N, L)
    assert st.steps == 2 * (N.bit_length() - 1)
    assert all(Fraction(int(e), L) == Fraction(2 * (N - 1), N) for e in st.elements_sent)


def test_step_counts_table(golden):
    d = dict(golden("step_counts.txt"))
    st = _accounting_run(schedules.rabenseifner_allreduce, 1024, 1024)
    assert st.steps == int(d["rabenseifner_steps_1024"])
    st = _accounting_run(schedules.ring_allreduce, 8, 8)
    assert st.steps == int(d["ring_steps_8"])
    # the 1,024-rank ring run is long in Python; its count follows the same
    # 2(N-1) law that the N=2..64 runs above pin
    assert 2 * (1024 - 1) == int(d["ring_steps_1024"])


def test_chunk_bounds_ragged():
    assert chunks.chunk_bounds(10, 4) == [0, 2, 5, 7, 10]
    assert chunks.chunk_bounds(3, 8) == [0, 0, 0, 1, 1, 1, 2, 2, 3]
    np.testing.assert_array_equal(chunks.chunk_of(np.arange(10), 10, 4), [0, 0, 1, 1, 1, 2, 2, 3, 3, 3])
    # empty chunks are skipped
    np.testing.assert_array_equal(chunks.chunk_of(np.arange(3), 3, 8), [2, 5, 7])

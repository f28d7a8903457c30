"""Pins of the oracle's schedule variants: recursive doubling, the double binary
tree and the dimension-ordered torus all-reduce. Each is checked against what
the pages print (figures, the comparison table, step counts), against an
independent closed form of its summation order, and against exact arithmetic."""

import math

import numpy as np
import pytest

import workloads
from oracle import cost, numerics, schedules

U32 = 2.0 ** -24


def _inputs(N, L, dist="uniform", seed=0):
    return workloads.all_ranks(workloads.small_spec(N, L, dist=dist, seed=seed), threads=1)


def _provenance(N, L=1):
    return (np.uint64(1) << np.arange(N, dtype=np.uint64))[:, None].repeat(L, axis=1)


def _contributors(w):
    return [int(bin(int(v)).count("1")) for v in w.x[:, 0]]


def _bits_equal(a, b, msg=""):
    np.testing.assert_array_equal(np.asarray(a, np.float32).view(np.uint32),
                                  np.asarray(b, np.float32).view(np.uint32), err_msg=msg)


# ------------------------------------------------------------ recursive doubling


def test_recursive_doubling_fig_4_5(golden):
    rows = dict(golden("recursive_doubling_n8.txt"))
    N, L = 8, 64
    _, st = schedules.recursive_doubling_allreduce(
        _provenance(N, L), combine=np.bitwise_or, trace=_contributors)
    for k in (1, 2, 3):
        want = {tuple(sorted(map(int, p.split("-")))) for p in rows[f"pairs {k}"].split()}
        got = {tuple(sorted((s, d))) for step, s, d, _, _ in st.sends if step == k - 1}
        assert got == want
    contrib = [int(v) for v in rows["contributions"].split()]
    assert [t[1][0] for t in st.trace] == contrib[1:] and contrib[0] == 1
    assert all(len(set(t[1])) == 1 for t in st.trace)  # every rank alike at every step
    per_step = [int(v) for v in rows["doubling sends"].split()]
    for k, frac in enumerate(per_step):
        assert all(sum(hi - lo for step, s, _, lo, hi in st.sends if step == k and s == r) == frac * L
                   for r in range(N))
    assert np.all(st.elements_sent == int(rows["doubling total"]) * L)


def test_recursive_doubling_1024_ranks(golden):
    rows = dict(golden("recursive_doubling_n8.txt"))
    N, L = 1024, 1 << 20
    _, st = schedules.recursive_doubling_allreduce(np.zeros((N, 0), np.float32), idx=np.zeros(0, np.int64), L=L)
    assert st.steps == int(rows["steps_1024"])
    _, ring = schedules.ring_allreduce(np.zeros((N, 0), np.float32), idx=np.zeros(0, np.int64), L=L)
    assert ring.steps == int(rows["ring_steps_1024"])
    assert round(st.elements_sent.max() / ring.elements_sent.max()) == int(rows["bytes_vs_ring_1024"])


@pytest.mark.parametrize("N", [1, 2, 4, 8, 16])
def test_recursive_doubling_order_is_the_balanced_tree(N):
    """Distance 1 first pairs neighbours, then pairs of pairs: the sum is the
    balanced binary tree over ranks in index order -- the fused sum's tree
    order, written independently."""
    for L in (1, 7, 64, 1001):
        x = _inputs(N, L, dist="normal", seed=N + L)
        out, _ = schedules.recursive_doubling_allreduce(x)
        for r in range(N):
            _bits_equal(out[r], out[0])
        _bits_equal(out[0], numerics.fused_sum(x, "tree"))
        ref = numerics.reference_sum_f64(x)
        assert np.all(np.abs(out[0] - ref) <= (N - 1) * U32 * numerics.abs_sum_f64(x))


def test_recursive_doubling_cost_is_the_tree_formula():
    """Round model over the simulation on uniform links: (log2 N) alpha +
    (log2 N) S/B, the primer's tree formula (§4.3)."""
    for N in (2, 8, 64):
        L, alpha, bw = 4096, 5e-6, 450e9
        _, st = schedules.recursive_doubling_allreduce(np.zeros((N, 0), np.float32), idx=np.zeros(0, np.int64),
                                                       L=L)
        got = cost.round_time(st, alpha, lambda s, d: bw, 4)
        assert got == pytest.approx(cost.doubling_formula(alpha, N, 4 * L, bw), rel=1e-12)


def test_recursive_doubling_rejects_other_counts():
    with pytest.raises(ValueError):
        schedules.recursive_doubling_allreduce(np.zeros((6, 4), np.float32))


# ----------------------------------------------------------- double binary tree


def _edges(text):
    return {tuple(map(int, e.split("-"))) for e in text.split()}


def test_double_binary_tree_fig_4_6(golden):
    rows = dict(golden("double_binary_tree_n8.txt"))
    trees = schedules.double_binary_trees(8)
    for t, (parent, children) in enumerate(trees, start=1):
        depth = schedules.tree_depths(parent)
        levels = [sorted(r for r in range(8) if depth[r] == d) for d in range(max(depth) + 1)]
        want = [sorted(map(int, lv.split())) for lv in rows[f"tree{t} levels"].split("|")]
        assert levels == want
        assert {(parent[r], r) for r in range(8) if parent[r] >= 0} == _edges(rows[f"tree{t} edges"])
        assert sorted(r for r in range(8) if children[r]) == sorted(map(int, rows[f"tree{t} inner"].split()))
    assert len(trees) == int(rows["trees"])


@pytest.mark.parametrize("N", range(2, 65, 2))
def test_double_binary_tree_inner_nodes_disjoint(N):
    """No node is an inner node in both trees (Fig. 4.6): even ranks forward in
    tree 1, odd ranks in tree 2. Each tree spans every rank."""
    (p1, c1), (p2, c2) = schedules.double_binary_trees(N)
    inner1 = {r for r in range(N) if c1[r]}
    inner2 = {r for r in range(N) if c2[r]}
    assert not inner1 & inner2
    assert inner1 <= set(range(0, N, 2)) and inner2 <= set(range(1, N, 2))
    for parent in (p1, p2):
        assert sum(1 for r in range(N) if parent[r] < 0) == 1
        assert all(d <= N for d in schedules.tree_depths(parent))  # no cycles


def test_single_binary_tree_bytes_table(golden):
    """Not pipelined, a binary tree makes a leaf send S (up) and an inner GPU
    with a parent and two children 3S (S up, S to each child)."""
    rows = dict(golden("double_binary_tree_n8.txt"))
    N, L = 16, 100
    _, st = schedules.double_binary_tree_allreduce(np.zeros((N, L), np.float32), n_trees=1)
    parent, children = schedules.binary_tree(N)
    for r in range(N):
        if not children[r]:
            assert st.elements_sent[r] == int(rows["single_tree_leaf_sends"]) * L
        elif parent[r] >= 0 and len(children[r]) == 2:
            assert st.elements_sent[r] == int(rows["single_tree_inner_sends"]) * L


def test_tree_steps_are_about_two_log2_n(golden):
    rows = dict(golden("double_binary_tree_n8.txt"))
    _, st = schedules.double_binary_tree_allreduce(np.zeros((1024, 0), np.float32), idx=np.zeros(0, np.int64),
                                                   L=1 << 20)
    assert st.steps == int(rows["tree_steps_1024"])
    _, st8 = schedules.double_binary_tree_allreduce(np.zeros((8, 4), np.float32))
    assert st8.steps == 2 * 3


def _tree_fold(x, children, r, cols):
    """Closed form of a tree's sum order: P(r) = (g_r + P(c1)) + P(c2), the
    children c1 < c2 in rank order."""
    acc = x[r, cols].astype(np.float32)
    for c in sorted(children[r]):
        acc = (acc + _tree_fold(x, children, c, cols)).astype(np.float32)
    return acc


@pytest.mark.parametrize("N", [2, 3, 5, 8, 12, 16])
def test_double_binary_tree_order_closed_form(N, golden):
    """Each half is the recursive fold of its tree, from the root; every rank
    ends with the same bits; integer inputs give the exact sum."""
    L = 37
    x = _inputs(N, L, dist="normal", seed=N)
    out, st = schedules.double_binary_tree_allreduce(x)
    trees = schedules.double_binary_trees(N)
    if N == 8:  # the figure's own edges, not the construction's
        rows = dict(golden("double_binary_tree_n8.txt"))
        trees = []
        for t in (1, 2):
            ch = [[] for _ in range(N)]
            for a, b in sorted(_edges(rows[f"tree{t} edges"])):
                ch[a].append(b)
            par = [-1] * N
            for a, b in _edges(rows[f"tree{t} edges"]):
                par[b] = a
            trees.append((par, [sorted(c) for c in ch]))
    h = L // 2
    for t, (lo, hi) in enumerate(((0, h), (h, L))):
        parent, children = trees[t]
        want = _tree_fold(x, children, parent.index(-1), np.arange(lo, hi))
        for r in range(N):
            _bits_equal(out[r, lo:hi], want, f"tree {t + 1} rank {r}")
    xi = _inputs(N, 501, dist="int")
    outi, _ = schedules.double_binary_tree_allreduce(xi)
    np.testing.assert_array_equal(outi, np.broadcast_to(numerics.reference_sum_f64(xi).astype(np.float32),
                                                        outi.shape))


def test_double_binary_tree_busiest_rank_sends_about_the_ring():
    """Each tree carries S/2: a rank inner in one tree sends S/2 up and S/2 to
    each of two children there and S/2 up as a leaf of the other, 2S at most,
    near the ring's 2(N-1)/N S (primer §4.3)."""
    N, L = 64, 1000
    _, st = schedules.double_binary_tree_allreduce(np.zeros((N, L), np.float32))
    assert st.elements_sent.max() == 2 * L
    _, ring = schedules.ring_allreduce(np.zeros((N, L), np.float32))
    assert st.elements_sent.max() / ring.elements_sent.max() < 1.02


# ------------------------------------------------------------------------ torus


def test_torus_4x4_steps(golden):
    rows = dict(golden("torus_4x4.txt"))
    X, Y = map(int, rows["dims"].split())
    x = _provenance(X * Y)
    _, st = schedules.torus_allreduce(x, (X, Y), combine=np.bitwise_or, trace=_contributors)
    assert st.steps == int(rows["torus_steps"])
    px, py = map(int, rows["phase_steps"].split())
    names = [t[0] for t in st.trace]
    assert sum(n.startswith("dim X") for n in names) == px and sum(n.startswith("dim Y") for n in names) == py
    _, flat = schedules.ring_allreduce(np.zeros((X * Y, 16), np.float32))
    assert flat.steps == int(rows["flat_ring_steps"])
    assert flat.steps / st.steps == float(rows["step_ratio"])
    # after phase 1 (its all-gather included) every rank holds its row's X
    # inputs; after phase 2 all of them
    assert set(st.trace[px - 1][1]) == {X}
    assert set(st.trace[-1][1]) == {X * Y}


def _nested_fold(x, dims, e, L):
    """Closed form of the dimension-ordered sum of element e: along each line,
    the ring's left fold from the position that owns e's chunk; the lines'
    results folded the same way along the next dimension."""
    X, Y, Z = list(dims) + [1] * (3 - len(dims))
    cx, cy, cz = (int(np.searchsorted(np.array([(c * L) // D for c in range(D + 1)]), e, side="right")) - 1
                  for D in (X, Y, Z))

    def fold(vals, start):
        n = len(vals)
        acc = np.float32(vals[start % n])
        for j in range(1, n):
            acc = np.float32(acc + vals[(start + j) % n])
        return acc

    def line(y, z):
        return fold([x[xx + X * (y + Y * z), e] for xx in range(X)], cx)

    def plane(z):
        return fold([line(y, z) for y in range(Y)], cy)

    return fold([plane(z) for z in range(Z)], cz)


@pytest.mark.parametrize("dims", [(4, 4), (2, 8), (8, 2), (3, 5), (2, 3, 2), (2, 2, 2), (1, 6), (5, 1), (1, 1)])
def test_torus_order_closed_form(dims):
    N = math.prod(dims)
    L = 53
    x = _inputs(N, L, dist="normal", seed=N * 7 + len(dims))
    out, _ = schedules.torus_allreduce(x, dims)
    want = np.array([_nested_fold(x, dims, e, L) for e in range(L)], np.float32)
    for r in range(N):
        _bits_equal(out[r], want, f"rank {r}")


def test_torus_of_one_line_is_the_ring():
    x = _inputs(6, 301, dist="normal", seed=5)
    ring, _ = schedules.ring_allreduce(x)
    for dims in ((6,), (6, 1), (1, 6), (1, 1, 6)):
        out, st = schedules.torus_allreduce(x, dims)
        _bits_equal(out, ring, str(dims))
        assert st.steps == 10


def test_torus_rejects_wrong_dims():
    with pytest.raises(ValueError):
        schedules.torus_allreduce(np.zeros((16, 4), np.float32), (4, 3))

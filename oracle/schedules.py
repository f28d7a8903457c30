"""Step-by-step simulations of the all-reduce schedules, one virtual rank at a time.

Every schedule is a sequence of synchronous steps. In a step every rank first
puts its outgoing payload in the receiver's mailbox (a copy taken before any
rank changes its buffer), then every receiver combines what arrived with its
own copy (reduce-scatter: add; all-gather: overwrite). This is the step
semantics the primer states (ch. 4 "Collective communication: algorithms,
cost and the library that runs them", §4.2 "The ring, one step at a time": in
each step all links carry one chunk at the same time, and a step cannot
start until the previous chunk has arrived and been added).

A simulation runs on K elements of every rank's buffer: by default all of
them, or a sample given by their indices ``idx`` in the full buffer of L
elements. Elements never interact, so a sample gives exactly the values the
full run would give at those indices; byte and step counters are always
counted for the full buffer.

``combine`` is the reduce-scatter operation (default: fp32 addition). Passing
``numpy.bitwise_or`` with inputs 1 << r ("provenance mode") records which
ranks contributed to each element.

``finish`` is applied by each owner to its complete part at the end of the
reduce-scatter, before the all-gather copies it around: scaling by 1/N and
rounding to bf16 happen there, once per element.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .chunks import chunk_bounds


@dataclass
class RunStats:
    steps: int = 0
    elements_sent: np.ndarray = None  # per rank, over the full buffer
    element_reads: int = 0  # buffer reads by senders and receivers, all ranks
    element_writes: int = 0  # buffer writes by receivers, all ranks
    cross_elements: int = 0  # elements sent between ranks on different servers
    owned: dict = field(default_factory=dict)  # rank -> (lo, hi) complete after reduce-scatter
    sends: list = field(default_factory=list)  # (step, src, dst, lo, hi) for every send
    trace: list = field(default_factory=list)


class _World:
    def __init__(self, x, idx, L, server_of, trace):
        self.x = np.array(x, copy=True)
        self.N, K = self.x.shape
        self.idx = np.arange(K, dtype=np.int64) if idx is None else np.asarray(idx, dtype=np.int64)
        if self.idx.shape != (K,):
            raise ValueError("idx must give one buffer index per column")
        self.L = K if L is None else int(L)
        self.server_of = server_of
        self.stats = RunStats(elements_sent=np.zeros(self.N, dtype=np.int64))
        self.trace_fn = trace

    def cols(self, lo, hi):
        return np.nonzero((self.idx >= lo) & (self.idx < hi))[0]

    def count_send(self, src, dst, lo, hi, reduce):
        s = self.stats
        n = hi - lo
        s.sends.append((s.steps, src, dst, lo, hi))
        s.elements_sent[src] += n
        # a send reads the sender's copy; the receiver reads its own copy when
        # it adds, and writes its copy either way
        s.element_reads += n * (2 if reduce else 1)
        s.element_writes += n
        if self.server_of is not None and self.server_of[src] != self.server_of[dst]:
            s.cross_elements += n

    def end_step(self, name):
        self.stats.steps += 1
        if self.trace_fn is not None:
            self.stats.trace.append((name, self.trace_fn(self)))


def _ring_phase(w: _World, rings, rule, reduce, combine, name):
    """Run one ring phase on several independent rings in lockstep.

    ``rings`` is a list of (members, lo, hi): the ranks of one ring in ring
    order (position p sends to position p+1, the last wraps to the first) and
    the element segment [lo, hi) that ring works on, cut into len(members)
    parts. ``rule(p, s)`` is the part that position p sends at step s.
    Returns, per ring, the part each position received last.
    """
    n = len(rings[0][0])
    assert all(len(m) == n for m, _, _ in rings)
    last = [[None] * n for _ in rings]
    for s in range(n - 1):
        mailbox = []
        for ri, (members, lo, hi) in enumerate(rings):
            b = [lo + (p * (hi - lo)) // n for p in range(n + 1)]
            for p in range(n):
                part = rule(p, s) % n
                q = (p + 1) % n
                cols = w.cols(b[part], b[part + 1])
                payload = w.x[members[p], cols].copy()
                mailbox.append((ri, q, members[q], part, cols, payload))
                w.count_send(members[p], members[q], b[part], b[part + 1], reduce)
        for ri, q, dst, part, cols, payload in mailbox:
            if reduce:
                w.x[dst, cols] = combine(payload, w.x[dst, cols])
            else:
                w.x[dst, cols] = payload
            last[ri][q] = part
        w.end_step(f"{name} {s}")
    return last


def _apply_finish(w, rank, lo, hi, finish):
    if finish is None:
        return
    cols = w.cols(lo, hi)
    if cols.size:
        w.x[rank, cols] = finish(w.x[rank, cols])


def _add(a, b):
    return a + b


def ring_allreduce(x, idx=None, L=None, combine=_add, finish=None, server_of=None, trace=None):
    """Ring all-reduce (primer §4.2, Fig. 4.1-4.3; Scaling ML Systems, "Ring AllReduce").

    Ranks 0..N-1 form a ring; rank i sends to rank i+1 mod N. The buffer is cut
    into N chunks. Reduce-scatter step s = 0..N-2: rank i sends chunk
    (i - s) mod N and the receiver adds its own copy. All-gather step
    s = 0..N-2: rank i sends the complete chunk (i + 1 - s) mod N and the
    receiver overwrites its copy. Returns (buffers, RunStats).
    """
    w = _World(x, idx, L, server_of, trace)
    N = w.N
    ring = [(list(range(N)), 0, w.L)]
    if N > 1:
        last = _ring_phase(w, ring, lambda p, s: p - s, True, combine, "reduce-scatter")[0]
        b = chunk_bounds(w.L, N)
        for i in range(N):
            c = last[i]
            w.stats.owned[i] = (b[c], b[c + 1])
            _apply_finish(w, i, b[c], b[c + 1], finish)
        _ring_phase(w, ring, lambda p, s: p + 1 - s, False, combine, "all-gather")
    else:
        w.stats.owned[0] = (0, w.L)
        _apply_finish(w, 0, 0, w.L, finish)
    return w.x, w.stats


def rabenseifner_allreduce(x, idx=None, L=None, combine=_add, finish=None, server_of=None,
                           trace=None):
    """Rabenseifner's all-reduce: recursive halving, then recursive doubling.

    Primer §4.3 (Fig. 4.5, Animation 4.2) and Scaling ML Systems ("Recursive
    halving and doubling (butterfly)"). N must be a power of two. Each rank
    keeps a current range of chunk indices, initially all N chunks.
    Reduce-scatter step k = 1..log2 N: rank i pairs with p = i xor 2^(k-1),
    keeps the lower half of its range if bit k-1 of i is 0 and the upper half
    otherwise, sends the other half to p and adds the half that p sends. The
    all-gather runs the same pairs in reverse order (k = log2 N..1) and copies
    the partner's range, doubling the range each step.
    """
    w = _World(x, idx, L, server_of, trace)
    N = w.N
    if N & (N - 1):
        raise ValueError("Rabenseifner needs a power-of-two rank count")
    b = chunk_bounds(w.L, N)
    rng = [(0, N) for _ in range(N)]  # chunk index ranges
    n_steps = N.bit_length() - 1
    for k in range(1, n_steps + 1):
        d = 1 << (k - 1)
        mailbox = []
        new_rng = list(rng)
        for i in range(N):
            p = i ^ d
            lo, hi = rng[i]
            mid = (lo + hi) // 2
            keep, send = ((lo, mid), (mid, hi)) if ((i >> (k - 1)) & 1) == 0 else ((mid, hi), (lo, mid))
            new_rng[i] = keep
            cols = w.cols(b[send[0]], b[send[1]])
            mailbox.append((p, cols, w.x[i, cols].copy()))
            w.count_send(i, p, b[send[0]], b[send[1]], True)
        for p, cols, payload in mailbox:
            w.x[p, cols] = combine(payload, w.x[p, cols])
        rng = new_rng
        w.end_step(f"reduce-scatter {k}")
    for i in range(N):
        lo, hi = b[rng[i][0]], b[rng[i][1]]
        w.stats.owned[i] = (lo, hi)
        _apply_finish(w, i, lo, hi, finish)
    for k in range(n_steps, 0, -1):
        d = 1 << (k - 1)
        mailbox = []
        for i in range(N):
            p = i ^ d
            lo, hi = rng[i]
            cols = w.cols(b[lo], b[hi])
            mailbox.append((p, cols, w.x[i, cols].copy()))
            w.count_send(i, p, b[lo], b[hi], False)
        for p, cols, payload in mailbox:
            w.x[p, cols] = payload
        rng = [(min(rng[i][0], rng[i ^ d][0]), max(rng[i][1], rng[i ^ d][1])) for i in range(N)]
        w.end_step(f"all-gather {k}")
    return w.x, w.stats


def hierarchical_allreduce(x, group_size, idx=None, L=None, combine=_add, finish=None,
                           server_of=None, trace=None):
    """Hierarchical all-reduce over M = N/G groups of G consecutive ranks.

    Primer §4.4 (Fig. 4.8, Animation 4.3); AI Infra Book ch. 7 ("Data-center
    networks"), §7.2.1, task 7.2. The buffer is cut into G slices.

    1. Reduce-scatter inside every group, a ring over local ranks 0..G-1 in
       which local rank l sends slice (l - 1 - s) mod G at step s, so that
       local rank k ends owning slice k.
    2. For every slice k, a ring all-reduce among the M ranks that own it (local
       rank k of every group, in group order), over slice k cut into M
       sub-chunks, by the ring rules of ``ring_allreduce``.
    3. All-gather inside every group: local rank l sends slice (l - s) mod G.

    ``finish`` runs on each sub-chunk's owner after the reduce-scatter of
    phase 2, the point where its sum is complete.
    """
    w = _World(x, idx, L, server_of, trace)
    N, G = w.N, int(group_size)
    if G < 1 or N % G:
        raise ValueError("group size must divide the rank count")
    M = N // G
    groups = [[g * G + l for l in range(G)] for g in range(M)]
    sb = chunk_bounds(w.L, G)
    if G > 1:
        _ring_phase(w, [(m, 0, w.L) for m in groups], lambda p, s: p - 1 - s, True, combine,
                    "intra-group reduce-scatter")
    peers = [([g * G + k for g in range(M)], sb[k], sb[k + 1]) for k in range(G)]
    if M > 1:
        last = _ring_phase(w, peers, lambda p, s: p - s, True, combine, "inter-group reduce-scatter")
    for k, (members, lo, hi) in enumerate(peers):
        sub = [lo + (j * (hi - lo)) // M for j in range(M + 1)]
        for p, r in enumerate(members):
            j = last[k][p] if M > 1 else 0
            w.stats.owned[r] = (sub[j], sub[j + 1])
            _apply_finish(w, r, sub[j], sub[j + 1], finish)
    if M > 1:
        _ring_phase(w, peers, lambda p, s: p + 1 - s, False, combine, "inter-group all-gather")
    if G > 1:
        _ring_phase(w, [(m, 0, w.L) for m in groups], lambda p, s: p - s, False, combine,
                    "intra-group all-gather")
    return w.x, w.stats


def ring_reduce_scatter(x, idx=None, L=None, combine=_add, finish=None, server_of=None, trace=None):
    """Standalone ring reduce-scatter: every rank ends with one chunk of the sum.

    The primer's table of collectives (§4.1) defines the operation (all ranks
    hold S, each ends with S/N of the sum, sending (N-1)/N*S) but not which
    chunk each rank keeps. Reading taken: rank i keeps chunk i, the usual
    assignment. On the ring that is the slice rule of the hierarchical
    reduce-scatter (primer §4.4): at step s = 0..N-2 rank i sends chunk
    (i - 1 - s) mod N to rank i+1, which adds its own copy. After N-1 steps
    rank i holds the complete chunk i; its other chunks hold partial sums.
    """
    w = _World(x, idx, L, server_of, trace)
    N = w.N
    b = chunk_bounds(w.L, N)
    if N > 1:
        last = _ring_phase(w, [(list(range(N)), 0, w.L)], lambda p, s: p - 1 - s, True, combine,
                           "reduce-scatter")[0]
    else:
        last = [0]
    for i in range(N):
        c = last[i]
        w.stats.owned[i] = (b[c], b[c + 1])
        _apply_finish(w, i, b[c], b[c + 1], finish)
    return w.x, w.stats


def ring_allgather(x, idx=None, L=None, server_of=None, trace=None):
    """Standalone ring all-gather: rank i contributes chunk i of its buffer and
    every rank ends with all N chunks (primer §4.1 table: (N-1)/N*S sent per
    rank). Step s = 0..N-2: rank i sends chunk (i - s) mod N to rank i+1, which
    overwrites its copy (the slice rule of the hierarchical all-gather, §4.4)."""
    w = _World(x, idx, L, server_of, trace)
    N = w.N
    if N > 1:
        _ring_phase(w, [(list(range(N)), 0, w.L)], lambda p, s: p - s, False, _add, "all-gather")
    return w.x, w.stats


def recursive_doubling_allreduce(x, idx=None, L=None, combine=_add, finish=None, server_of=None,
                                 trace=None):
    """Recursive doubling (primer §4.3, "Trees: latency-optimal, bandwidth-poor",
    Fig. 4.5). N must be a power of two. Step k = 1..log2 N: every rank i sends
    its whole buffer to p = i xor 2^(k-1) and adds the whole buffer p sends.
    After log2 N steps every rank holds the full sum, so ``finish`` runs on
    every rank's whole buffer and every rank owns [0, L)."""
    w = _World(x, idx, L, server_of, trace)
    N = w.N
    if N & (N - 1):
        raise ValueError("recursive doubling needs a power-of-two rank count")
    every = w.cols(0, w.L)
    for k in range(1, N.bit_length()):
        d = 1 << (k - 1)
        mailbox = []
        for i in range(N):
            mailbox.append((i ^ d, w.x[i, every].copy()))
            w.count_send(i, i ^ d, 0, w.L, True)
        for p, payload in mailbox:
            w.x[p, every] = combine(payload, w.x[p, every])
        w.end_step(f"doubling {k}")
    for i in range(N):
        w.stats.owned[i] = (0, w.L)
        _apply_finish(w, i, 0, w.L, finish)
    return w.x, w.stats


def binary_tree(N):
    """Tree 1 of the double binary tree over ranks 0..N-1 (primer §4.3, Fig. 4.6).

    Reading of the figure (8 nodes: root 0 above 4, then 2 and 6, then the odd
    ranks as leaves; the inner nodes are the even ranks): ranks 1..N-1 form the
    in-order binary tree in which rank r with lowest set bit b >= 2 has
    children r - b/2 and r + b/2 (the right child's offset halved until it
    names a rank below N; none if it reaches 0), and the top of that tree, the
    largest power of two below N, hangs under the root, rank 0. Odd ranks are
    leaves. Returns (parent, children): parent[0] = -1, children in ascending
    rank order.
    """
    parent = [-1] * N
    children = [[] for _ in range(N)]

    def link(a, c):
        assert parent[c] == -1 and c != 0, (a, c)
        parent[c] = a
        children[a].append(c)

    if N > 1:
        link(0, 1 << ((N - 1).bit_length() - 1))
        for r in range(1, N):
            b = r & -r
            if b < 2:
                continue
            link(r, r - b // 2)
            off = b // 2
            while off >= 1 and r + off >= N:
                off //= 2
            if off >= 1:
                link(r, r + off)
    for c in children:
        c.sort()
    return parent, children


def double_binary_trees(N):
    """The two trees of the double binary tree: tree 1 from ``binary_tree`` and
    tree 2 its mirror, rank r becoming N-1-r (primer §4.3, Fig. 4.6). Returns
    [(parent, children), (parent, children)]."""
    p1, c1 = binary_tree(N)
    m = [N - 1 - r for r in range(N)]
    p2 = [-1] * N
    c2 = [[] for _ in range(N)]
    for r in range(N):
        if p1[r] >= 0:
            p2[m[r]] = m[p1[r]]
        c2[m[r]] = sorted(m[c] for c in c1[r])
    return [(p1, c1), (p2, c2)]


def tree_depths(parent):
    """Depth of every node below its root (root 0)."""
    depth = []
    for r in range(len(parent)):
        d, q = 0, r
        while parent[q] >= 0:
            q = parent[q]
            d += 1
        depth.append(d)
    return depth


def double_binary_tree_allreduce(x, idx=None, L=None, combine=_add, finish=None, server_of=None,
                                 trace=None, n_trees=2):
    """All-reduce over NCCL-style double binary trees (primer §4.3, Fig. 4.6 and
    the table of ring, tree and Rabenseifner; Scaling ML Systems, "Double
    binary tree").

    With two trees, tree t carries half t of the buffer ([0, floor(L/2)) and
    the rest); with ``n_trees=1``, tree 1 carries all of it (a plain binary
    tree). Reduce: level by level from the deepest inner nodes up, every inner
    node receives its children's partial sums of its tree's half and folds
    them into its own copy: (own + first child) + second child, children in
    ascending rank order. Both trees run their levels in the same steps (tree
    2 is a mirror image, so the levels line up). The root's sum is complete:
    ``finish`` runs there. Broadcast: level by level from the root down, every
    parent sends the result to its children, which overwrite their copies.

    Byte counters follow the data movement of a step: a child's send reads its
    copy; a receiving node reads its own copy once and writes it once, however
    many children it has.
    """
    w = _World(x, idx, L, server_of, trace)
    N = w.N
    if n_trees not in (1, 2):
        raise ValueError("one or two trees")
    trees = double_binary_trees(N)[:n_trees]
    halves = chunk_bounds(w.L, n_trees)
    depths = [tree_depths(p) for p, _ in trees]
    top = max(max(d) for d in depths) if N > 1 else 0
    s = w.stats
    for level in range(top - 1, -1, -1):
        mailbox = []
        for t, (parent, children) in enumerate(trees):
            lo, hi = halves[t], halves[t + 1]
            cols = w.cols(lo, hi)
            for r in range(N):
                if depths[t][r] != level or not children[r]:
                    continue
                payloads = [w.x[c, cols].copy() for c in children[r]]
                for c in children[r]:
                    s.sends.append((s.steps, c, r, lo, hi))
                    s.elements_sent[c] += hi - lo
                    s.element_reads += hi - lo
                    if server_of is not None and server_of[c] != server_of[r]:
                        s.cross_elements += hi - lo
                s.element_reads += hi - lo
                s.element_writes += hi - lo
                mailbox.append((r, cols, payloads))
        for r, cols, payloads in mailbox:
            acc = w.x[r, cols]
            for pl in payloads:
                acc = combine(pl, acc)
            w.x[r, cols] = acc
        w.end_step(f"tree reduce {level}")
    for t, (parent, _) in enumerate(trees):
        root = parent.index(-1)
        s.owned[(t, root)] = (halves[t], halves[t + 1])
        _apply_finish(w, root, halves[t], halves[t + 1], finish)
    for level in range(top):
        mailbox = []
        for t, (parent, children) in enumerate(trees):
            lo, hi = halves[t], halves[t + 1]
            cols = w.cols(lo, hi)
            for r in range(N):
                if depths[t][r] != level:
                    continue
                for c in children[r]:
                    mailbox.append((c, cols, w.x[r, cols].copy()))
                    w.count_send(r, c, lo, hi, False)
        for c, cols, payload in mailbox:
            w.x[c, cols] = payload
        w.end_step(f"tree broadcast {level}")
    return w.x, w.stats


def torus_allreduce(x, dims, idx=None, L=None, combine=_add, finish=None, server_of=None, trace=None):
    """Dimension-ordered all-reduce on an X x Y (x Z) torus (Scaling ML Systems,
    "Collective communication", section on torus topologies, the TPU-pod
    figure and the three-step list).

    Rank (x, y, z) is x + X*(y + Y*z). Dimension by dimension (X, then Y, then
    Z) every line of ranks along that dimension, in coordinate order, runs the
    ring all-reduce of ``ring_allreduce`` over the whole buffer cut into as many
    chunks as the line has ranks; all lines of a dimension run in lockstep.
    The next dimension reduces the partial sums the previous one left on every
    rank. ``finish`` runs once, on the owners of the last dimension's chunks.
    Steps: the sum of 2(D-1) over the dimensions (4 x 4: 12, against 30 for a
    flat ring of 16).
    """
    w = _World(x, idx, L, server_of, trace)
    N = w.N
    dims = [int(d) for d in dims] + [1] * (3 - len(dims))
    X, Y, Z = dims
    if min(dims) < 1 or X * Y * Z != N:
        raise ValueError("torus dimensions must multiply to the rank count")
    stride = [1, X, X * Y]
    active = [d for d in range(3) if dims[d] > 1]
    if not active:
        w.stats.owned[0] = (0, w.L)
        _apply_finish(w, 0, 0, w.L, finish)
        return w.x, w.stats
    for d in active:
        D = dims[d]
        lines = []
        for r in range(N):
            if (r // stride[d]) % D == 0:  # first rank of its line
                lines.append(([r + p * stride[d] for p in range(D)], 0, w.L))
        last = _ring_phase(w, lines, lambda p, s: p - s, True, combine, f"dim {'XYZ'[d]} reduce-scatter")
        if d == active[-1]:
            b = chunk_bounds(w.L, D)
            for li, (members, _, _) in enumerate(lines):
                for p, r in enumerate(members):
                    c = last[li][p]
                    w.stats.owned[r] = (b[c], b[c + 1])
                    _apply_finish(w, r, b[c], b[c + 1], finish)
        _ring_phase(w, lines, lambda p, s: p + 1 - s, False, combine, f"dim {'XYZ'[d]} all-gather")
    return w.x, w.stats


# ----------------------------------------------------------------- helpers


def finish_scale(scale: float):
    """The owner's final step for an fp32 result: multiply once by ``scale``."""
    s = np.float32(scale)
    return None if scale == 1.0 else (lambda v: (np.asarray(v, np.float32) * s).astype(np.float32))


def finish_bf16(scale: float = 1.0):
    """The owner's final step for a bf16 result: multiply by ``scale`` in fp32,
    then round once to bf16 (kept here as the fp32 value of the bf16 number)."""
    from .numerics import bf16_to_f32, f32_to_bf16_rne

    s = np.float32(scale)
    return lambda v: bf16_to_f32(f32_to_bf16_rne(np.asarray(v, np.float32) * s))


SCHEDULES = {
    "ring_reduce_scatter": ring_reduce_scatter,
    "ring_allgather": ring_allgather,
    "ring": ring_allreduce,
    "rabenseifner": rabenseifner_allreduce,
    "hier": hierarchical_allreduce,
    "recdoubling": recursive_doubling_allreduce,
    "dbtree": double_binary_tree_allreduce,
    "torus": torus_allreduce,
}

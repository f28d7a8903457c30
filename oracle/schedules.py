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
}

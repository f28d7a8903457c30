"""Critical path of a training step whose gradient communication overlaps the
backward computation.

AI Infra Book ch. 7 (zh-tw edition, "資料中心網路"), §7.6.1 and §7.6.2 (example
7.6): a collective can start only when its data are ready (the start of a
group exchange is the latest readiness time of its members); communication
that starts before the computation ends runs beside it on resources that do
not contend; the update waits for both. For one message ready at r with
communication time T_n, computation ending at T_c and an update of T_u:
T_step = max(T_c, r + T_n) + T_u.

Buckets generalise this (Scaling ML Systems, "Collective communication",
sections on layer-wise overlap and bucket fusion): bucket b becomes ready at
r_b, the buckets' collectives run one after another on one communication
stream, so bucket b starts at max(r_b, end of bucket b-1).
"""

from __future__ import annotations


def group_completion(ready_times, exchange: float) -> float:
    """A group exchange starts when its last member is ready (§7.6.1)."""
    return max(ready_times) + exchange


def comm_timeline(ready, durations):
    """(start, end) of each bucket's collective on one communication stream."""
    out, end = [], 0.0
    for r, d in zip(ready, durations):
        start = max(r, end)
        end = start + d
        out.append((start, end))
    return out


def step_time(ready, durations, compute_end: float, update: float = 0.0) -> float:
    """T_step = max(end of computation, end of the last collective) + update."""
    tl = comm_timeline(ready, durations)
    last = tl[-1][1] if tl else 0.0
    return max(compute_end, last) + update


def exposed(ready, durations, compute_end: float) -> float:
    """Communication time that the computation does not hide."""
    tl = comm_timeline(ready, durations)
    return max(0.0, (tl[-1][1] if tl else 0.0) - compute_end)


def speedup(t_unaffected: float, t_comm: float, s: float) -> float:
    """Whole-step speedup when only the communication gets s times faster (§7.6.2):
    S = (T_c + T_n) / (T_c + T_n / s)."""
    return (t_unaffected + t_comm) / (t_unaffected + t_comm / s)

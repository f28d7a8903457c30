"""The benchmark's multi-process harness on CPU: two gloo ranks, barrier-bracketed
timing, maximum over ranks, and the reference arm's rank-0-only rule."""

import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    w, r, _ = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    steps = []

    def step():  # rank 1 is the straggler: 20 ms per step against 1 ms
        time.sleep(0.02 if r == 1 else 0.001)
        steps.append(1)

    ms = bench.timed(dist, step, lambda: None, n_steps=5, n_warmup=3)
    q.put((r, ms, len(steps)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ms = {r: v for r, v, _ in out}
    assert all(n == 8 for _, _, n in out)  # 3 warm-up + 5 timed steps each
    assert ms[0] == ms[1]  # both ranks hold the maximum
    assert ms[0] >= 5 * 20  # the straggler's time, not rank 0's


def _leaver(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    w, r, _ = bench.dist_env()
    dist = bench.init_dist(w, "gloo", timeout_s=10)
    if r == 1:  # leaves between steps, before the timed region: never reaches its barrier
        q.put((r, "left", 0.0))
        q.close()
        q.join_thread()  # flush the queue before the hard exit
        os._exit(0)
    t0 = time.time()
    try:
        bench.timed(dist, lambda: None, lambda: None, n_steps=5, n_warmup=3)
        q.put((r, "no error", time.time() - t0))
    except Exception as e:  # the barrier fails instead of waiting for the missing rank
        q.put((r, type(e).__name__, time.time() - t0))
    q.close()
    q.join_thread()
    os._exit(0)


def test_missing_rank_fails_the_barrier_instead_of_hanging():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_leaver, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = {r: (what, secs) for r, what, secs in (q.get(timeout=120) for _ in procs)}
    for p in procs:
        p.join(timeout=60)
    assert out[1][0] == "left"
    assert out[0][0] != "no error", out
    assert out[0][1] < 60, out


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True,
                         timeout=300)
    assert res.returncode == 0 and res.stdout.strip() == ""


def test_reference_arm_line():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_warmup_floor():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                         capture_output=True, text=True, timeout=120)
    assert res.returncode != 0

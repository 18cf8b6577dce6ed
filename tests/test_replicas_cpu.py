"""The N-process host logic of bench.py (replicas: one per rank, no data-path
collective) on two CPU ranks over gloo: barriers, the maximum over ranks,
whole-job throughput, and the reference arm's rank-0-only rule."""
from __future__ import annotations

import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    reps = bench.Replicas("gloo")
    reps.barrier()
    ms_local = 10.0 + 5.0 * rank          # rank 1 is the slower one
    ms = reps.max(ms_local)
    rate = reps.throughput(2.0e9, ms)     # 2 GFLOP per rank per step
    reps.close()
    q.put((rank, reps.world, ms, rate))


def test_two_gloo_ranks_max_and_whole_job_throughput():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, world, ms, rate in results:
        assert world == 2
        assert ms == 15.0                 # the slowest rank's time, on every rank
        assert rate == pytest.approx(2 * 2.0e9 / 15.0e-3)


def test_single_process_needs_no_process_group(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    sys.path.insert(0, ROOT)
    import bench
    reps = bench.Replicas("gloo")
    assert reps.dist is None and reps.world == 1
    assert reps.max(3.5) == 3.5
    assert reps.throughput(1.0e9, 2.0) == pytest.approx(5.0e11)
    reps.close()


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    # under torchrun the other ranks leave without work (and print nothing)
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1",
                                      "--warmup", "3"])
    sys.path.insert(0, ROOT)
    import bench
    called = []
    monkeypatch.setattr(bench, "reference_arm", lambda args: called.append(args))
    assert bench.main() is None
    assert called == []


def _rank_leaves_main(rank, world, port, q, stall_s=0.0):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import time

    import bench
    reps = bench.Replicas("gloo", timeout_s=5.0)
    if rank == 1:
        if stall_s:
            time.sleep(stall_s)           # alive but stuck: never reaches the barrier
        q.put((rank, "left", 0.0))
        q.close()
        q.join_thread()                   # the message is out before the process is
        os._exit(0)                       # leaves between steps, without a word
    t0 = time.monotonic()
    try:
        reps.barrier()
        q.put((rank, "passed", time.monotonic() - t0))
    except Exception as e:                # the backend reports the missing peer
        q.put((rank, type(e).__name__, time.monotonic() - t0))
    q.close()
    q.join_thread()
    os._exit(0)


def test_a_rank_that_leaves_makes_the_next_barrier_fail_not_hang():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_leaves_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict((r, (what, dt)) for r, what, dt in (q.get(timeout=120) for _ in procs))
    for p in procs:
        p.join(timeout=60)
    assert results[1][0] == "left"
    what, dt = results[0]
    assert what != "passed" and dt < 60.0, results


def test_a_stuck_rank_makes_the_next_barrier_fail_after_the_timeout():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_leaves_main, args=(r, 2, port, q, 15.0)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict((r, (what, dt)) for r, what, dt in (q.get(timeout=120) for _ in procs))
    for p in procs:
        p.join(timeout=60)
    what, dt = results[0]
    assert what != "passed" and 3.0 < dt < 14.0, results   # the 5 s timeout, not the peer

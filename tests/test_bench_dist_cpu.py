"""The benchmark's multi-process host logic on CPU: two ranks over gloo (127.0.0.1).

Each replica times its own work; the job's time is the slowest rank's and its rate counts
the units every rank processed (weak scaling, replicas only: no data-path collective)."""
import os
import queue
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    dist, ws2, rank2, _ = bench._dist()
    try:
        ms = bench.max_over_ranks(dist, 1.0 + rank)  # rank 1 is the slow one
        rate = bench.job_rate(ws2, 1000, ms)
        q.put((rank2, ws2, ms, rate, dist.get_backend()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_time_and_all_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = []
    try:
        for _ in procs:
            res.append(q.get(timeout=180))
    except queue.Empty:
        pytest.fail("a rank did not report")
    finally:
        for p in procs:
            p.join(60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    for rank, ws, ms, rate, backend in sorted(res):
        assert backend == "gloo" and ws == 2
        assert ms == 2.0  # max over the ranks, seen by both
        assert rate == pytest.approx(2 * 1000 / 2e-3)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.job_rate(1, 32768, 1.0) == pytest.approx(32768e3)

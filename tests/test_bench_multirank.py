"""bench.py's multi-rank path on the CPU: two gloo ranks (world size 2).

Every GPU run of this project has one GPU, so the N > 1 logic of the bench
(max over ranks of the timed region, whole-job throughput, the reference
arm run by rank 0 alone) is covered here with gloo process groups.
"""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, ms_per_rank, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(ms_per_rank[rank], "cpu", dist.group.WORLD)
        sec, value, per_launch = bench.job_throughput(1_000_000, world, ms, 10)
        ref = bench.run_reference(None, world, rank) if rank != 0 else None
        q.put((rank, ms, sec, value, per_launch, ref))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ms_per_rank = [3.0, 5.0]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, ms_per_rank, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, sec, value, per_launch, ref in got:
        assert ms == 5.0                       # max over ranks, on every rank
        assert sec == pytest.approx(5e-4)      # 5 ms / 10 steps
        assert value == pytest.approx(2 * 1e6 / 5e-4 / 1e9)   # both ranks' bytes
        assert per_launch == pytest.approx(1e6 / 5e-4 / 1e9)
    assert got[1][5] == 0                      # reference arm: rank 1 exits without work


def test_single_rank_passes_time_through():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, "cpu", None) == 7.5
    sec, value, per_launch = bench.job_throughput(2_000_000, 1, 4.0, 8)
    assert sec == pytest.approx(5e-4) and value == pytest.approx(per_launch)

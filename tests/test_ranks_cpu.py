"""The bench's cross-rank logic on two gloo ranks (CPU, no GPU): the timed
region is the slowest rank's, and the reported rate counts the units of
every rank (replicas of the step, weak scaling)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, ms_of_rank, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.max_over_ranks(dist, ms_of_rank[rank], "cpu")
        q.put((rank, m, bench.whole_job_rate(4096, world, m)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_every_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ms_of_rank = [3.0, 5.0]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, ms_of_rank, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    for _ in procs:
        rank, m, v = q.get(timeout=120)
        got[rank] = (m, v)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        m, v = got[rank]
        assert m == 5.0
        assert v == pytest.approx(4096 * 2 / 5e-3)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(None, 2.5, "cpu") == 2.5
    assert bench.whole_job_rate(64, 1, 0.5) == pytest.approx(128000.0)

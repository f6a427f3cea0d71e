"""The bench's multi-rank path on CPU: two gloo ranks, each timing its own
replica, reduce to the slowest rank's time and report the whole-job value."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 20.0][rank]
        m = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
        v = bench.job_value(1e12, 10, world, m)
        dist.barrier()
        q.put((rank, m, v))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, v in res:
        assert m == 20.0                                            # slowest rank's time on every rank
        assert v == pytest.approx(2 * 1e12 * 10 / 0.020 / 1e12)     # both replicas' work / that time


def test_single_process_helpers():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, None, None) == 3.0
    assert bench.job_value(2e12, 5, 1, 1000.0) == pytest.approx(10.0)

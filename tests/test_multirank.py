"""Multi-rank host logic of the benchmark with two gloo ranks on the CPU:
each rank is an independent replica (own requests, own pool); the step time is
the slowest rank's, and the whole-job rate counts every rank's units."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench._dist() == (world, rank, rank)
    ms = 0.1 + 0.05 * rank  # rank 1 is the slower one
    slow = bench.max_over_ranks(ms)
    rate = bench.whole_job_rate(1.0, world, slow)
    out.put((rank, slow, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_max_and_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, slow, rate in res:
        assert slow == pytest.approx(0.15)
        assert rate == pytest.approx(2 / 0.15e-3)


def test_single_process_helpers():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(32 * 2048, 1, 0.5) == pytest.approx(32 * 2048 / 0.5e-3)

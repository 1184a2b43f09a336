"""bench.py's multi-rank timing on CPU: two gloo ranks, barrier + max over
ranks + whole-job rate (replicas: every rank runs the same workload)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(True)
        t = bench.max_over_ranks(10.0 + rank, True)       # rank 1 is the slowest
        rate = bench.whole_job_rate(100.0, world, t)
        out.put((rank, t, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, rate in res:
        assert t == 11.0                      # max over ranks
        assert rate == pytest.approx(200.0 / 11.0)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, False) == 3.5
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0

"""The bench's multi-rank aggregation on CPU: two gloo ranks, each timing a
different step time; the job's value is every rank's units over the slowest
rank's time, and every rank agrees on it."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [2.0, 5.0][rank]
    value, t_max = bench.job_throughput(ms, 48, world, "cpu")
    q.put((rank, value, t_max))
    dist.barrier()
    dist.destroy_process_group()


def test_job_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for _, value, t_max in got:
        assert t_max == 5.0
        assert value == pytest.approx(48 * 2 / 5.0e-3)


def test_job_throughput_one_rank_is_local():
    import bench
    value, t_max = bench.job_throughput(4.0, 48, 1, "cpu")
    assert t_max == 4.0 and value == pytest.approx(48 / 4.0e-3)

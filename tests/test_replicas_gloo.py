"""The replica path of bench.py on two CPU ranks (gloo): every rank gets the
slowest rank's time, and the whole-job rate counts the tokens of all ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [0.5, 2.0][rank]
    slowest = bench.max_over_ranks(elapsed, dist, "cpu")
    rate = bench.whole_job_rate(world, 10, 256.0, slowest)
    q.put((rank, slowest, rate))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_replicas_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=100) for _ in range(world))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for rank, slowest, rate in out:
        assert slowest == 2.0
        assert rate == pytest.approx(2 * 10 * 256.0 / 2.0)

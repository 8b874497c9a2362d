"""The N>1 bench path on CPU: two gloo ranks, max-over-ranks timing and the
whole-job (weak-scaling) throughput, with no data-path collective."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [100.0, 250.0][rank]
    value, ms = bench.aggregate_throughput(1e12, 10, local_ms, world)
    q.put((rank, value, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, value, ms in got:
        assert ms == 250.0                      # every rank sees the slowest rank's time
        assert value == pytest.approx(2 * 1e12 * 10 / 0.25 / 1e12)  # both ranks' work over that time


def test_single_process_is_identity():
    import bench
    value, ms = bench.aggregate_throughput(2e12, 5, 50.0, 1)
    assert ms == 50.0 and value == pytest.approx(2e12 * 5 / 0.05 / 1e12)

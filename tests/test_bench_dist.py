"""The multi-rank bench path on CPU: two gloo ranks with different step times
must both see the slower rank's time, and the job throughput counts the keys
of every rank over that time (independent replicas, no data exchange)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [3.0, 5.0][rank]
        ms = bench.reduce_max_ms(local, dist, torch.device("cpu"))
        q.put((rank, ms, bench.job_throughput(ms / 2, 1 << 28, world)))
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
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in got:
        assert ms == 5.0
        assert value == pytest.approx(2 * (1 << 28) / 2.5e-3 / 1e9)


def test_single_process_passthrough():
    import bench
    assert bench.reduce_max_ms(4.0, None, None) == 4.0
    assert bench.job_throughput(2.0, 1000, 1) == pytest.approx(1000 / 2e-3 / 1e9)

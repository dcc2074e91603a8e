"""Multi-rank host logic of bench.py on CPU: two gloo ranks run replicas with
different step times; the job time is the slowest rank's and the value is
the bytes of all ranks over that time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, e2e = bench.reduce_times_over_ranks(10.0 + 5.0 * rank, 2.0 - rank, world, "cpu")
    q.put((rank, ms, e2e, bench.aggregate_value(1_000_000_000, world, ms / 1e3)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, e2e, value in out:
        assert ms == 15.0            # max of 10 and 15
        assert e2e == 2.0            # max of 2 and 1
        assert value == pytest.approx(2 * 1e9 / 0.015 / 1e12)


def test_single_rank_is_unchanged():
    import bench
    assert bench.reduce_times_over_ranks(3.0, 4.0, 1) == (3.0, 4.0)
    assert bench.aggregate_value(10**12, 1, 1.0) == 1.0

"""The N > 1 path of bench.py on CPU: two gloo ranks, each timing its own batch (weak scaling).

Rows are independent, so ranks exchange nothing on the data path; the only cross-rank step is the
maximum of the per-rank times, from which the whole-job value is computed.
"""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local_ms = [120.0, 200.0][rank]  # the second rank is slower
    value, max_ms = bench.aggregate_ranks(local_ms, 1000)
    q.put((rank, value, max_ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, value, max_ms in got:
        assert max_ms == 200.0
        assert value == pytest.approx(2 * 1000 / 0.2)


def test_single_process_value():
    import bench

    value, max_ms = bench.aggregate_ranks(50.0, 100)
    assert max_ms == 50.0 and value == pytest.approx(2000.0)

"""The N > 1 path of bench.py on CPU: two gloo ranks, each timing its own batch (weak scaling).

Rows are independent, so ranks exchange nothing on the data path; the only cross-rank step is the
maximum of the per-rank times, from which the whole-job value is computed. The ranks' batches form one
batch: bench.shard_rows gives each rank its rows and its row_offset, which keys every row's race noise by
the row's index in the whole batch; the oracle run shard by shard with those keys must then draw what it
draws over the whole batch.
"""
import os
import socket

import numpy as np
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


def _shard_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from oracle import sample_row, widen_logits
    from top_support_capture_gb300 import workloads as wl

    w = wl.config2(step=5)  # the job's batch: 64 rows of 32000 bf16 logits
    per = w.B // world
    row0, row1 = bench.shard_rows(rank, per)

    def shard(keys):  # this rank's rows, the race keyed by `keys`
        return [sample_row(widen_logits(w.logits[r], w.dtype), float(w.temperature[r]), int(w.top_k[r]),
                           float(w.top_p[r]), float(w.min_p[r]), w.seed, w.step, int(k)).token
                for r, k in zip(range(row0, row1), keys)]

    mine = torch.tensor([row0, row1] + shard(range(row0, row1)), dtype=torch.int64)
    local_keys = torch.tensor(shard(range(0, row1 - row0)), dtype=torch.int64)  # row_offset left at 0
    got = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(got, mine)
    got_local = [torch.empty_like(local_keys) for _ in range(world)]
    dist.all_gather(got_local, local_keys)
    if rank == 0:
        q.put(([g.numpy() for g in got], [g.numpy() for g in got_local]))
    dist.barrier()
    dist.destroy_process_group()


def test_shards_with_global_row_keys_draw_the_whole_batch():
    from oracle import sample_filter_capture
    from top_support_capture_gb300 import workloads as wl

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got, got_local = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    w = wl.config2(step=5)
    whole = sample_filter_capture(w.logits, w.dtype, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, w.step,
                                  w.capture, w.packed_width)
    # the shards tile the batch in rank order
    assert [(int(g[0]), int(g[1])) for g in got] == [(0, 32), (32, 64)]
    tokens = np.concatenate([g[2:] for g in got])
    np.testing.assert_array_equal(tokens, whole.tokens)
    # keyed by the shard's own row indices instead, the second shard draws other tokens
    assert (got_local[1] != whole.tokens[32:]).any()
    np.testing.assert_array_equal(got_local[0], whole.tokens[:32])

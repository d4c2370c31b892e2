"""The multi-GPU story is replicas: each rank runs its own batch with no data-path collective;
the benchmark only takes the max elapsed time and the summed work over ranks.  This checks
that reduction with two gloo ranks on the CPU."""

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

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, _ = bench.dist_env()
    elapsed = [0.5, 0.8][rank]
    units = [100.0, 300.0][rank]
    bench.barrier()
    t, u = bench.reduce_max_sum(elapsed, units)
    q.put((r, ws, t, u))
    dist.destroy_process_group()


def test_two_rank_reduction_takes_max_time_and_sum_of_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 0.8, 400.0), (1, 2, 0.8, 400.0)]


def test_single_process_reduction_is_identity():
    import bench
    assert bench.reduce_max_sum(1.25, 7.0) == (1.25, 7.0)

"""The benchmark's multi-rank path on CPU: two gloo ranks, each timing its own
replica, agree on the slowest rank's duration (weak scaling: no data-path
collective, only the timing reduction)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [0.25, 0.75][rank]
    q.put((rank, bench.reduce_max(local, "cpu"), bench.dist_setup()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [0.75, 0.75]
    assert [g[2] for g in got] == [(2, 0, 0), (2, 1, 1)]


def test_single_process_identity():
    import bench
    assert bench.reduce_max(1.5, "cpu") == 1.5

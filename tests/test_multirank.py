"""The multi-GPU path of bench.py is independent replicas (the layer has no
exchange step without expert parallelism): each rank times its own batch,
the job time is the slowest rank's, and throughput counts every rank's
tokens.  Checked with world_size 2 over gloo on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [12.0, 20.0][rank]
    total = bench.max_over_ranks(local_ms, dist)
    value = bench.replica_throughput(world, 4096, total / 4)
    q.put((rank, total, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
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
    for rank, total, value in res:
        assert total == 20.0
        assert value == pytest.approx(2 * 4096 / (5.0 / 1000.0))

"""The benchmark's multi-process bookkeeping on the CPU: N replicas (world
size 2, gloo) agree on the slowest rank's time, and the whole-job value
counts every rank's rows over that time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [30.0, 45.0][rank]          # rank 1 is the slow one
    value, ms_per_step = bench.aggregate_throughput(8192, 40, local_ms, world, torch.device("cpu"))
    bench.barrier(world)
    out[rank] = (value, ms_per_step)
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    ms = 45.0 / 40
    for rank in range(world):
        value, ms_per_step = res[rank]
        assert ms_per_step == pytest.approx(ms)
        assert value == pytest.approx(8192 * world / (ms / 1e3))

"""bench.py's multi-process path on the CPU: two gloo ranks stand in for two
GPUs running independent replicas; the job's step time is the slowest
rank's and the value counts every rank's bytes."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local_ms = [2.0, 3.5][rank]
    step_ms, value = bench.aggregate(local_ms, 10**9, world)
    bench.barrier(world)
    out[rank] = (step_ms, value)
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        step_ms, value = res[r]
        assert step_ms == pytest.approx(3.5)
        assert value == pytest.approx(2 * 1e9 / 3.5e-3 / 1e9)

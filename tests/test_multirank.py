"""The replica path of bench.py with two ranks over gloo on the CPU: every
rank reports the slowest rank's step time, and the throughput counts the
tokens of both replicas.  No GPU and no collective on the data path."""
import os
import socket

import pytest
import torch
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
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        def all_reduce_max(v):
            t = torch.tensor([v], dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            return float(t.item())

        ms_local = 0.010 + 0.005 * rank          # rank 1 is the slow one
        ms, value = bench.aggregate(ms_local, 32, world, all_reduce_max)
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_slowest_rank_and_all_tokens():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in range(world):
        ms, value = res[rank]
        assert ms == pytest.approx(0.015)
        assert value == pytest.approx(world * 32 / 0.015e-3)


def test_single_replica_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.aggregate(0.02, 32, 1, lambda v: v)
    assert ms == 0.02 and value == pytest.approx(32 / 0.02e-3)

"""The multi-GPU path of bench.py runs independent replicas (the decode hot path has no
exchange step on one GPU): the step time is the slowest rank's and the bytes are summed.
Checked here with two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms_local = [4.0, 5.0][rank]
    ms, total, value = bench.aggregate_replicas(torch, world, ms_local, 1_000_000_000 * (rank + 1),
                                                torch.device("cpu"))
    out[rank] = (ms, total, value)
    bench.barrier(torch, world)
    dist.destroy_process_group()


def test_two_replicas_take_slowest_time_and_sum_bytes():
    import torch.multiprocessing as mp
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        for rank in range(2):
            ms, total, value = out[rank]
            assert ms == 5.0
            assert total == 3e9
            assert value == pytest.approx(3e9 / 5e-3 / 1e9)


def test_single_rank_is_identity():
    import torch
    sys.path.insert(0, ROOT)
    import bench
    ms, total, value = bench.aggregate_replicas(torch, 1, 2.5, 5e9, torch.device("cpu"))
    assert (ms, total) == (2.5, 5e9) and value == pytest.approx(2000.0)

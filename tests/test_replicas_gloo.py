"""The multi-GPU path is replicas only: every rank runs its own verify step
and the benchmark reports the slowest rank's time.  This checks that host
logic (barrier + max over ranks) with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dist.barrier()
    got = bench.max_over_ranks(1.5 + rank)       # rank 1 is the slow replica
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_process_returns_its_own_value():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25

"""The multi-rank host logic of bench.py on CPU ranks (gloo, world size 2).

Each rank smooths its own replica; the job figure is the units summed over
ranks divided by the slowest rank's time.  No GPU is used here.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_setup()
        assert (ws, r, local) == (world, rank, rank)
        ms, units = bench.aggregate(100.0 + 50.0 * rank, 1000.0 * (rank + 1))
        results[rank] = (ms, units)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_aggregate_two_ranks_gloo():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_rank, args=(world, _free_port(), results), nprocs=world,
                       start_method="spawn", join=True)
    assert dict(results) == {0: (150.0, 3000.0), 1: (150.0, 3000.0)}


def test_aggregate_single_process():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(12.5, 7.0) == (12.5, 7.0)

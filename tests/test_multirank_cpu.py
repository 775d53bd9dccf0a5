"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the job's
time is the slowest rank's, and throughput counts every rank's work.  The
attention path itself has no exchange between ranks (independent replicas),
so this aggregation is the only cross-rank step."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [10.0 + rank, 5.0 - rank, 3.0 * (rank + 1)]
    res = bench.max_over_ranks(mine, world, "cpu")
    out[rank] = torch.tensor(res)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    for r in range(world):
        assert out[r].tolist() == [11.0, 5.0, 6.0]


def test_single_rank_is_identity_and_job_throughput():
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1, "cpu") == [1.5, 2.5]
    # 2 ranks x 10 TFLOP per step x 3 steps in 0.06 s = 1000 TFLOP/s
    assert bench.job_tflops(10e12, 2, 3, 0.06) == pytest.approx(1000.0)

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


def _bench(args, env_extra):
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    env.update(env_extra)
    return subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], env=env,
                          capture_output=True, text=True, timeout=600)


def test_bench_gpus_flag_must_match_the_launcher():
    """Under a launcher that started one rank, --gpus 2 is refused (exit 2)
    instead of reporting one GPU's work as two."""
    r = _bench(["--gpus", "2", "--impl", "reference", "--workload", "tiny_causal"],
               {"WORLD_SIZE": "1", "RANK": "0"})
    assert r.returncode == 2 and "WORLD_SIZE" in r.stderr


def test_bench_gpus_flag_starts_its_own_ranks():
    """Without a launcher, --gpus 2 starts two ranks itself (torch.distributed.run,
    gloo for the reference arm on CPU); rank 0 alone prints the line."""
    import json
    r = _bench(["--gpus", "2", "--impl", "reference", "--workload", "tiny_causal",
                "--steps", "1", "--warmup", "3", "--ref-rows", "4"], {})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1 and lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2

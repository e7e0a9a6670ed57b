"""The benchmark's multi-rank path on CPU with the gloo backend (world size 2).

Ranks run independent replicas of the batch (weak scaling): each draws its
own inputs of the same shape, and the only exchange is the max over ranks of
the step timings.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads as wl


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's own timings; the job's are the max over ranks
        mine = [1.0 + rank, 0.5 * (2 - rank), 3.0 + 0.25 * rank]
        got = bench.max_over_ranks(mine, world)
        # replicas: same shape, different draws
        step = wl.make_workload("tiny-decode", seed=bench.replica_seed("tiny-decode", rank))
        sig = torch.tensor([float(step.query.float().sum()), float(step.num_tokens)], dtype=torch.float64)
        sigs = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(sigs, sig)
        torch.save({"max": got, "sigs": [s.tolist() for s in sigs]}, os.path.join(out_dir, f"r{rank}.pt"))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_run_distinct_replicas(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [torch.load(os.path.join(tmp_path, f"r{r}.pt")) for r in range(world)]
    for r in res:
        assert r["max"] == [2.0, 1.0, 3.25]
    sigs = res[0]["sigs"]
    assert sigs[0][1] == sigs[1][1]                 # same shape
    assert sigs[0][0] != sigs[1][0]                 # different draws


def test_job_throughput_counts_every_rank():
    assert bench.job_throughput(1e9, 1, 1.0) == pytest.approx(1000.0)
    assert bench.job_throughput(1e9, 4, 2.0) == pytest.approx(2000.0)
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]


def test_step_percentiles_are_nearest_rank():
    assert bench.percentiles(list(range(1, 11))) == [1, 5, 9]
    assert bench.percentiles([7.5]) == [7.5, 7.5, 7.5]
    assert bench.percentiles([3.0, 1.0, 2.0], (0.0, 1.0)) == [1.0, 3.0]

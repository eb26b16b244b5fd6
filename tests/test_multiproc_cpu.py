"""The multi-rank benchmark path on CPU: two gloo ranks, as torchrun would
start them.  Each rank gets its own batch (no shared data), the timed region
is the maximum over ranks, and the job value counts every rank's work over
that maximum.  No collective touches the data path, so none is tested."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from attention_distillation_kl_gb300.workloads import WORKLOADS, generate_head


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.rank_workload(WORKLOADS["pr1"], rank)
        q1 = generate_head(w, 0, 0)[0]
        # every rank reports its own "time"; the job time is the slowest one
        t = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
        seeds = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(seeds, torch.tensor([w.seed]))
        firsts = [torch.zeros(4) for _ in range(world)]
        dist.all_gather(firsts, q1[0, :4].float())
        dist.barrier()
        out[rank] = (t, [int(x) for x in seeds], [f.tolist() for f in firsts])
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    t0, seeds0, firsts0 = out[0]
    t1, _, _ = out[1]
    assert t0 == t1 == 15.0                      # max over ranks, seen by all
    assert len(set(seeds0)) == world             # each rank its own seed
    assert firsts0[0] != firsts0[1]              # hence its own data


def test_job_value_counts_every_rank():
    assert bench.job_tflops(1, 2e12, 1000.0) == pytest.approx(2.0)
    assert bench.job_tflops(4, 2e12, 1000.0) == pytest.approx(8.0)
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5

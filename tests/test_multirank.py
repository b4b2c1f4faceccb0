"""The N > 1 path of bench.py on CPU: world-size-2 gloo ranks run the same rank bookkeeping the
GPU job runs (per-rank replica seeds, the maximum step time over ranks, whole-job throughput).
The units of the hot path are independent, so ranks exchange nothing but this timing."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 1.5 + rank  # rank 1 is the slow one
        ms = bench.slowest_rank_ms(my_ms, world, "cpu")
        value = bench.job_throughput(1000, world, ms)
        seed = bench.replica_seed(7, rank)
        # every rank must agree on the job's numbers
        t = torch.tensor([ms, value, float(seed)], dtype=torch.float64)
        gathered = [torch.zeros(3, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(gathered, t)
        out[rank] = [g.tolist() for g in gathered]
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(rank_main, args=(world, free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        rows = out[rank]
        for r, (ms, value, seed) in enumerate(rows):
            assert ms == pytest.approx(2.5)                     # max over ranks
            assert value == pytest.approx(1000 * 2 / 2.5e-3)     # all ranks' entries / slowest
            assert seed == 7 + r                                  # one replica per rank


def test_single_rank_is_unchanged():
    assert bench.slowest_rank_ms(3.25, 1, "cpu") == 3.25
    assert bench.job_throughput(500, 1, 2.0) == pytest.approx(250000.0)

"""The multi-rank aggregation of bench.py, on CPU with two gloo ranks.

Under torchrun every rank times its own replica of the workload; the job's step
lasts as long as its slowest rank, so bench.py takes the element-wise maximum of
the per-rank times over the process group and reports the bytes of all ranks
over that time.  Two spawned gloo ranks with different times check the maximum
reaches every rank, and the whole-job throughput uses it.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: step times (1 + r) ms and (5 - r) ms
        out[rank] = bench.max_over_ranks([1.0 + rank, 5.0 - rank])
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(rank_main, args=(world, free_port(), out), nprocs=world, join=True)
        got = dict(out)
    assert got == {0: [2.0, 5.0], 1: [2.0, 5.0]}


def test_max_over_ranks_without_process_group():
    assert bench.max_over_ranks([3, 1.5]) == [3.0, 1.5]


def test_whole_job_throughput_uses_the_slowest_rank():
    # two ranks of 1 GB each, slowest step 0.5 ms: 4000 GB/s for the job
    assert bench.whole_job_gbs(10 ** 9, 2, 0.5) == pytest.approx(4000.0)
    assert bench.whole_job_gbs(10 ** 9, 1, 0.5) == pytest.approx(2000.0)

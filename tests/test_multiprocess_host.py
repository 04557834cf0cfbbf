"""The N > 1 host logic of bench.py on CPU with two gloo ranks: each rank gets
its own workload, the job's step time is the slowest rank's, and the job-wide
throughput counts every rank's work.  (No GPU: the ranks only exchange
timings, the data path has no collective.)"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [2.5, 4.0][rank]                      # rank 1 is the slow one
    ms_max = bench.max_over_ranks(ms)
    value = bench.job_throughput_tflops(1e12, world, ms_max)
    results[rank] = (ms_max, value, bench.rank_seed(7, rank))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_reduction_and_seeds():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), results), nprocs=world,
                       start_method="spawn", join=True)
    assert results[0][0] == results[1][0] == 4.0          # max over ranks
    assert results[0][1] == pytest.approx(2e12 / 4e-3 / 1e12)   # both ranks' work / slowest time
    assert results[0][2] != results[1][2]                 # distinct workloads per rank


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_throughput_tflops(4e11, 1, 0.5) == pytest.approx(800.0)


def test_rank_workloads_differ():
    import bench
    import workloads
    a = workloads.prefix_loguniform_blocks(64, 128, 32768, 64, bench.rank_seed(0, 0))
    b = workloads.prefix_loguniform_blocks(64, 128, 32768, 64, bench.rank_seed(0, 1))
    assert a != b

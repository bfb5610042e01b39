"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): every rank
gets the slowest rank's time, and the job throughput counts every rank's
work over that time.  The GPU path uses the same functions over NCCL."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 1000.0 + 250.0 * rank  # rank 1 is slower
        out[rank] = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == 1250.0


def test_single_process_is_identity():
    assert bench.max_over_ranks(12.5) == 12.5


def test_job_tflops_counts_all_ranks():
    fl = bench._flops(1, 32, 262144, 128, 14)
    one = bench.job_tflops(fl, 2000.0, 1)
    assert bench.job_tflops(fl, 2000.0, 4) == pytest.approx(4 * one)
    # 14 * D * B * H * S(S+1)/2 at S = 262144 is 1.970e15 FLOP
    assert fl == pytest.approx(1.970e15, rel=1e-3)
    assert one == pytest.approx(fl / 2.0 / 1e12)

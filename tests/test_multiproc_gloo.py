"""The multi-rank path of the benchmark on CPU: two gloo ranks, each a
replica with its own workload seed, reduce their timings to the slowest
rank and report whole-job throughput (weak scaling; no data-path
collective exists, requests are independent)."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    from self_speculative_verification_gb300 import workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 10.0 + 5.0 * rank                  # rank 1 is the slow one
        slowest = bench.max_over_ranks(my_ms, "cpu")
        wl = W.make_workload("tiny_la", 0 + rank)  # each replica has its own seed
        value = bench.job_throughput(wl.verified_tokens(), 4, world, slowest)
        out[rank] = (slowest, value, int(wl.seq_len.sum()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_slowest():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    ctx = mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 15.0
    assert out[0][1] == out[1][1] == pytest.approx(8 * 4 * 2 / 0.015)
    assert out[0][2] == out[1][2]          # same shapes; tiny_la fixes the lengths


def test_single_process_reduction_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(512, 10, 1, 1000.0) == pytest.approx(5120.0)

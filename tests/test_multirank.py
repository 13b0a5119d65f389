"""The multi-GPU (weak scaling) host logic of bench.py, on two gloo ranks on the CPU.

Every rank decodes its own batch of the workload's shape with no data-path
collective; the only exchange is the max over ranks of the time per step.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from paged_kv_cache_61_gb300 import synth, traffic


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's own batch: same shape, different seed
        case = synth.workload("gqa_tiny", seed=rank)
        kv = traffic.gqa_kv_bytes(case.context_lens.tolist(), case.num_kv_heads, case.head_dim_qk, 2)
        local_ms = 1.0 + rank                      # rank 1 is the slower one
        ms = bench.reduce_step_time(local_ms, dist, "cpu")
        results[rank] = (ms, kv, int(case.context_lens.sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    port = _free_port()
    manager = mp.Manager()
    results = manager.dict()
    mp.spawn(_rank_main, args=(2, port, results), nprocs=2, join=True)
    assert results[0][0] == results[1][0] == 2.0
    # the ranks drew different batches of the same shape
    assert results[0][2] != results[1][2]


def test_weak_scaling_rate_counts_every_rank():
    assert bench.whole_job_rate(1e9, 1, 1.0) == pytest.approx(1e12)
    assert bench.whole_job_rate(1e9, 4, 2.0) == pytest.approx(2e12)
    assert bench.reduce_step_time(3.5, None, "cpu") == 3.5

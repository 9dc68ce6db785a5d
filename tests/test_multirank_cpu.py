"""The N>1 host logic of bench.py with two gloo ranks on CPU: the timed
interval is the max over ranks on every rank, the whole-job value counts the
work of all ranks, and only rank 0 of the reference arm does any work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([10.0 + rank, 5.0 - rank, 3.0])
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == [11.0, 5.0, 3.0] and out[1] == [11.0, 5.0, 3.0]


def test_single_process_max_is_identity():
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]


def test_whole_job_value_counts_every_rank():
    one = bench.whole_job_tflops(549.76e9, 1, 10, 10 * 0.4)
    two = bench.whole_job_tflops(549.76e9, 2, 10, 10 * 0.4)
    assert abs(one - 1374.4) < 0.1 and abs(two - 2 * one) < 1e-9


def test_reference_arm_runs_on_rank_zero_only():
    class A:
        steps, warmup, cpu_seconds = 1, 0, 0.1
    from tiled_attention_forward_gb300.inputs import WORKLOADS
    assert bench.run_reference(A(), WORKLOADS[0], 2, 1) is None

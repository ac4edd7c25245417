"""The N > 1 path of bench.py on the CPU: two gloo ranks (no GPU).

Every (b, h) is independent, so N GPUs run N independent replicas (weak
scaling, no collective on the data path); the only cross-rank steps are the
barrier and the max over ranks of the timings, and the whole-job value is
N x the per-replica FLOPs over the slowest replica's time."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        mine = [10.0 + rank, 5.0 - rank, 7.0 * (rank + 1), 0.0]
        got = bench.reduce_max_over_ranks(mine, dist, "cpu")
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    want = [11.0, 5.0, 14.0, 0.0]
    assert res[0] == want and res[1] == want


def test_single_rank_reduce_is_identity():
    assert bench.reduce_max_over_ranks([1.5, 2.5], None, "cpu") == [1.5, 2.5]


def test_job_throughput_is_weak_scaling():
    # each replica does 4 TFLOP in 2 ms -> 2000 TFLOP/s per replica
    assert bench.job_tflops(1, 4e12, 2.0) == pytest.approx(2000.0)
    assert bench.job_tflops(8, 4e12, 2.0) == pytest.approx(16000.0)


def test_reference_arm_other_ranks_exit_quietly(capsys):
    w = bench.synth.workload("tiny")
    bench.run_reference(argparse_ns(steps=1, warmup=1), w, w.K(0.2), rank=1)
    assert capsys.readouterr().out == ""


def argparse_ns(**kw):
    import argparse
    return argparse.Namespace(**kw)

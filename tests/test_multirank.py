"""The N > 1 path on the CPU: two gloo ranks (no GPU).

Every (b, h) head is independent, so each rank owns a contiguous range of the
flattened heads (token_sparse_attention_gb300.shard) and keeps its heads'
groups, index sets and residual; nothing crosses ranks on the data path.  The
only cross-rank steps of bench.py are the barrier, the max over ranks of the
timings and the sum of the heads processed.  Here the per-rank compute is the
oracle's (this is a CPU test): head ranges computed on two ranks and gathered
in rank order must equal the whole problem computed in one process."""

import os
import socket

import numpy as np

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from oracle import mcs_oracle as orc
from token_sparse_attention_gb300 import mcs, shard, synth


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


@pytest.mark.parametrize("world,n", [(1, 5), (2, 6), (2, 7), (3, 40), (8, 40), (8, 5), (4, 0)])
def test_head_ranges_cover_every_head_once_in_order(world, n):
    ranges = [shard.head_range(r, world, n) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == n
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0  # contiguous, rank order
    sizes = [b - a for a, b in ranges]
    assert max(sizes) - min(sizes) <= 1 and sum(sizes) == n


def test_head_slices_are_views_and_params_match():
    t = torch.arange(2 * 3 * 5 * 4, dtype=torch.float32).reshape(2, 3, 5, 4)
    v = shard.head_slice(t, 2, 5)  # heads (0,2), (1,0), (1,1)
    assert v.shape == (1, 3, 5, 4) and v.data_ptr() == t[0, 2].data_ptr()
    assert torch.equal(v[0, 1], t[1, 0])
    p = mcs.params(2, 3, 5, 4, 16, 2)
    sp = shard.slice_params(p, 2, 5)
    assert (sp.B, sp.H, sp.N, sp.D, sp.C, sp.K) == (1, 3, 5, 4, 16, 2)
    with pytest.raises(ValueError):
        shard.slice_params(mcs.params(2, 3, 5, 4, 16, 2, layout=mcs.LAYOUT_BNHD), 0, 1)
    with pytest.raises(ValueError):
        shard.slice_params(p, 4, 7)


def test_pddp_launch_count_matches_the_launch_list():
    # the large video workload's grouping launched 55 kernels in the ncu launch
    # list of one call (10 depths x 4, reduce at depths 0-4, block split at
    # depths 0-6, init, node table, finalize); the 3D workload's nodes of 1024
    # rows at depth 6 take the warp split only
    assert bench.pddp_launches(75600, 128) == 55
    assert bench.pddp_launches(65536, 64) == 3 + 40 + 5 + 6
    assert bench.pddp_launches(100, 128) == 2  # one group: no depth, no table


def test_bench_rank_heads_weak_and_strong():
    w = synth.workload("large")
    wg, h0, h1 = bench.rank_heads(w, 0, 1, "weak")
    assert (wg.B, h0, h1) == (1, 0, 40)
    wg, h0, h1 = bench.rank_heads(w, 3, 8, "weak")
    assert (wg.B, h0, h1) == (8, 120, 160)  # every rank a full layer's 40 heads
    wg, h0, h1 = bench.rank_heads(w, 3, 8, "strong")
    assert (wg.B, h0, h1) == (1, 15, 20)


def _anchor_and_reuse(q0, k0, v0, q1, k1, v1, C, K):
    """One head through the oracle: anchor on step-0 inputs, reuse on step 1."""
    scale = orc.default_scale(q0.shape[1])
    a = orc.anchor_step(q0, k0, v0, C, K, scale)
    out = orc.reuse_step(q1, k1, v1, a["perm"], a["idx"], a["residual"], C, scale)
    return np.concatenate([a["perm"].astype(np.float64), a["idx"].ravel().astype(np.float64),
                           a["dense"].ravel(), a["residual"].ravel(), out.ravel()])


def _shard_rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step0, step1 = _problem()
        h0, h1 = shard.head_range(rank, world, step0[0].shape[0] * step0[0].shape[1])
        mine = [_anchor_and_reuse(*(shard.head_slice(t, h0, h1)[0, i].double().numpy()
                                    for t in step0 + step1), C=_C, K=_K)
                for i in range(h1 - h0)]
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        if rank == 0:
            out["heads"] = [h for part in gathered for h in part]
    finally:
        dist.destroy_process_group()


_C, _K = 16, 20


def _problem():
    # B = 2 batches of H = 3 heads: 6 flattened heads over the ranks
    step0 = synth.make_qkv_like(2, 3, 96, 16, seed=5)
    step1 = tuple(t + 0.05 * torch.randn(t.shape, generator=torch.Generator().manual_seed(6 + i))
                  .to(t.dtype) for i, t in enumerate(step0))
    return list(step0), list(step1)


def test_two_gloo_ranks_head_ranges_assemble_the_whole_problem():
    import numpy  # noqa: F401  (spawned ranks import the module again)
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_shard_rank, args=(world, port, out), nprocs=world, join=True)
        got = list(out["heads"])
    step0, step1 = _problem()
    B, H = step0[0].shape[:2]
    assert len(got) == B * H
    for bh in range(B * H):
        b, h = divmod(bh, H)
        want = _anchor_and_reuse(*(t[b, h].double().numpy() for t in step0 + step1), C=_C, K=_K)
        np.testing.assert_array_equal(got[bh], want)

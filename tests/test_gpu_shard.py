"""Head ranges on one GPU: the calls a multi-GPU job makes, one per rank's
contiguous range of flattened heads, run here one after the other, give
bit-identical results to one call over all heads (every (b, h) head is
independent at every step of the path).  Anchor step (grouping, dense + LSE,
exact selection, residual record) and reuse step, through the C ABI."""

import pytest
import torch

from tests import parity as P
from token_sparse_attention_gb300 import build as mcs_build
from token_sparse_attention_gb300 import mcs, shard

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mcs_build.build()
    mcs.lib()
    assert torch.cuda.is_available()


def _buffers(p, q):
    G = p.G
    b = dict(perm=torch.empty(p.B, p.H, G * p.C, dtype=torch.int32, device="cuda"),
             idx=torch.empty(p.B, p.H, G, p.K, dtype=torch.int32, device="cuda"),
             dense=torch.empty_like(q), lse=torch.empty(p.B, p.H, p.N, device="cuda"),
             res=torch.empty_like(q), ret=torch.empty(p.B, p.H, G, device="cuda"),
             out=torch.empty_like(q))
    if mcs.mcs_pair_bytes(p):
        b["pout"] = torch.empty_like(q)
    return b


def _run(p, q0, k0, v0, q1, k1, v1, b):
    ws = mcs.empty_workspace(mcs.mcs_anchor_workspace(p))
    mcs.mcs_anchor_select(p, q0, k0, v0, b["perm"], b["idx"], b["dense"], b["lse"], b["res"],
                          ws, retained=b["ret"])
    mcs.mcs_sparse_attn(p, q1, k1, v1, b["perm"], b["idx"], b["res"], b["out"])
    if "pout" in b:  # C = 64: each rank builds its heads' sibling-pair lists
        pairs = mcs.empty_pairs(p)
        mcs.mcs_pair_lists(p, b["idx"], pairs)
        mcs.mcs_sparse_attn_pairs(p, q1, k1, v1, b["perm"], pairs, b["res"], b["pout"])


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("B,H,N,D,C,K", [(2, 3, 700, 128, 128, 150), (1, 5, 1000, 64, 64, 333)])
def test_head_ranges_equal_one_call(world, B, H, N, D, C, K):
    step0 = [t.cuda() for t in P.random_qkv(B, H, N, D, seed=N + world)]
    step1 = [t.cuda() for t in P.random_qkv(B, H, N, D, seed=N + world + 1)]
    p = mcs.params(B, H, N, D, C, K)
    whole = _buffers(p, step0[0])
    _run(p, *step0, *step1, whole)
    parts = _buffers(p, step0[0])
    for r in range(world):
        h0, h1 = shard.head_range(r, world, B * H)
        sp = shard.slice_params(p, h0, h1)
        views = {n: shard.head_slice(t, h0, h1) for n, t in parts.items()}
        _run(sp, *(shard.head_slice(t, h0, h1) for t in step0 + step1), views)
    assert mcs.mcs_device_status() == 0
    for n in whole:
        assert torch.equal(whole[n], parts[n]), f"{n} differs between head ranges and one call"

"""GPU parity of the diagnostic selectors and error measures (mcs_block_topk,
mcs_pooled_block_select, mcs_gather_mass, mcs_rel_l1, and the per-query oracle
as one-query groups) against the fp64 oracle.  Every call goes through the C
ABI (libmcs.so)."""

import numpy as np
import pytest
import torch

from oracle import mcs_oracle as orc
from tests import parity as P
from token_sparse_attention_gb300 import build as mcs_build
from token_sparse_attention_gb300 import mcs
from token_sparse_attention_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mcs_build.build()
    mcs.lib()
    assert torch.cuda.is_available()
    yield
    assert mcs.mcs_device_status() == 0


def _blocks(idx, block):
    idx = np.asarray(idx)
    b = idx.reshape(-1, block)
    assert np.all(b == b[:, :1] + np.arange(block)), "kept tokens are not whole blocks"
    return b[:, 0] // block


def _assert_block_sets_within_ties(got_idx, want_idx, block, score, rel):
    # both sides keep whole blocks, ascending; a block may differ only when
    # its score is within `rel` of the last kept block's score (the fp32 and
    # fp64 rankings can order near-equal blocks differently)
    g, w = set(_blocks(got_idx, block)), set(_blocks(want_idx, block))
    assert np.all(np.diff(np.asarray(got_idx)) > 0)
    if g == w:
        return
    kth = min(score[b] for b in w)
    tol = rel * max(abs(kth), 1e-30)
    for b in g ^ w:
        assert abs(score[b] - kth) <= tol, (b, score[b], kth)


@pytest.mark.parametrize("N,block,K", [(1000, 64, 256), (1001, 64, 960), (517, 16, 32),
                                       (300, 1, 37)])
def test_block_topk_matches_oracle(N, block, K):
    rows = 4  # <= the B*H*G = ceil(N / 64) group rows the parameters describe
    rng = np.random.default_rng(N + block)
    mass = rng.random((rows, N)).astype(np.float32) ** 4   # spread out, no exact ties
    p = mcs.params(1, 1, N, 128, 64, K)
    d_mass = torch.from_numpy(mass).cuda()
    idx = torch.empty(rows, K, dtype=torch.int32, device="cuda")
    ret = torch.empty(rows, dtype=torch.float32, device="cuda")
    ws = mcs.empty_workspace(mcs.mcs_block_workspace(p, block))
    mcs.mcs_block_topk(p, d_mass, block, idx, ws, retained=ret)
    assert mcs.mcs_device_status() == 0
    nb = N // block
    for r in range(rows):
        want, want_ret = orc.block_topk_select(mass[r], K, block)
        bm = mass[r][:nb * block].astype(np.float64).reshape(nb, block).sum(axis=1)
        _assert_block_sets_within_ties(idx[r].cpu().numpy(), want, block, bm, 1e-5)
        assert float(ret[r]) == pytest.approx(want_ret, rel=1e-5)
        assert idx[r].max().item() < nb * block


@pytest.mark.parametrize("N,D,C,block,K", [(1000, 64, 64, 64, 256), (1500, 128, 128, 128, 512),
                                           (777, 128, 64, 32, 96)])
def test_pooled_block_select_matches_oracle(N, D, C, block, K):
    H = 2
    q, k, _ = P.random_qkv(1, H, N, D, seed=N + D)
    p = mcs.params(1, H, N, D, C, K)
    qd, kd = q.cuda(), k.cuda()
    perm = torch.empty(1, H, p.G * C, dtype=torch.int32, device="cuda")
    mcs.mcs_group(p, qd, perm, mcs.empty_workspace(mcs.mcs_group_workspace(p)))
    idx = torch.empty(1, H, p.G, K, dtype=torch.int32, device="cuda")
    ws = mcs.empty_workspace(mcs.mcs_block_workspace(p, block))
    mcs.mcs_pooled_block_select(p, qd, kd, perm, block, idx, ws)
    assert mcs.mcs_device_status() == 0
    scale = orc.default_scale(D)
    for h in range(H):
        pm = perm[0, h].cpu().numpy()
        for g in range(p.G):
            members = orc.group_members(pm, g, C)
            want, score = orc.pooled_block_select(P.f64(q[0, h]), P.f64(k[0, h]), members, K,
                                                  block, scale)
            _assert_block_sets_within_ties(idx[0, h, g].cpu().numpy(), want, block, score, 1e-4)


def test_gather_mass_matches_oracle():
    rows, N, K = 5, 3001, 700
    rng = np.random.default_rng(7)
    mass = rng.random((rows, N)).astype(np.float32)
    sel = np.stack([np.sort(rng.choice(N, K, replace=False)) for _ in range(rows)])
    p = mcs.params(1, 1, N, 128, 64, K)
    ret = torch.empty(rows, dtype=torch.float32, device="cuda")
    mcs.mcs_gather_mass(p, torch.from_numpy(mass).cuda(),
                        torch.from_numpy(sel.astype(np.int32)).cuda(), ret)
    for r in range(rows):
        assert float(ret[r]) == pytest.approx(orc.retained_mass(mass[r], sel[r]), rel=1e-5)


def test_rel_l1_matches_oracle_all_rows_and_subset():
    B, H, N, D = 1, 3, 500, 64
    g = torch.Generator().manual_seed(9)
    want = torch.randn(B, H, N, D, generator=g).to(torch.bfloat16)
    got = (want.float() + 0.05 * torch.randn(B, H, N, D, generator=g)).to(torch.bfloat16)
    p = mcs.params(B, H, N, D, 64, 1)
    e, w = mcs.mcs_rel_l1(p, got.cuda(), want.cuda())
    assert e / w == pytest.approx(orc.rel_l1(P.f64(got), P.f64(want)), rel=1e-9)
    rows = np.array([0, 7, 499, 500, 1499], dtype=np.int32)   # flat (b*H + h)*N + token rows
    e, w = mcs.mcs_rel_l1(p, got.cuda(), want.cuda(), torch.from_numpy(rows).cuda())
    flat_g, flat_w = P.f64(got).reshape(-1, D), P.f64(want).reshape(-1, D)
    assert e / w == pytest.approx(orc.rel_l1(flat_g[rows], flat_w[rows]), rel=1e-9)


def _one_query_groups(N, C, G, rows):
    """perm with query rows[g] alone in group g (the rest of every group, and
    groups past len(rows), padding)."""
    perm = np.full(G * C, -1, dtype=np.int32)
    perm[np.arange(len(rows)) * C] = rows
    return perm


def test_per_query_oracle_as_one_query_groups():
    N, D, C, K = 2000, 128, 128, 300
    q, k, v = P.random_qkv(1, 1, N, D, seed=31)
    p = mcs.params(1, 1, N, D, C, K)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    lse = torch.empty(1, 1, N, dtype=torch.float32, device="cuda")
    mcs.mcs_dense_attn(p, qd, kd, vd, torch.empty_like(qd), lse)
    rows = np.array([0, 5, 999, 1998, 1999, 1234, 17], dtype=np.int32)
    perm = torch.from_numpy(_one_query_groups(N, C, p.G, rows)).view(1, 1, -1).cuda()
    mass = torch.empty(1, p.G, N, dtype=torch.float32, device="cuda")
    mcs.mcs_group_mass(p, qd, kd, lse, perm, 0, 1, mass)
    idx = torch.empty(p.G, K, dtype=torch.int32, device="cuda")
    ret = torch.empty(p.G, dtype=torch.float32, device="cuda")
    mcs.mcs_topk(p, mass, idx, ret)
    assert mcs.mcs_device_status() == 0
    scale = orc.default_scale(D)
    _, lse64 = orc.dense_attention(P.f64(q[0, 0]), P.f64(k[0, 0]), P.f64(v[0, 0]), scale)
    for g, row in enumerate(rows):
        want, want_ret = orc.per_query_select(P.f64(q[0, 0]), P.f64(k[0, 0]), lse64, int(row), K,
                                              scale)
        prob = np.exp(scale * (P.f64(k[0, 0]) @ P.f64(q[0, 0])[row]) - lse64[row])
        P.assert_topk_within_ties(idx[g].cpu().numpy(), want, prob, K)
        assert float(ret[g]) == pytest.approx(want_ret, rel=1e-4)


def test_selector_recall_ordering_on_workload():
    # at the same number of kept tokens, on the small video workload (one
    # head): pooled blocks <= block oracle <= token oracle (group recall)
    w = synth.workload("small")
    block = 128
    K = 6528  # 51 blocks of 128, density ~0.2
    q, k, v = [t.cuda() for t in synth.make_qkv(w, 0, heads=[0])]
    p = mcs.params(1, 1, w.N, w.D, w.C, K)
    perm = torch.empty(1, 1, p.G * w.C, dtype=torch.int32, device="cuda")
    mcs.mcs_group(p, q, perm, mcs.empty_workspace(mcs.mcs_group_workspace(p)))
    lse = torch.empty(1, 1, w.N, dtype=torch.float32, device="cuda")
    mcs.mcs_dense_attn(p, q, k, v, torch.empty_like(q), lse)
    mass = torch.empty(1, p.G, w.N, dtype=torch.float32, device="cuda")
    mcs.mcs_group_mass(p, q, k, lse, perm, 0, 1, mass)
    ws = mcs.empty_workspace(mcs.mcs_block_workspace(p, block))
    tok_idx = torch.empty(p.G, K, dtype=torch.int32, device="cuda")
    tok = torch.empty(p.G, dtype=torch.float32, device="cuda")
    mcs.mcs_topk(p, mass, tok_idx, tok)
    blk_idx = torch.empty(p.G, K, dtype=torch.int32, device="cuda")
    blk = torch.empty(p.G, dtype=torch.float32, device="cuda")
    mcs.mcs_block_topk(p, mass, block, blk_idx, ws, retained=blk)
    pool_idx = torch.empty(1, 1, p.G, K, dtype=torch.int32, device="cuda")
    mcs.mcs_pooled_block_select(p, q, k, perm, block, pool_idx, ws)
    pool = torch.empty(p.G, dtype=torch.float32, device="cuda")
    mcs.mcs_gather_mass(p, mass, pool_idx, pool)
    assert mcs.mcs_device_status() == 0
    slack = 1e-5 * w.C
    assert torch.all(pool <= blk + slack) and torch.all(blk <= tok + slack)
    assert float(pool.sum()) < float(blk.sum()) < float(tok.sum())

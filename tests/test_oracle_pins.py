"""Pins of the fp64 oracle against things other than itself.

Each test ties one oracle function to a textbook or library routine, a closed
form, a hand-worked fixture (tests/golden), brute force or an invariant the
method fixes, chosen so that a plausible slip (a dropped term, a wrong sign or
index, a transposed operand) fails at least one of them.  CPU only.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import mcs_oracle as orc
from tests.parity import separated_clusters

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


def _bf16(a):
    return orc.round_to_bf16(a)


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_rounding_matches_torch():
    rng = _rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-30).astype(np.float32),
        (rng.standard_normal(2000) * 1e4).astype(np.float32),
        # exact half-way cases: bf16 value + half an ulp, both parities
        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(2.0 + 2.0 ** -7), 0.0], np.float32),
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(orc.round_to_bf16(x.astype(np.float64)), want)


# ---------------------------------------------------------------- dense + LSE

@pytest.mark.parametrize("N,D", [(37, 16), (128, 64), (200, 128)])
def test_dense_matches_torch_sdpa(N, D):
    rng = _rng(N)
    q, k, v = (_bf16(rng.standard_normal((N, D)) * s) for s in (2.0, 1.0, 1.0))
    scale = orc.default_scale(D)
    O, lse = orc.dense_attention(q, k, v, scale)
    tq, tk, tv = (torch.from_numpy(a)[None, None] for a in (q, k, v))
    want = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)[0, 0]
    np.testing.assert_allclose(O, want.numpy(), rtol=1e-10, atol=1e-12)
    S = torch.from_numpy(q) @ torch.from_numpy(k).T * scale
    np.testing.assert_allclose(lse, torch.logsumexp(S, dim=1).numpy(), rtol=1e-12)


def test_dense_lse_bounds_and_rows_sum_to_one():
    rng = _rng(3)
    N, D = 150, 32
    q, k, v = (rng.standard_normal((N, D)) for _ in range(3))
    scale = 0.7
    _, lse = orc.dense_attention(q, k, v, scale)
    S = scale * q @ k.T
    assert np.all(lse >= S.max(1) - 1e-12)
    assert np.all(lse <= S.max(1) + math.log(N) + 1e-12)
    np.testing.assert_allclose(np.exp(S - lse[:, None]).sum(1), 1.0, rtol=1e-12)


def test_dense_closed_form_identical_keys():
    # every key equal -> every score in a row equal -> uniform weights:
    # O_i = mean of V rows, lse_i = s_i + log N
    rng = _rng(4)
    N, D = 64, 16
    q = rng.standard_normal((N, D))
    k = np.tile(rng.standard_normal(D), (N, 1))
    v = rng.standard_normal((N, D))
    O, lse = orc.dense_attention(q, k, v, 0.5)
    np.testing.assert_allclose(O, np.tile(v.mean(0), (N, 1)), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, 0.5 * q @ k[0] + math.log(N), rtol=1e-12)


def test_dense_rows_subset_equals_full():
    rng = _rng(5)
    q, k, v = (rng.standard_normal((90, 8)) for _ in range(3))
    O, lse = orc.dense_attention(q, k, v, 0.3)
    rows = np.array([0, 17, 89])
    O2, lse2 = orc.dense_attention(q, k, v, 0.3, rows=rows)
    np.testing.assert_array_equal(O2, O[rows])
    np.testing.assert_array_equal(lse2, lse[rows])


# ---------------------------------------------------------------- power iteration

def test_principal_direction_matches_eigh():
    rng = _rng(6)
    D = 24
    Q, _ = np.linalg.qr(rng.standard_normal((D, D)))
    evals = np.concatenate([[20.0, 6.0], rng.uniform(0.1, 5.0, D - 2)])
    cov = (Q * evals) @ Q.T
    v = orc.principal_direction(cov, 64)
    w, U = np.linalg.eigh(cov)
    u = U[:, -1]
    lead = int(np.argmax(np.abs(u)))
    u = u if u[lead] > 0 else -u
    np.testing.assert_allclose(v, u, atol=1e-8)
    assert v[np.argmax(np.abs(v))] > 0


def test_principal_direction_sign_rule_and_degenerate():
    # rank one along u whose largest component is negative -> result is -u/|u|
    u = np.array([0.1, -3.0, 0.5, 1.0])
    v = orc.principal_direction(np.outer(u, u), 5)
    np.testing.assert_allclose(v, -u / np.linalg.norm(u), atol=1e-14)
    # zero covariance: the start vector is kept
    v0 = orc.principal_direction(np.zeros((4, 4)), 5)
    np.testing.assert_allclose(v0, np.full(4, 0.5))


# ---------------------------------------------------------------- PDDP

def _check_valid_perm(perm, N, C):
    G = -(-N // C)
    assert perm.shape == (G * C,)
    real = perm[perm >= 0]
    assert np.array_equal(np.sort(real), np.arange(N))
    for g in range(G):
        seg = perm[g * C:(g + 1) * C]
        n_real = int((seg >= 0).sum())
        assert n_real == (C if g < G - 1 else N - (G - 1) * C)
        assert np.all(seg[:n_real] >= 0) and np.all(seg[n_real:] == -1)
        assert np.all(np.diff(seg[:n_real]) > 0)


def test_pddp_golden_four_pairs():
    fx = json.load(open(os.path.join(GOLDEN, "pddp_four_pairs.json")))
    x = np.array(fx["points"])
    perm = orc.pddp_perm(x, fx["C"], 32)
    assert perm.tolist() == fx["expected_perm"]


@pytest.mark.parametrize("N,C", [(256, 32), (300, 32), (1000, 64), (97, 16)])
def test_pddp_on_a_line_is_sorting(N, C):
    # x_i = t_i * u: every node's covariance has rank one along u, so each split
    # orders by t (u's largest component is positive) and the leaves are
    # consecutive C-chunks of the order by (t, index).
    rng = _rng(N + C)
    D = 8
    u = rng.standard_normal(D)
    u[np.argmax(np.abs(u))] = abs(u[np.argmax(np.abs(u))]) + 1.0
    t = rng.standard_normal(N)
    t[::7] = t[3]  # some exact ties, broken by token index
    x = np.outer(t, u)
    perm = orc.pddp_perm(x, C, 32)
    order = np.lexsort((np.arange(N), t))
    G = -(-N // C)
    want = np.full(G * C, -1)
    for g in range(G):
        chunk = np.sort(order[g * C:(g + 1) * C])
        want[g * C:g * C + chunk.shape[0]] = chunk
    np.testing.assert_array_equal(perm, want)


@pytest.mark.parametrize("N,C,D", [(512, 64, 16), (2048, 64, 128), (1000, 128, 64), (3000, 128, 128)])
def test_pddp_recovers_separated_clusters(N, C, D):
    x, want = separated_clusters(N, C, D, seed=N + D)
    np.testing.assert_array_equal(orc.pddp_perm(x, C, 32), want)


def test_pddp_valid_and_translation_invariant():
    rng = _rng(8)
    N, C, D = 777, 32, 12
    x = rng.standard_normal((N, D)) * rng.uniform(0.5, 2.0, D)
    perm = orc.pddp_perm(x, C, 32)
    _check_valid_perm(perm, N, C)
    # centring: shifting every point by the same vector changes nothing
    shifted = orc.pddp_perm(x + 50.0 * rng.standard_normal(D), C, 32)
    np.testing.assert_array_equal(perm, shifted)


# ---------------------------------------------------------------- group mass, top-K

def _head(N, D, seed, qs=2.0):
    rng = _rng(seed)
    q, k, v = (_bf16(rng.standard_normal((N, D)) * s) for s in (qs, 1.0, 1.0))
    return q, k, v


def test_group_mass_matches_torch_softmax_and_sums_to_group_size():
    N, D = 300, 32
    q, k, _ = _head(N, D, 9)
    scale = orc.default_scale(D)
    _, lse = orc.dense_attention(q, k, k, scale)
    members = np.array([3, 50, 51, 199, 299])
    mass = orc.group_mass(q, k, lse, members, scale)
    P = torch.softmax(torch.from_numpy(q @ k.T * scale), dim=1).numpy()
    np.testing.assert_allclose(mass, P[members].sum(0), rtol=1e-11, atol=1e-15)
    assert math.isclose(mass.sum(), members.shape[0], rel_tol=1e-12)


def test_group_mass_several_groups_of_one_perm():
    """Every group of one grouping against torch's softmax rows summed over
    that group's own members (a group read through another group's rows, or
    through the wrong perm slots, fails), and the groups together account for
    every query: summed over all groups the masses are the column sums of the
    full probability matrix."""
    N, D, C = 230, 16, 32  # 8 groups, the last one short (6 rows)
    q, k, _ = _head(N, D, 21)
    scale = orc.default_scale(D)
    _, lse = orc.dense_attention(q, k, k, scale)
    perm = orc.pddp_perm(q, C, 32)
    G = -(-N // C)
    P = torch.softmax(torch.from_numpy(q @ k.T * scale), dim=1).numpy()
    total = np.zeros(N)
    for g in range(G):
        members = orc.group_members(perm, g, C)
        assert members.shape[0] == (C if g < G - 1 else N - (G - 1) * C)
        mass = orc.group_mass(q, k, lse, members, scale)
        np.testing.assert_allclose(mass, P[members].sum(0), rtol=1e-11, atol=1e-15)
        total += mass
    np.testing.assert_allclose(total, P.sum(0), rtol=1e-11, atol=1e-14)
    assert math.isclose(total.sum(), N, rel_tol=1e-12)


def test_topk_golden_ties():
    fx = json.load(open(os.path.join(GOLDEN, "topk_ties.json")))
    for case in fx["cases"]:
        idx, kept = orc.topk_select(np.array(fx["mass"]), case["K"])
        assert idx.tolist() == case["idx"]
        assert math.isclose(kept, sum(fx["mass"][i] for i in case["idx"]))


@pytest.mark.parametrize("n,K", [(8, 3), (12, 5), (10, 1), (9, 9)])
def test_topk_brute_force(n, K):
    mass = _rng(n * 10 + K).uniform(0, 1, n)
    best = max(itertools.combinations(range(n), K), key=lambda s: sum(mass[list(s)]))
    idx, kept = orc.topk_select(mass, K)
    assert idx.tolist() == list(best)
    assert math.isclose(kept, mass[list(best)].sum(), rel_tol=1e-14)


def test_retained_mass_bounds():
    N, D, C, K = 512, 32, 32, 60
    q, k, _ = _head(N, D, 10)
    scale = orc.default_scale(D)
    _, lse = orc.dense_attention(q, k, k, scale)
    perm = orc.pddp_perm(q, C, 32)
    rng = _rng(11)
    for g in (0, 5, 15):
        members = orc.group_members(perm, g, C)
        mass = orc.group_mass(q, k, lse, members, scale)
        idx, kept = orc.topk_select(mass, K)
        # the per-query oracle is an upper bound for any shared selection
        bound = orc.per_query_topk_mass(q, k, lse, members, K, scale).sum()
        assert kept <= bound + 1e-12
        # and the chosen set beats random sets of the same size
        for _ in range(50):
            other = rng.choice(N, size=K, replace=False)
            assert kept >= mass[other].sum() - 1e-12


# ---------------------------------------------------------------- sparse + residual

def test_sparse_full_density_equals_dense():
    N, D, C = 200, 32, 32
    q, k, v = _head(N, D, 12)
    scale = orc.default_scale(D)
    perm = orc.pddp_perm(q, C, 32)
    G = -(-N // C)
    idx = np.tile(np.arange(N), (G, 1))
    sparse = orc.sparse_attention(q, k, v, perm, idx, C, scale)
    dense, _ = orc.dense_attention(q, k, v, scale)
    np.testing.assert_allclose(sparse, dense, rtol=1e-11, atol=1e-13)


def test_sparse_fixed_subset_equals_sdpa_on_subset():
    N, D, C, K = 160, 16, 16, 23
    q, k, v = _head(N, D, 13)
    scale = orc.default_scale(D)
    rng = _rng(14)
    perm = np.concatenate([rng.permutation(N), np.full((-(-N // C)) * C - N, -1)])
    perm = perm.reshape(-1, C)
    perm = np.stack([np.concatenate([np.sort(r[r >= 0]), r[r < 0]]) for r in perm]).reshape(-1)
    sub = np.sort(rng.choice(N, K, replace=False))
    idx = np.tile(sub, (-(-N // C), 1))
    sparse = orc.sparse_attention(q, k, v, perm, idx, C, scale)
    want = torch.nn.functional.scaled_dot_product_attention(
        *(torch.from_numpy(a)[None, None] for a in (q, k[sub], v[sub])), scale=scale)[0, 0]
    np.testing.assert_allclose(sparse, want.numpy(), rtol=1e-10, atol=1e-12)


def test_sparse_distinct_idx_per_group_equals_sdpa_per_group():
    """Each group attends to its OWN selected keys: with a different index set
    per group, every group's rows equal torch SDPA of those queries over that
    group's K/V subset, written back at the group's own token rows.  Reading
    idx[0] for every group, mixing up group and row, or scattering to perm
    positions instead of token indices fails here."""
    N, D, C, K = 150, 16, 32, 19  # 5 groups, the last one short (22 rows)
    q, k, v = _head(N, D, 22)
    scale = orc.default_scale(D)
    rng = _rng(23)
    G = -(-N // C)
    perm = np.full(G * C, -1, dtype=np.int64)
    order = rng.permutation(N)
    for g in range(G):
        seg = np.sort(order[g * C:(g + 1) * C])
        perm[g * C:g * C + seg.shape[0]] = seg
    idx = np.stack([np.sort(rng.choice(N, K, replace=False)) for _ in range(G)])
    assert len({tuple(r) for r in idx}) == G  # the sets really differ
    sparse = orc.sparse_attention(q, k, v, perm, idx, C, scale)
    assert not np.any(np.isnan(sparse))
    for g in range(G):
        rows = perm[g * C:(g + 1) * C]
        rows = rows[rows >= 0]
        want = torch.nn.functional.scaled_dot_product_attention(
            *(torch.from_numpy(a)[None, None] for a in (q[rows], k[idx[g]], v[idx[g]])),
            scale=scale)[0, 0]
        np.testing.assert_allclose(sparse[rows], want.numpy(), rtol=1e-10, atol=1e-12)
    # the same groups processed one at a time agree with the whole-head call
    for g in (0, G - 1):
        rows = orc.group_members(perm, g, C)
        np.testing.assert_array_equal(
            orc.sparse_attention_group(q, k, v, rows, idx[g], scale), sparse[rows])


def test_anchor_identity_and_reuse_reproduces_dense():
    N, D, C, K = 256, 32, 32, 40
    q, k, v = _head(N, D, 15)
    scale = orc.default_scale(D)
    a = orc.anchor_step(q, k, v, C, K, scale)
    _check_valid_perm(a["perm"], N, C)
    # the residual is stored in bf16: sparse + R equals the stored dense output
    # up to half a bf16 spacing of R
    half_ulp_r = np.ldexp(1.0, np.frexp(a["residual"])[1] - 9)
    assert np.all(np.abs(a["sparse"] + a["residual"] - a["dense_bf16"]) <= half_ulp_r + 1e-15)
    # reuse with unchanged inputs gives the dense output back
    out = orc.reuse_step(q, k, v, a["perm"], a["idx"], a["residual"], C, scale)
    assert np.max(np.abs(out - a["dense"])) < 1e-2
    assert np.max(np.abs(orc.round_to_bf16(out) - a["dense_bf16"])) <= np.max(np.abs(a["dense"])) * 2 ** -7
    # restricted to some groups, the reuse step gives exactly those groups' rows
    part = orc.reuse_step(q, k, v, a["perm"], a["idx"], a["residual"], C, scale, groups=[1, 6])
    rows = np.concatenate([orc.group_members(a["perm"], g, C) for g in (1, 6)])
    np.testing.assert_array_equal(part[rows], out[rows])
    others = np.setdiff1d(np.arange(N), rows)
    assert np.all(np.isnan(part[others]))
    # the selection keeps most of the mass on these peaked inputs, never more than
    # the group size
    sizes = np.array([orc.group_members(a["perm"], g, C).shape[0] for g in range(a["idx"].shape[0])])
    assert np.all(a["retained"] <= sizes + 1e-9)
    np.testing.assert_allclose(a["mass"].sum(1), sizes, rtol=1e-12)


# ---------------------------------------------------------------- diagnostic selectors

def test_block_select_with_unit_blocks_is_token_topk():
    m = _rng(40).random(37)
    for K in (1, 5, 37):
        i1, r1 = orc.block_topk_select(m, K, 1)
        i2, r2 = orc.topk_select(m, K)
        np.testing.assert_array_equal(i1, i2)
        assert r1 == pytest.approx(r2, rel=1e-15)


@pytest.mark.parametrize("N,block,kb", [(12, 2, 2), (13, 3, 2), (16, 4, 3)])
def test_block_select_brute_force(N, block, kb):
    # the chosen blocks maximise the kept mass over every set of kb full
    # blocks; the partial tail block (13 = 4*3 + 1) is never chosen
    m = _rng(41 + N).random(N)
    idx, ret = orc.block_topk_select(m, kb * block, block)
    nb = N // block
    best = max(itertools.combinations(range(nb), kb),
               key=lambda bs: sum(m[b * block:(b + 1) * block].sum() for b in bs))
    want = np.concatenate([np.arange(b * block, (b + 1) * block) for b in best])
    np.testing.assert_array_equal(idx, want)
    assert ret == pytest.approx(m[want].sum(), rel=1e-14)
    assert idx.max() < nb * block


def test_block_select_rejects_budget_not_in_blocks():
    with pytest.raises(ValueError):
        orc.block_topk_select(np.ones(10), 3, 2)
    with pytest.raises(ValueError):
        orc.block_topk_select(np.ones(10), 12, 2)


def test_pooled_block_select_hand_example():
    # two KV blocks of two keys; the mean query (1, 1) scores block 0
    # (mean key (1, 0)) at 1 and block 1 (mean key (0.5, 1.5)) at 2
    q = np.array([[2.0, 0.0], [0.0, 2.0]])
    k = np.array([[1.0, 1.0], [1.0, -1.0], [0.0, 1.0], [1.0, 2.0]])
    idx, score = orc.pooled_block_select(q, k, [0, 1], 2, 2, scale=1.0)
    np.testing.assert_allclose(score, [1.0, 2.0])
    np.testing.assert_array_equal(idx, [2, 3])


def test_pooled_block_select_single_query_unit_blocks_is_per_query_oracle():
    # one query, blocks of one key: the pooled score is the query's own
    # score, whose order is its probability order
    rng = _rng(43)
    q = _bf16(rng.standard_normal((5, 16)))
    k = _bf16(rng.standard_normal((40, 16)))
    scale = orc.default_scale(16)
    _, lse = orc.dense_attention(q, k, k, scale)
    for row in range(5):
        idx, _ = orc.pooled_block_select(q, k, [row], 9, 1, scale)
        want, _ = orc.per_query_select(q, k, lse, row, 9, scale)
        np.testing.assert_array_equal(idx, want)


def test_per_query_select_matches_per_query_topk_mass_and_sdpa_probabilities():
    rng = _rng(44)
    q = _bf16(rng.standard_normal((6, 32)))
    k = _bf16(rng.standard_normal((50, 32)))
    scale = orc.default_scale(32)
    _, lse = orc.dense_attention(q, k, k, scale)
    P = torch.softmax(torch.from_numpy(q) @ torch.from_numpy(k).T * scale, dim=-1).numpy()
    masses = orc.per_query_topk_mass(q, k, lse, np.arange(6), 12, scale)
    for row in range(6):
        idx, ret = orc.per_query_select(q, k, lse, row, 12, scale)
        want = np.sort(np.argsort(-P[row], kind="stable")[:12])
        np.testing.assert_array_equal(idx, want)
        assert ret == pytest.approx(masses[row], rel=1e-12)


def test_recall_ordering_per_query_token_block():
    # at the same number of kept tokens: the per-query optimum keeps at least
    # what the group's token optimum keeps (summed over the group), which
    # keeps at least what the best whole blocks keep; all reach the group
    # size when every token is kept
    rng = _rng(45)
    N, D, C, block = 64, 16, 8, 4
    q = _bf16(rng.standard_normal((N, D)))
    k = _bf16(rng.standard_normal((N, D)))
    scale = orc.default_scale(D)
    _, lse = orc.dense_attention(q, k, k, scale)
    members = np.arange(8, 16)
    mass = orc.group_mass(q, k, lse, members, scale)
    for K in (8, 16, 32, 64):
        pq = orc.per_query_topk_mass(q, k, lse, members, K, scale).sum()
        _, tok = orc.topk_select(mass, K)
        _, blk = orc.block_topk_select(mass, K, block)
        pidx, _ = orc.pooled_block_select(q, k, members, K, block, scale)
        pooled = orc.retained_mass(mass, pidx)
        assert pq >= tok - 1e-12 >= blk - 2e-12 >= pooled - 3e-12
    assert tok == pytest.approx(C, rel=1e-12) and blk == pytest.approx(C, rel=1e-12)


def test_rel_l1_closed_forms():
    w = _rng(46).standard_normal((7, 3))
    assert orc.rel_l1(w, w) == 0.0
    assert orc.rel_l1(2 * w, w) == pytest.approx(1.0)
    assert orc.rel_l1(np.zeros_like(w), w) == pytest.approx(1.0)
    assert orc.rel_l1(w + 0.5, w) == pytest.approx(0.5 * w.size / np.abs(w).sum())


# ---------------------------------------------------------------- E4M3 K/V cache

def _torch_e4m3(x):
    """torch's float32 -> float8_e4m3fn conversion (round to nearest even)."""
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_decode(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.isnan(got).sum() == 2                      # S.1111.111 only
    fin = ~np.isnan(got)
    assert np.array_equal(got[fin], want[fin])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6
    assert got[0x38] == 1.0 and got[0xB8] == -1.0


def test_e4m3_encode_matches_torch_rounding_including_ties():
    table = orc.e4m3_decode(np.arange(0x7F, dtype=np.uint8))   # 0 .. 448, ascending
    assert np.all(np.diff(table) > 0)
    mids = (table[:-1] + table[1:]) / 2                        # exact ties (float32)
    rng = _rng(60)
    x = np.concatenate([
        table, -table, mids, -mids,
        rng.standard_normal(20000) * 20.0,
        rng.standard_normal(5000) * 0.01,
        np.ldexp(rng.uniform(0.5, 1.0, 5000), rng.integers(-14, 9, 5000)),
    ]).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    assert np.array_equal(orc.e4m3_encode(x, 1.0), _torch_e4m3(x))
    # ties go to the even mantissa: 1 + 1/16 -> 1.0, 1 + 3/16 -> 1.25
    assert list(orc.e4m3_encode(np.array([1.0625, 1.1875], np.float32), 1.0)) == [0x38, 0x3A]


def test_e4m3_encode_saturates_and_keeps_signs():
    x = np.array([448.0, 449.0, 464.0, 479.0, 480.0, 1e6, -500.0, -1e30], np.float32)
    assert list(orc.e4m3_encode(x, 1.0)) == [0x7E] * 6 + [0xFE] * 2
    z = orc.e4m3_encode(np.array([0.0, -0.0, 2.0 ** -11, -2.0 ** -11, np.nan], np.float32), 1.0)
    assert list(z) == [0x00, 0x80, 0x00, 0x80, 0x7F]
    # the smallest subnormal and half of it (a tie between 0 and 2**-9: to even, 0)
    assert list(orc.e4m3_encode(np.array([2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10], np.float32),
                                1.0)) == [0x01, 0x00, 0x02]


def test_e4m3_round_trip_and_scale():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF, 0x80)], np.uint8)
    vals = orc.e4m3_decode(codes)
    assert np.array_equal(orc.e4m3_encode(vals.astype(np.float32), 1.0), codes)
    # a power-of-two scale moves every finite value exactly: x = s * v encodes to v's code
    for s in (0.125, 4.0):
        inner = codes[np.abs(vals) * max(s, 1.0) <= 448.0]
        v = orc.e4m3_decode(inner)
        assert np.array_equal(orc.e4m3_encode((s * v).astype(np.float32), s), inner)
    # the quotient is a float32 division: 1/3 of 3 in float32 is exactly 1
    assert orc.e4m3_encode(np.array([3.0], np.float32), 3.0)[0] == 0x38


def test_sparse_attention_e4m3_is_sparse_attention_of_the_decoded_cache():
    rng = _rng(61)
    N, D, C, K = 96, 16, 32, 24
    q = _bf16(rng.standard_normal((N, D)))
    # K/V that are exactly k_scale/v_scale times E4M3 values decode to themselves
    k8 = rng.integers(0, 0x7E, (N, D)).astype(np.uint8) | (rng.integers(0, 2, (N, D)) << 7).astype(np.uint8)
    v8 = rng.integers(0x20, 0x50, (N, D)).astype(np.uint8)
    ks, vs = 0.0078125, 0.5
    k = ks * orc.e4m3_decode(k8)
    v = vs * orc.e4m3_decode(v8)
    perm = np.arange(N)
    idx = np.stack([np.sort(rng.choice(N, K, replace=False)) for _ in range(N // C)])
    scale = orc.default_scale(D)
    got = orc.sparse_attention_e4m3(q, k8, v8, ks, vs, perm, idx, C, scale)
    want = orc.sparse_attention(q, k, v, perm, idx, C, scale)
    assert np.array_equal(got, want)
    # and the encoder recovers those bytes from the values
    assert np.array_equal(orc.e4m3_encode(k.astype(np.float32), ks), k8)
    # per group: softmax over the group's own selected rows (SDPA on the subset)
    for g in range(N // C):
        rows = perm[g * C:(g + 1) * C]
        t = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[rows])[None], torch.from_numpy(k[idx[g]])[None],
            torch.from_numpy(v[idx[g]])[None], scale=scale)[0].numpy()
        assert np.allclose(got[rows], t, rtol=1e-10, atol=1e-12)

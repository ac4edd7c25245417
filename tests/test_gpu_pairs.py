"""Sibling-pair key lists for C = 64 groups, through the C ABI.

mcs_pair_lists turns the index sets of groups 2u and 2u+1 into their
ascending union with each key's group membership; mcs_sparse_attn_pairs runs
both groups as one 128-row tile over that union, each row restricted (by a
mask step on the tensor core) to its own group's keys.  The lists are checked
entry by entry against Python set logic; the attention against the fp64
oracle's token-sparse attention of each group over its own K keys (the same
tolerances as the unpaired kernel), with ragged tails, an odd number of
groups, K = 1, K = N, heavily and barely overlapping siblings, both head
dims, the residual add and the anchor record.
"""

import numpy as np
import pytest
import torch

from oracle import mcs_oracle as orc
from tests import parity as P
from token_sparse_attention_gb300 import build as mcs_build
from token_sparse_attention_gb300 import mcs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mcs_build.build()
    mcs.lib()
    assert torch.cuda.is_available()
    yield
    assert mcs.mcs_device_status() == 0


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _sibling_idx(N, G, K, overlap, seed):
    """[G, K] ascending index sets; group 2u+1 keeps about `overlap` of group
    2u's set and draws the rest elsewhere (siblings select similar keys)."""
    rng = np.random.default_rng(seed)
    out = np.empty((G, K), dtype=np.int64)
    for g in range(G):
        if g % 2 == 1 and overlap > 0:
            prev = out[g - 1]
            keep = rng.choice(prev, size=int(round(overlap * K)), replace=False)
            rest = np.setdiff1d(np.arange(N), keep)
            extra = rng.choice(rest, size=K - keep.shape[0], replace=False)
            out[g] = np.sort(np.concatenate([keep, extra]))
        else:
            out[g] = np.sort(rng.choice(N, size=K, replace=False))
    return out


def _pair_lists_host(buf, p, BH):
    """Unpack the pair-list buffer: per (head, pair) the entries up to its length."""
    G = p.G
    Pn = -(-G // 2)
    cap = -(-2 * p.K // 128) * 128
    off = -(-BH * Pn * 4 // 256) * 256
    raw = buf.cpu().numpy()
    lens = raw[:BH * Pn * 4].view(np.int32).reshape(BH, Pn)
    ent = raw[off:off + BH * Pn * cap * 4].view(np.int32).reshape(BH, Pn, cap)
    return lens, ent, cap


@pytest.mark.parametrize("B,H,N,K,overlap", [(1, 2, 1000, 300, 0.6), (2, 1, 517, 77, 0.0),
                                             (1, 1, 640, 640, 1.0), (1, 3, 300, 1, 0.0),
                                             (1, 1, 4100, 1500, 0.9)])
def test_pair_lists_are_unions_with_membership(B, H, N, K, overlap):
    C = 64
    p = mcs.params(B, H, N, 128, C, K)
    G, BH = p.G, B * H
    idx = np.stack([_sibling_idx(N, G, K, overlap, seed=N + h) for h in range(BH)])
    pairs = mcs.empty_pairs(p)
    mcs.mcs_pair_lists(p, _i32(idx.reshape(B, H, G, K)), pairs)
    assert mcs.mcs_device_status() == 0
    lens, ent, cap = _pair_lists_host(pairs, p, BH)
    for h in range(BH):
        for u in range(-(-G // 2)):
            a = set(idx[h, 2 * u].tolist())
            b = set(idx[h, 2 * u + 1].tolist()) if 2 * u + 1 < G else set()
            want = sorted(a | b)
            n = int(lens[h, u])
            assert n == len(want)
            e = ent[h, u].astype(np.int64)
            tok = e[:n] & ((1 << 28) - 1)
            bits = (e[:n] >> 28) & 3
            np.testing.assert_array_equal(tok, want)
            np.testing.assert_array_equal(bits & 1, [t in a for t in want])
            np.testing.assert_array_equal(bits >> 1, [t in b for t in want])
            assert np.all(e[n:cap] == 0)


@pytest.mark.parametrize("B,H,N,D,K,overlap", [(1, 2, 512, 128, 200, 0.6), (2, 1, 300, 128, 129, 0.3),
                                               (1, 2, 517, 64, 77, 0.0), (1, 1, 640, 64, 128, 0.9),
                                               (1, 1, 333, 64, 333, 1.0), (1, 1, 200, 128, 1, 0.0),
                                               (1, 2, 2048, 128, 410, 0.6), (1, 1, 1100, 64, 600, 0.5)])
def test_sparse_attn_pairs_matches_oracle(B, H, N, D, K, overlap):
    C = 64
    q, k, v = P.random_qkv(B, H, N, D, seed=N + K + D)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    p = mcs.params(B, H, N, D, C, K)
    G, BH = p.G, B * H
    perm = np.stack([P.random_groups(N, C, seed=N * 7 + h) for h in range(BH)])
    idx = np.stack([_sibling_idx(N, G, K, overlap, seed=N * 3 + h) for h in range(BH)])
    permd = _i32(perm.reshape(B, H, G * C))
    pairs = mcs.empty_pairs(p)
    mcs.mcs_pair_lists(p, _i32(idx.reshape(B, H, G, K)), pairs)
    out = torch.full_like(qd, float("nan"))
    mcs.mcs_sparse_attn_pairs(p, qd, kd, vd, permd, pairs, None, out)
    # residual add and anchor record through the same lists
    g_res = torch.Generator().manual_seed(N)
    res = (0.05 * torch.randn(q.shape, generator=g_res, dtype=torch.float64)).to(torch.bfloat16)
    out_add = torch.empty_like(qd)
    mcs.mcs_sparse_attn_pairs(p, qd, kd, vd, permd, pairs, res.cuda(), out_add)
    dense_in = (0.3 * torch.randn(q.shape, generator=g_res, dtype=torch.float64)).to(torch.bfloat16)
    rec = torch.empty_like(qd)
    mcs.mcs_sparse_attn_pairs_record(p, qd, kd, vd, permd, pairs, dense_in.cuda(), rec)
    assert mcs.mcs_device_status() == 0
    scale = orc.default_scale(D)
    for h in range(BH):
        b, hh = divmod(h, H)
        want = orc.sparse_attention(P.f64(q[b, hh]), P.f64(k[b, hh]), P.f64(v[b, hh]),
                                    perm[h], idx[h], C, scale)
        P.assert_close(out[b, hh], want, f"pairs b{b} h{hh}")
        P.assert_close(out_add[b, hh], want + P.f64(res[b, hh]), f"pairs + residual b{b} h{hh}")
        P.assert_close(rec[b, hh], P.f64(dense_in[b, hh]) - want, f"pairs record b{b} h{hh}")

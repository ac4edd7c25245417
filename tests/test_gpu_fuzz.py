"""Seeded random shapes through every attention entry point, against the
oracle.

Each case draws B, H, N (1 to 1500, so most are ragged; four more cases
take N = 1, 37, 64 and 129: shorter than a group, one group, one token past
it), D in {64, 128}, C in {64, 128}, K in [1, N], the activation
layout and whether a residual is added, then checks every output row of
mcs_dense_attn (+ LSE), mcs_sparse_attn, mcs_sparse_attn_e4m3 and, for C = 64,
mcs_sparse_attn_pairs against the fp64 oracle with the fixed tolerances of the
other parity tests.  The inputs come from the shared seeded generator; the
groups and index sets from the seeded helpers of tests/parity.py.
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


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
    N = int(rng.integers(1, 1501)) if seed < 16 else [1, 37, 64, 129][seed - 16]
    D, C = int(rng.choice([64, 128])), int(rng.choice([64, 128]))
    K = int(rng.integers(1, N + 1))
    layout = int(rng.integers(0, 2))
    with_res = bool(rng.integers(0, 2))
    return B, H, N, D, C, K, layout, with_res


def _lay(t, layout):
    return t.transpose(1, 2).contiguous() if layout == mcs.LAYOUT_BNHD else t.contiguous()


def _unlay(t, layout):
    return t.transpose(1, 2) if layout == mcs.LAYOUT_BNHD else t


@pytest.mark.parametrize("seed", range(20))
def test_random_shapes_match_oracle(seed):
    B, H, N, D, C, K, layout, with_res = _case(seed)
    q, k, v = P.random_qkv(B, H, N, D, seed=7 * seed + 3)
    G = -(-N // C)
    perm = np.stack([np.stack([P.random_groups(N, C, 97 * seed + b * H + h) for h in range(H)])
                     for b in range(B)])
    idx = np.stack([np.stack([P.random_idx(N, G, K, 89 * seed + b * H + h) for h in range(H)])
                    for b in range(B)])
    res = None
    if with_res:
        g = torch.Generator().manual_seed(seed)
        res = (0.05 * torch.randn(B, H, N, D, generator=g, dtype=torch.float64)).to(torch.bfloat16)
    p = mcs.params(B, H, N, D, C, K, layout=layout)
    qd, kd, vd = (_lay(t, layout).cuda() for t in (q, k, v))
    rd = None if res is None else _lay(res, layout).cuda()
    pd, xd = _i32(perm), _i32(idx)
    scale = orc.default_scale(D)
    what = f"seed {seed}: B={B} H={H} N={N} D={D} C={C} K={K} layout={layout} res={with_res}"

    dense = torch.full_like(qd, float("nan"))
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    mcs.mcs_dense_attn(p, qd, kd, vd, dense, lse)
    sparse = torch.full_like(qd, float("nan"))
    mcs.mcs_sparse_attn(p, qd, kd, vd, pd, xd, rd, sparse)
    ks = float(k.float().abs().max()) / 448.0
    vs = float(v.float().abs().max()) / 448.0
    k8 = torch.empty(kd.shape, dtype=torch.uint8, device="cuda")
    v8 = torch.empty_like(k8)
    mcs.mcs_quantize_e4m3(kd, ks, k8)
    mcs.mcs_quantize_e4m3(vd, vs, v8)
    e4 = torch.full_like(qd, float("nan"))
    mcs.mcs_sparse_attn_e4m3(p, qd, k8, v8, ks, vs, pd, xd, rd, e4)
    paired = None
    if mcs.mcs_pair_bytes(p):
        pairs = mcs.empty_pairs(p)
        mcs.mcs_pair_lists(p, xd, pairs)
        paired = torch.full_like(qd, float("nan"))
        mcs.mcs_sparse_attn_pairs(p, qd, kd, vd, pd, pairs, rd, paired)
    assert mcs.mcs_device_status() == 0, what

    dense, sparse, e4 = (_unlay(t, layout) for t in (dense, sparse, e4))
    k8h, v8h = (_unlay(t, layout) for t in (k8, v8))
    if paired is not None:
        paired = _unlay(paired, layout)
    for b in range(B):
        for h in range(H):
            qh, kh, vh = P.f64(q[b, h]), P.f64(k[b, h]), P.f64(v[b, h])
            O, L = orc.dense_attention(qh, kh, vh, scale)
            P.assert_close(dense[b, h], O, f"{what} dense b{b} h{h}")
            assert np.max(np.abs(P.f64(lse[b, h]) - L)) <= P.LSE_ABS, what
            r = 0.0 if res is None else P.f64(res[b, h])
            want = orc.sparse_attention(qh, kh, vh, perm[b, h], idx[b, h], C, scale) + r
            P.assert_close(sparse[b, h], want, f"{what} sparse b{b} h{h}")
            if paired is not None:
                P.assert_close(paired[b, h], want, f"{what} pairs b{b} h{h}")
            ko = orc.e4m3_encode(k[b, h].float().numpy(), ks)
            vo = orc.e4m3_encode(v[b, h].float().numpy(), vs)
            assert np.array_equal(k8h[b, h].contiguous().cpu().numpy(), ko), what
            assert np.array_equal(v8h[b, h].contiguous().cpu().numpy(), vo), what
            want8 = orc.sparse_attention_e4m3(qh, ko, vo, ks, vs, perm[b, h], idx[b, h], C,
                                              scale) + r
            P.assert_close(e4[b, h], want8, f"{what} e4m3 b{b} h{h}")

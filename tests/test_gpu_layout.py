"""[B,N,H,D] activations (the layout DiT blocks hold) give bit-identical
results to [B,H,N,D] through every entry point that reads or writes them:
only addresses change, never the arithmetic.  Every call goes through the C
ABI (libmcs.so)."""

import numpy as np
import pytest
import torch

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


def bnhd(t):
    return t.transpose(1, 2).contiguous()


def same(a, b, what):
    assert torch.equal(a.cpu(), b.cpu()), what


CASES = [(2, 3, 1000, 128, 128, 300), (1, 2, 777, 64, 64, 200), (2, 2, 300, 128, 64, 300)]


@pytest.mark.parametrize("B,H,N,D,C,K", CASES)
def test_anchor_and_reuse_are_layout_independent(B, H, N, D, C, K):
    q, k, v = [t.cuda() for t in P.random_qkv(B, H, N, D, seed=N + D)]
    q1, k1, v1 = [t.cuda() for t in P.random_qkv(B, H, N, D, seed=N + D + 1)]
    res = {}
    for layout in (mcs.LAYOUT_BHND, mcs.LAYOUT_BNHD):
        p = mcs.params(B, H, N, D, C, K, layout=layout)
        cv = bnhd if layout == mcs.LAYOUT_BNHD else (lambda t: t)
        back = bnhd if layout == mcs.LAYOUT_BNHD else (lambda t: t)
        qa, ka, va = cv(q), cv(k), cv(v)
        perm = torch.empty(B, H, p.G * C, dtype=torch.int32, device="cuda")
        idx = torch.empty(B, H, p.G, K, dtype=torch.int32, device="cuda")
        dense, resid = torch.empty_like(qa), torch.empty_like(qa)
        lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
        ret = torch.empty(B, H, p.G, dtype=torch.float32, device="cuda")
        ws = mcs.empty_workspace(mcs.mcs_anchor_workspace(p))
        mcs.mcs_anchor_select(p, qa, ka, va, perm, idx, dense, lse, resid, ws, retained=ret)
        out = torch.empty_like(qa)
        mcs.mcs_sparse_attn(p, cv(q1), cv(k1), cv(v1), perm, idx, resid, out)
        # the entry points one at a time
        perm2 = torch.empty_like(perm)
        mcs.mcs_group(p, qa, perm2, mcs.empty_workspace(mcs.mcs_group_workspace(p)))
        perm3 = torch.empty_like(perm)
        mcs.mcs_group_noalloc(p, qa, perm3)
        mass = torch.empty(B * H, p.G, N, dtype=torch.float32, device="cuda")
        mcs.mcs_group_mass(p, qa, ka, lse, perm, 0, B * H, mass)
        rec = torch.empty_like(qa)
        mcs.mcs_sparse_attn_record(p, qa, ka, va, perm, idx, dense, rec)
        plain = torch.empty_like(qa)
        mcs.mcs_sparse_attn(p, qa, ka, va, perm, idx, None, plain)
        blk = 16 if K % 16 == 0 else 1
        pb = mcs.params(B, H, N, D, C, (K // blk) * blk, layout=layout)
        pidx = torch.empty(B, H, p.G, pb.K, dtype=torch.int32, device="cuda")
        mcs.mcs_pooled_block_select(pb, qa, ka, perm, blk, pidx,
                                    mcs.empty_workspace(mcs.mcs_block_workspace(pb, blk)))
        extra = {}
        if mcs.mcs_pair_bytes(p):  # C = 64: the sibling-pair path
            pairs = mcs.empty_pairs(p)
            mcs.mcs_pair_lists(p, idx, pairs)
            pout = torch.empty_like(qa)
            mcs.mcs_sparse_attn_pairs(p, cv(q1), cv(k1), cv(v1), perm, pairs, resid, pout)
            prec = torch.empty_like(qa)
            mcs.mcs_sparse_attn_pairs_record(p, qa, ka, va, perm, pairs, dense, prec)
            extra = dict(pout=back(pout), prec=back(prec))  # (the lists come from idx)
        assert mcs.mcs_device_status() == 0
        res[layout] = dict(perm=perm, idx=idx, dense=back(dense), lse=lse, resid=back(resid),
                           ret=ret, out=back(out), perm2=perm2, perm3=perm3, mass=mass,
                           rec=back(rec), plain=back(plain), pidx=pidx, **extra)
    a, b = res[mcs.LAYOUT_BHND], res[mcs.LAYOUT_BNHD]
    for name in a:
        same(a[name], b[name], name)
    # sanity: the anchor produced groups and a residual that reproduces dense
    P.check_valid_perm(a["perm"][0, 0].cpu().numpy(), N, C)
    assert np.isfinite(P.f64(a["dense"])).all()


def test_bad_layout_is_rejected_before_launch():
    p = mcs.params(1, 1, 256, 128, 64, 40, layout=2)
    q = torch.zeros(1, 1, 256, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mcs.McsError):
        mcs.mcs_dense_attn(p, q, q, q, torch.empty_like(q))


@pytest.mark.parametrize("name,density", [("large", 0.2), ("asset3d", 0.15)])
def test_full_size_dense_and_reuse_layout_independent(name, density):
    # full size (all heads), the launches the benchmark times; D = C = 128
    # and D = C = 64
    from token_sparse_attention_gb300 import synth
    w = synth.workload(name)
    K = w.K(density)
    q, k, v = synth.make_qkv(w, 0, device="cuda")
    p0 = mcs.params(w.B, w.H, w.N, w.D, w.C, K)
    p1 = mcs.params(w.B, w.H, w.N, w.D, w.C, K, layout=mcs.LAYOUT_BNHD)
    G = p0.G
    # groups and indices: any valid ones (a strided selection per group)
    perm = torch.arange(G * w.C, dtype=torch.int32, device="cuda").clamp_max(w.N - 1)
    perm[w.N:] = -1
    perm = perm.expand(w.B, w.H, -1).contiguous()
    step = w.N // K
    idx = (torch.arange(K, dtype=torch.int32, device="cuda") * step)
    idx = (idx[None, :] + torch.arange(G, dtype=torch.int32, device="cuda")[:, None] % step)
    idx = idx.expand(w.B, w.H, G, K).contiguous()
    res = (0.01 * q).contiguous()
    outs = {}
    for p, cv in ((p0, lambda t: t), (p1, bnhd)):
        d = torch.empty_like(cv(q))
        lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device="cuda")
        mcs.mcs_dense_attn(p, cv(q), cv(k), cv(v), d, lse)
        o = torch.empty_like(d)
        mcs.mcs_sparse_attn(p, cv(q), cv(k), cv(v), perm, idx, cv(res), o)
        assert mcs.mcs_device_status() == 0
        outs[p.layout] = (cv(d), lse, cv(o))   # bnhd() is its own inverse
        del d, o
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)

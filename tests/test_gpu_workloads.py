"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times.

The oracle cannot run whole heads of 75600 queries, so each workload is
checked on sampled units the oracle computes one by one, plus properties that
hold at any size:
  * the whole anchor step on the GPU: valid groups for every head, selected
    indices ascending and in range, retained mass at most the group size, the
    fused selection equal to group mass + radix top-K on head 0, index sets
    unchanged through the metadata entry's bitmaps, and reuse with the
    anchor's own inputs reproducing the dense output;
  * dense attention and LSE on sampled query rows of two heads;
  * group mass, top-K and sparse attention (+ residual) on sampled groups of
    head 0, with the groups, LSE values and indices made by the oracle;
  * agreement of the GPU grouping of head 0 with the oracle's;
  * the multi-step schedules (small: anchor then four reuse steps; long:
    anchors at steps 0 and 5 of ten), each step on its own drifted inputs,
    with the last reuse step's sampled groups checked against the oracle's
    reuse step under the oracle's own metadata from the last anchor.
"""

import numpy as np
import pytest
import torch

from oracle import mcs_oracle as orc
from tests import parity as P
from token_sparse_attention_gb300 import build as mcs_build
from token_sparse_attention_gb300 import mcs
from token_sparse_attention_gb300 import synth

pytestmark = pytest.mark.gpu

CASES = [("small", 0.1), ("small", 0.2), ("small", 0.3), ("large", 0.2), ("long", 0.15),
         ("long", 0.25), ("asset3d", 0.15)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mcs_build.build()
    mcs.lib()
    assert torch.cuda.is_available()


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


@pytest.mark.parametrize("name,density", CASES)
def test_workload_full_size(name, density):
    w = synth.workload(name)
    K = w.K(density)
    BH = w.B * w.H
    q, k, v = synth.make_qkv(w, 0, device="cuda")
    p = mcs.params(w.B, w.H, w.N, w.D, w.C, K)
    G = p.G
    perm = torch.empty(w.B, w.H, G * w.C, dtype=torch.int32, device="cuda")
    idx = torch.empty(w.B, w.H, G, K, dtype=torch.int32, device="cuda")
    dense = torch.empty_like(q)
    res = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device="cuda")
    ret = torch.empty(w.B, w.H, G, dtype=torch.float32, device="cuda")
    ws = mcs.empty_workspace(mcs.mcs_anchor_workspace(p))
    mcs.mcs_anchor_select(p, q, k, v, perm, idx, dense, lse, res, ws, retained=ret)
    assert mcs.mcs_device_status() == 0
    del ws

    # ---- properties of the whole anchor step
    pm = perm.view(BH, -1).cpu().numpy()
    for h in range(BH):
        P.check_valid_perm(pm[h], w.N, w.C)
    sizes = np.array([min(w.C, w.N - g * w.C) for g in range(G)])
    assert np.all(P.f64(ret).reshape(BH, G) <= sizes * (1 + 1e-4))
    for h in (0, BH - 1):
        ih = idx.view(BH, G, K)[h].cpu().numpy()
        assert ih.min() >= 0 and ih.max() < w.N and np.all(np.diff(ih, axis=1) > 0)
    # the anchor's fused selection (mass histogram + one-read top-K) against
    # mcs_group_mass + mcs_topk (four-read radix select) on the same groups and
    # LSE: identical index sets for head 0
    m0 = torch.empty(1, G, w.N, dtype=torch.float32, device="cuda")
    mcs.mcs_group_mass(p, q, k, lse, perm, 0, 1, m0)
    s0 = torch.empty(G, K, dtype=torch.int32, device="cuda")
    mcs.mcs_topk(p, m0, s0)
    assert torch.equal(s0, idx.view(BH, G, K)[0]), f"{name}: fused selection differs"
    del m0, s0
    # the metadata entry's index bitmaps carry every head's sets unchanged
    entry = torch.empty(mcs.mcs_meta_bytes(p), dtype=torch.uint8, device="cuda")
    mcs.mcs_meta_pack(p, idx, entry)
    back = torch.empty_like(idx)
    mcs.mcs_meta_unpack(p, entry, back)
    assert mcs.mcs_device_status() == 0 and torch.equal(back, idx)
    del entry, back
    same = torch.empty_like(q)
    mcs.mcs_sparse_attn(p, q, k, v, perm, idx, res, same)
    d = (same.float() - dense.float()).abs()
    assert d.max().item() <= 2 ** -5 and d.mean().item() <= 2e-3 * dense.float().abs().mean().item()

    # ---- dense + LSE on sampled rows of two heads
    scale = orc.default_scale(w.D)
    rng = np.random.default_rng(7)
    host = {}
    for h in (0, BH - 1):
        b, hh = divmod(h, w.H)
        qh, kh, vh = (P.f64(t[b, hh]) for t in (q, k, v))
        host[h] = (qh, kh, vh)
        rows = np.sort(rng.choice(w.N, 64, replace=False))
        O, L = orc.dense_attention(qh, kh, vh, scale, rows=rows)
        P.assert_close(dense[b, hh][rows], O, f"{name} dense rows h{h}")
        assert np.max(np.abs(P.f64(lse[b, hh][rows]) - L)) <= P.LSE_ABS

    # ---- selection and sparse attention on oracle-made groups of head 0
    qh, kh, vh = host[0]
    operm = orc.pddp_perm(qh, w.C, 32)
    groups = [0, G - 1] + list(rng.choice(np.arange(1, G - 1), 6, replace=False))
    members = {g: orc.group_members(operm, g, w.C) for g in groups}
    olse = np.zeros(w.N)
    for g in groups:
        olse[members[g]] = orc.dense_attention(qh, kh, vh, scale, rows=members[g])[1]
    olse32 = olse.astype(np.float32)
    perm_in = perm.clone()
    perm_in.view(BH, -1)[0] = _i32(operm)
    lse_in = lse.clone()
    lse_in.view(BH, -1)[0] = torch.from_numpy(olse32).cuda()
    mass = torch.empty(1, G, w.N, dtype=torch.float32, device="cuda")
    mcs.mcs_group_mass(p, q, k, lse_in, perm_in, 0, 1, mass)
    sel = torch.empty(G, K, dtype=torch.int32, device="cuda")
    mcs.mcs_topk(p, mass, sel)
    mass_h, sel_h = mass[0].cpu().numpy().astype(np.float64), sel.cpu().numpy()
    oidx = idx.view(BH, G, K)[0].cpu().numpy().copy()  # any valid sets for other groups
    for g in groups:
        want = orc.group_mass(qh, kh, olse32.astype(np.float64), members[g], scale)
        got = mass_h[g]
        assert np.all(np.abs(got - want) <= P.MASS_REL * want + 1e-12 * len(members[g])), \
            f"{name} mass g{g}"
        o_sel = orc.topk_select(want, K)[0]
        P.assert_topk_within_ties(sel_h[g], o_sel, want, K)
        oidx[g] = o_sel
    idx_in = idx.clone()
    idx_in.view(BH, G, K)[0] = _i32(oidx)
    g_res = torch.Generator().manual_seed(3)
    r0 = (0.05 * torch.randn(w.N, w.D, generator=g_res, dtype=torch.float64)).to(torch.bfloat16)
    res_in = res.clone()
    res_in.view(BH, w.N, w.D)[0] = r0.cuda()
    out = torch.empty_like(q)
    mcs.mcs_sparse_attn(p, q, k, v, perm_in, idx_in, res_in, out)
    out0 = out.view(BH, w.N, w.D)[0]
    for g in groups:
        m = members[g]
        want = orc.sparse_attention_group(qh, kh, vh, m, oidx[g], scale) + P.f64(r0)[m]
        P.assert_close(out0[torch.from_numpy(m).cuda()], want, f"{name} sparse g{g}")
    assert mcs.mcs_device_status() == 0
    if mcs.mcs_pair_bytes(p):
        # C = 64: the sibling-pair path on the same groups and index sets
        pairs = mcs.empty_pairs(p)
        mcs.mcs_pair_lists(p, idx_in, pairs)
        outp = torch.empty_like(q)
        mcs.mcs_sparse_attn_pairs(p, q, k, v, perm_in, pairs, res_in, outp)
        outp0 = outp.view(BH, w.N, w.D)[0]
        for g in groups:
            m = members[g]
            want = orc.sparse_attention_group(qh, kh, vh, m, oidx[g], scale) + P.f64(r0)[m]
            P.assert_close(outp0[torch.from_numpy(m).cuda()], want, f"{name} pairs g{g}")
        assert mcs.mcs_device_status() == 0
        del pairs, outp

    # ---- grouping of head 0 against the oracle's (fp32 vs fp64 projections
    # may move near-median tokens)
    gid_got, gid_want = np.empty(w.N, int), np.empty(w.N, int)
    for g in range(G):
        gid_got[orc.group_members(pm[0], g, w.C)] = g
        gid_want[orc.group_members(operm, g, w.C)] = g
    agree = np.mean(gid_got == gid_want)
    print(f"{name}: token groups agreeing with the oracle {agree:.4f}")
    assert agree >= 0.9


SCHEDULES = [("small", 0.3), ("long", 0.25)]


def _oracle_anchor_groups(qa, ka, va, C, K, groups_seed):
    """The oracle's anchor metadata for sampled groups of one head: its own
    grouping, LSE (rounded to fp32 as the GPU stores it), group masses,
    top-K sets and bf16 residual bf16(dense_bf16 - O') of each group's rows
    (wispaper.ai, "Reused exact selection beats recomputed mean pooling";
    "Residual correction recovers the discarded tail")."""
    N = qa.shape[0]
    G = -(-N // C)
    scale = orc.default_scale(qa.shape[1])
    operm = orc.pddp_perm(qa, C, 32)
    rng = np.random.default_rng(groups_seed)
    groups = [0, G - 1] + list(rng.choice(np.arange(1, G - 1), 6, replace=False))
    meta = {}
    for g in groups:
        m = orc.group_members(operm, g, C)
        O, L = orc.dense_attention(qa, ka, va, scale, rows=m)
        L32 = L.astype(np.float32)
        lse = np.zeros(N)
        lse[m] = L32
        mass = orc.group_mass(qa, ka, lse, m, scale)
        sel = orc.topk_select(mass, K)[0]
        sp = orc.sparse_attention_group(qa, ka, va, m, sel, scale)
        meta[g] = dict(members=m, lse32=L32, mass=mass, idx=sel,
                       residual=orc.round_to_bf16(orc.round_to_bf16(O) - sp))
    return operm, meta


@pytest.mark.parametrize("name,density", SCHEDULES)
def test_schedule_drifted_reuse(name, density):
    """The workload's denoising schedule on the GPU: an anchor step (grouping,
    dense + LSE, exact selection, residual record) at each anchor and reuse
    steps (sparse attention under the cached groups and indices + cached
    residual) in between, every step on its own drifted inputs.  Checked:
      * at the last anchor, the selection kernels fed the oracle's grouping
        and LSE reproduce the oracle's masses and top-K sets on sampled
        groups of head 0;
      * at the last reuse step, sparse attention on that step's inputs under
        the oracle's anchor metadata (grouping, index sets, residual) matches
        the oracle's reuse step on those groups;
      * the GPU's own reuse output stays closer to that step's dense
        attention than the same sparse pass without the residual."""
    w = synth.workload(name)
    K = w.K(density)
    BH = w.B * w.H
    p = mcs.params(w.B, w.H, w.N, w.D, w.C, K)
    G = p.G
    scale = orc.default_scale(w.D)
    last = w.steps - 1
    a_last = max(a for a in w.anchors if a < last)
    perm = torch.empty(w.B, w.H, G * w.C, dtype=torch.int32, device="cuda")
    idx = torch.empty(w.B, w.H, G, K, dtype=torch.int32, device="cuda")
    shape = (w.B, w.H, w.N, w.D)
    res = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    dense = torch.empty_like(res)
    out = torch.empty_like(res)
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device="cuda")
    ws = mcs.empty_workspace(mcs.mcs_anchor_workspace(p))
    operm = meta = None
    for t in range(w.steps):
        q, k, v = synth.make_qkv(w, t, device="cuda")
        if t in w.anchors:
            mcs.mcs_anchor_select(p, q, k, v, perm, idx, dense, lse, res, ws)
            assert mcs.mcs_device_status() == 0, f"{name} anchor step {t}"
            if t == a_last:
                qa, ka, va = (P.f64(x[0, 0]) for x in (q, k, v))
                operm, meta = _oracle_anchor_groups(qa, ka, va, w.C, K, 11 + t)
                perm_in = perm.clone()
                perm_in.view(BH, -1)[0] = _i32(operm)
                lse_in = lse.clone()
                for g, mg in meta.items():
                    lse_in.view(BH, -1)[0][torch.from_numpy(mg["members"]).cuda()] = \
                        torch.from_numpy(mg["lse32"]).cuda()
                mass = torch.empty(1, G, w.N, dtype=torch.float32, device="cuda")
                mcs.mcs_group_mass(p, q, k, lse_in, perm_in, 0, 1, mass)
                sel = torch.empty(G, K, dtype=torch.int32, device="cuda")
                mcs.mcs_topk(p, mass, sel)
                for g, mg in meta.items():
                    got = mass[0, g].double().cpu().numpy()
                    want = mg["mass"]
                    assert np.all(np.abs(got - want) <= P.MASS_REL * want
                                  + 1e-12 * len(mg["members"])), f"{name} step {t} mass g{g}"
                    P.assert_topk_within_ties(sel[g].cpu().numpy(), mg["idx"], want, K)
                del mass, sel, lse_in
            continue
        mcs.mcs_sparse_attn(p, q, k, v, perm, idx, res, out)
        assert mcs.mcs_device_status() == 0, f"{name} reuse step {t}"
        assert torch.isfinite(out).all()
        if t != last:
            continue
        # ---- the GPU schedule's own reuse output against this step's dense attention
        dense_t = torch.empty_like(out)
        mcs.mcs_dense_attn(p, q, k, v, dense_t, None)
        bare = torch.empty_like(out)
        mcs.mcs_sparse_attn(p, q, k, v, perm, idx, None, bare)
        l1_res = ((out.float() - dense_t.float()).abs().sum() / dense_t.float().abs().sum()).item()
        l1_bare = ((bare.float() - dense_t.float()).abs().sum() / dense_t.float().abs().sum()).item()
        print(f"{name} s={density} step {t}: rel L1 to dense {l1_res:.4f} with the residual, "
              f"{l1_bare:.4f} without")
        assert l1_res < l1_bare
        del dense_t, bare
        # ---- oracle reuse step on sampled groups of head 0, under the oracle's metadata
        qT, kT, vT = (P.f64(x[0, 0]) for x in (q, k, v))
        perm_in = perm.clone()
        perm_in.view(BH, -1)[0] = _i32(operm)
        idx_in = idx.clone()
        res_in = res.clone()
        for g, mg in meta.items():
            idx_in.view(BH, G, K)[0][g] = _i32(mg["idx"])
            res_in.view(BH, w.N, w.D)[0][torch.from_numpy(mg["members"]).cuda()] = \
                P.bf16_tensor(mg["residual"])
        got = torch.empty_like(out)
        mcs.mcs_sparse_attn(p, q, k, v, perm_in, idx_in, res_in, got)
        assert mcs.mcs_device_status() == 0
        got0 = got.view(BH, w.N, w.D)[0]
        oidx = np.zeros((G, K), dtype=np.int64)
        ores = np.zeros((w.N, w.D))
        for g, mg in meta.items():
            oidx[g] = mg["idx"]
            ores[mg["members"]] = mg["residual"]
        want = orc.reuse_step(qT, kT, vT, operm, oidx, ores, w.C, scale, groups=list(meta))
        for g, mg in meta.items():
            m = mg["members"]
            P.assert_close(got0[torch.from_numpy(m).cuda()], want[m], f"{name} step {t} reuse g{g}")


@pytest.mark.parametrize("N,C,D", [(75600, 128, 128), (65536, 64, 64)])
def test_pddp_full_size_clusters(N, C, D):
    x, want = P.separated_clusters(N, C, D, seed=N)
    q = P.bf16_tensor(x)[None, None]
    p = mcs.params(1, 1, N, D, C, 1)
    perm = torch.empty(1, 1, p.G * C, dtype=torch.int32, device="cuda")
    ws = mcs.empty_workspace(mcs.mcs_group_workspace(p))
    mcs.mcs_group(p, q, perm, ws)
    np.testing.assert_array_equal(perm[0, 0].cpu().numpy(), want)

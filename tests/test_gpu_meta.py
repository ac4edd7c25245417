"""GPU tests of the metadata cache staging (mcs_meta_*, mcs_stager_*): index
lists packed into bitmaps and unpacked again are unchanged; entries offloaded
to pinned host memory and prefetched back into device slots, one layer ahead,
give the same reuse-step outputs as metadata kept on the device.  Every call
goes through the C ABI (libmcs.so)."""

import numpy as np
import pytest
import torch

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


def _anchor_into(p, q, k, v, entry):
    """Anchor step whose perm and residual land in a device entry and whose
    indices are packed into it; returns the index list."""
    perm, _, res = mcs.meta_views(p, entry)
    idx = torch.empty(p.B, p.H, p.G, p.K, dtype=torch.int32, device="cuda")
    dense = torch.empty_like(q)
    lse = torch.empty(p.B, p.H, p.N, dtype=torch.float32, device="cuda")
    ws = mcs.empty_workspace(mcs.mcs_anchor_workspace(p))
    mcs.mcs_anchor_select(p, q, k, v, perm, idx, dense, lse, res, ws)
    mcs.mcs_meta_pack(p, idx, entry)
    return idx


def _layer_inputs(w, layer):
    # each layer has its own activations: the workload's generator at step
    # `layer` (anchor) and `layer + 1` (reuse)
    q0, k0, v0 = [t.cuda() for t in synth.make_qkv(w, layer)]
    q1, k1, v1 = [t.cuda() for t in synth.make_qkv(w, layer + 1)]
    return (q0, k0, v0), (q1, k1, v1)


@pytest.mark.parametrize("N,K,C", [(5000, 1000, 128), (4099, 4099, 64), (300, 1, 64),
                                   (70, 33, 64)])
def test_pack_unpack_round_trip(N, K, C):
    B, H = 2, 2
    p = mcs.params(B, H, N, 64, C, K)
    rng = np.random.default_rng(N + K)
    idx = np.stack([np.sort(rng.choice(N, K, replace=False)) for _ in range(B * H * p.G)])
    idx = torch.from_numpy(idx.astype(np.int32)).view(B, H, p.G, K).cuda()
    entry = torch.full((mcs.mcs_meta_bytes(p),), 0x5A, dtype=torch.uint8, device="cuda")
    mcs.mcs_meta_pack(p, idx, entry)
    got = torch.full_like(idx, -7)
    mcs.mcs_meta_unpack(p, entry, got)
    assert mcs.mcs_device_status() == 0
    assert torch.equal(got, idx)
    # the bitmap itself: bit j of a group's row set exactly for its indices
    _, bits, _ = mcs.meta_views(p, entry)
    b = bits[0, 0, 0].cpu().numpy().view(np.uint32)
    want = np.zeros(b.size, dtype=np.uint32)
    for j in idx[0, 0, 0].cpu().numpy():
        want[j >> 5] |= np.uint32(1) << np.uint32(j & 31)
    np.testing.assert_array_equal(b, want)


def test_pack_reports_repeated_index():
    p = mcs.params(1, 1, 256, 64, 64, 4)
    idx = torch.tensor([[3, 3, 5, 9]] * p.G, dtype=torch.int32).view(1, 1, p.G, 4).cuda()
    entry = torch.empty(mcs.mcs_meta_bytes(p), dtype=torch.uint8, device="cuda")
    mcs.mcs_meta_pack(p, idx, entry)
    assert mcs.mcs_device_status() == 6   # MCS_ERR_BOUNDS, and the word is cleared


def test_offload_prefetch_round_trip():
    w = synth.workload("tiny")
    p = mcs.params(w.B, w.H, w.N, w.D, w.C, w.K(0.2))
    nbytes = mcs.mcs_meta_bytes(p)
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    (q0, k0, v0), _ = _layer_inputs(w, 0)
    idx = _anchor_into(p, q0, k0, v0, dev)
    want = dev.clone()
    host = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    copy = torch.cuda.Stream()
    st = mcs.Stager(p, [dev], copy)
    cur = torch.cuda.current_stream()
    st.offload(0, host, after=cur)
    st.wait(0, cur)
    dev.zero_()               # queued on the compute stream after the offload
    st.prefetch(0, host, after=cur)
    st.wait(0, cur)
    got = dev.clone()         # ordered after the prefetch by the wait
    back = torch.empty_like(idx)
    mcs.mcs_meta_unpack(p, dev, back)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    assert torch.equal(back, idx)
    st.close()


def test_layer_pipeline_prefetch_one_ahead_matches_resident():
    # three layers, two device slots: while layer l runs from slot l % 2 the
    # entry of layer l + 1 is copied into the other slot
    w = synth.workload("tiny")
    p = mcs.params(w.B, w.H, w.N, w.D, w.C, w.K(0.2))
    L = 3
    nbytes = mcs.mcs_meta_bytes(p)
    resident, hosts, reuse_in, idxs = [], [], [], []
    for layer in range(L):
        (q0, k0, v0), (q1, k1, v1) = _layer_inputs(w, 2 * layer)
        e = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        idxs.append(_anchor_into(p, q0, k0, v0, e))
        resident.append(e)
        reuse_in.append((q1, k1, v1))
    copy = torch.cuda.Stream()
    cur = torch.cuda.current_stream()
    # offload each layer's entry to pinned host memory through one slot
    tmp = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    off = mcs.Stager(p, [tmp], copy)
    for layer in range(L):
        h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
        tmp.copy_(resident[layer])
        off.offload(0, h, after=cur)
        off.wait(0, cur)        # tmp is reused next iteration
        hosts.append(h)
    torch.cuda.synchronize()
    off.close()
    # resident reference outputs, from the anchor's own index lists
    want = []
    for layer in range(L):
        perm, _, res = mcs.meta_views(p, resident[layer])
        q1, k1, v1 = reuse_in[layer]
        out = torch.empty_like(q1)
        mcs.mcs_sparse_attn(p, q1, k1, v1, perm, idxs[layer], res, out)
        want.append(out)
    # staged: two slots, prefetch one layer ahead, indices unpacked per layer
    slots = [torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda") for _ in range(2)]
    st = mcs.Stager(p, slots, copy)
    st.prefetch(0, hosts[0], after=cur)
    idx = torch.empty(p.B, p.H, p.G, p.K, dtype=torch.int32, device="cuda")
    got = []
    for layer in range(L):
        s = layer % 2
        if layer + 1 < L:
            st.prefetch(1 - s, hosts[layer + 1], after=cur)
        st.wait(s, cur)
        perm, _, res = mcs.meta_views(p, slots[s])
        mcs.mcs_meta_unpack(p, slots[s], idx)
        q1, k1, v1 = reuse_in[layer]
        out = torch.empty_like(q1)
        mcs.mcs_sparse_attn(p, q1, k1, v1, perm, idx, res, out)
        got.append(out)
    torch.cuda.synchronize()
    st.close()
    assert mcs.mcs_device_status() == 0
    for layer in range(L):
        np.testing.assert_array_equal(got[layer].view(torch.int16).cpu().numpy(),
                                      want[layer].view(torch.int16).cpu().numpy())


def test_round_trip_in_bnhd_layout():
    # the entry's residual follows the activations' layout; one copy moves it
    w = synth.workload("tiny")
    p = mcs.params(w.B, w.H, w.N, w.D, w.C, w.K(0.2), layout=mcs.LAYOUT_BNHD)
    q, k, v = [t.cuda().transpose(1, 2).contiguous() for t in synth.make_qkv(w, 0)]
    entry = torch.empty(mcs.mcs_meta_bytes(p), dtype=torch.uint8, device="cuda")
    idx = _anchor_into(p, q, k, v, entry)
    assert mcs.meta_views(p, entry)[2].shape == (w.B, w.N, w.H, w.D)
    host = torch.empty_like(entry, device="cpu").pin_memory()
    copy = torch.cuda.Stream()
    cur = torch.cuda.current_stream()
    st = mcs.Stager(p, [entry], copy)
    want = entry.clone()
    st.offload(0, host, after=cur)
    st.wait(0, cur)
    entry.zero_()
    st.prefetch(0, host, after=cur)
    st.wait(0, cur)
    back = torch.empty_like(idx)
    mcs.mcs_meta_unpack(p, entry, back)
    torch.cuda.synchronize()
    st.close()
    assert torch.equal(entry, want) and torch.equal(back, idx)

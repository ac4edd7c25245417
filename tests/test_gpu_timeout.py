"""Bounded waits: a kernel whose loads are withheld must give up, report
MCS_ERR_TIMEOUT through the device status word, free its resources, and leave
the CUDA context usable.  The fault is injected on the host side
(MCS_TEST_FAULT=stall_load makes the producer warps stop after the first K/V
tile); no GPU fault, trap or endless wait is involved."""

import os

import numpy as np
import pytest
import torch

from oracle import mcs_oracle as orc
from tests import parity as P
from token_sparse_attention_gb300 import build as mcs_build
from token_sparse_attention_gb300 import mcs

pytestmark = pytest.mark.gpu


def test_withheld_load_times_out_and_context_survives(monkeypatch):
    mcs_build.build()
    mcs.lib()
    N, D, C, K = 512, 128, 128, 300  # 3 key tiles per group
    q, k, v = P.random_qkv(1, 1, N, D, seed=21)
    perm = P.random_groups(N, C, 22)[None, None]
    idx = P.random_idx(N, perm.shape[-1] // C, K, 23)[None, None]
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    pd = torch.from_numpy(perm.astype(np.int32)).cuda()
    xd = torch.from_numpy(idx.astype(np.int32)).cuda()
    p = mcs.params(1, 1, N, D, C, K)
    out = torch.zeros_like(qd)
    assert mcs.mcs_device_status() == 0
    monkeypatch.setenv("MCS_TEST_FAULT", "stall_load")
    mcs.mcs_sparse_attn(p, qd, kd, vd, pd, xd, None, out)
    assert mcs.mcs_device_status() == 5  # MCS_ERR_TIMEOUT
    dense = torch.zeros_like(qd)
    mcs.mcs_dense_attn(p, qd, kd, vd, dense, None)
    assert mcs.mcs_device_status() == 5
    monkeypatch.delenv("MCS_TEST_FAULT")
    # the context is still usable and the same calls now give correct results
    mcs.mcs_sparse_attn(p, qd, kd, vd, pd, xd, None, out)
    assert mcs.mcs_device_status() == 0
    want = orc.sparse_attention(P.f64(q[0, 0]), P.f64(k[0, 0]), P.f64(v[0, 0]), perm[0, 0],
                                idx[0, 0], C, orc.default_scale(D))
    P.assert_close(out[0, 0], want, "sparse after a timed-out launch")


def test_withheld_e4m3_load_times_out_and_context_survives(monkeypatch):
    """The same for the E4M3 K/V path, whose producers stage rows through
    registers instead of cp.async."""
    mcs_build.build()
    mcs.lib()
    N, D, C, K = 512, 128, 128, 300
    q, k, v = P.random_qkv(1, 1, N, D, seed=24)
    perm = P.random_groups(N, C, 25)[None, None]
    idx = P.random_idx(N, perm.shape[-1] // C, K, 26)[None, None]
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    ks = float(k.float().abs().max()) / 448.0
    vs = float(v.float().abs().max()) / 448.0
    k8 = torch.empty(kd.shape, dtype=torch.uint8, device="cuda")
    v8 = torch.empty_like(k8)
    mcs.mcs_quantize_e4m3(kd, ks, k8)
    mcs.mcs_quantize_e4m3(vd, vs, v8)
    pd = torch.from_numpy(perm.astype(np.int32)).cuda()
    xd = torch.from_numpy(idx.astype(np.int32)).cuda()
    p = mcs.params(1, 1, N, D, C, K)
    out = torch.zeros_like(qd)
    assert mcs.mcs_device_status() == 0
    monkeypatch.setenv("MCS_TEST_FAULT", "stall_load")
    mcs.mcs_sparse_attn_e4m3(p, qd, k8, v8, ks, vs, pd, xd, None, out)
    assert mcs.mcs_device_status() == 5  # MCS_ERR_TIMEOUT
    monkeypatch.delenv("MCS_TEST_FAULT")
    mcs.mcs_sparse_attn_e4m3(p, qd, k8, v8, ks, vs, pd, xd, None, out)
    assert mcs.mcs_device_status() == 0
    ko = orc.e4m3_encode(k[0, 0].float().numpy(), ks)
    vo = orc.e4m3_encode(v[0, 0].float().numpy(), vs)
    want = orc.sparse_attention_e4m3(P.f64(q[0, 0]), ko, vo, ks, vs, perm[0, 0], idx[0, 0], C,
                                     orc.default_scale(D))
    P.assert_close(out[0, 0], want, "e4m3 sparse after a timed-out launch")

"""mcs_group_noalloc: grouping for callers that cannot allocate device memory.

Some host programs cannot give the library a workspace: plugins that are
handed only their inputs and outputs, or servers that fix their device
memory use at start-up and allow no allocation afterwards.  For them the
library offers mcs_group_noalloc, whose scratch is a fixed 64 MiB array
inside the library.  These tests check, through the C ABI, that it returns
exactly what mcs_group (caller workspace) returns, on two calls in a row with
different inputs (the shared array keeps the previous call's contents), also
when the heads do not fit the array at once, and that a problem too large
for the array is refused without a launch.  This file is collected last.
"""

import ctypes

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


def _group_both(B, H, N, D, C, seed):
    q = P.random_qkv(B, H, N, D, seed)[0].cuda()
    p = mcs.params(B, H, N, D, C, 1)
    want = torch.empty(B, H, p.G * C, dtype=torch.int32, device="cuda")
    ws = mcs.empty_workspace(mcs.mcs_group_workspace(p))
    mcs.mcs_group(p, q, want, ws)
    got = torch.full_like(want, -7)
    mcs.mcs_group_noalloc(p, q, got)
    assert mcs.mcs_device_status() == 0
    return got.cpu().numpy(), want.cpu().numpy(), p


@pytest.mark.parametrize("B,H,N,D,C", [(1, 2, 2048, 128, 64), (1, 3, 1000, 64, 128)])
def test_noalloc_matches_workspace_grouping_twice(B, H, N, D, C):
    for call, seed in enumerate((11, 12)):
        got, want, p = _group_both(B, H, N, D, C, seed)
        np.testing.assert_array_equal(got, want, err_msg=f"call {call}")
        for b in range(B):
            for h in range(H):
                P.check_valid_perm(got[b, h], N, C)


def test_noalloc_heads_in_batches():
    # eight heads of 32760 tokens need more than 64 MiB of scratch together
    # while one head fits, so the entry point groups them a batch at a time
    B, H, N, D, C = 1, 8, 32760, 128, 128
    p = mcs.params(B, H, N, D, C, 1)
    assert mcs.mcs_group_workspace(p) > (64 << 20)
    assert mcs.mcs_group_workspace(mcs.params(1, 1, N, D, C, 1)) <= (64 << 20)
    for seed in (21, 22):
        got, want, _ = _group_both(B, H, N, D, C, seed)
        np.testing.assert_array_equal(got, want)


def test_noalloc_leaves_device_memory_unchanged():
    # once the library is loaded on the device (first call), a further call
    # takes no device memory: free memory before and after is the same
    B, H, N, D, C = 1, 4, 3000, 128, 128
    q = P.random_qkv(B, H, N, D, 31)[0].cuda()
    p = mcs.params(B, H, N, D, C, 1)
    perm = torch.empty(B, H, p.G * C, dtype=torch.int32, device="cuda")
    mcs.mcs_group_noalloc(p, q, perm)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    mcs.mcs_group_noalloc(p, q, perm)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert mcs.mcs_device_status() == 0


def test_noalloc_refuses_oversized_problem():
    # one head of 2^20 tokens in groups of 64 needs far more than 64 MiB
    p = mcs.params(1, 1, 1 << 20, 128, 64, 1)
    assert mcs.mcs_group_workspace(p) > (64 << 20)
    st = mcs.lib().mcs_group_noalloc(ctypes.byref(p), 16, 16, None)
    assert st == 3  # MCS_ERR_WORKSPACE, nothing launched
    assert mcs.mcs_device_status() == 0

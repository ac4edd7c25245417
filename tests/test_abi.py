"""Host-side checks of the C ABI (CPU only: no kernel runs here).

The library must build, load, export every function include/mcs.h declares,
and reject bad arguments on the host before any launch.
"""

import ctypes
import os
import re

import pytest

from token_sparse_attention_gb300 import build as mcs_build
from token_sparse_attention_gb300 import mcs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    mcs_build.build()
    return mcs.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "mcs.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mcs_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_binding_names():
    assert declared_functions() == sorted(mcs.EXPORTED)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    nm = os.popen(f"nm -D --defined-only {mcs.library_path()}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}\b", nm), name


def test_status_strings(L):
    for code, name in mcs.STATUS_NAMES.items():
        assert mcs.mcs_status_string(code) == name


def test_host_validation_rejects_bad_arguments(L):
    null = None
    # null params
    assert L.mcs_dense_attn(None, null, null, null, null, null, null) == 1
    # unsupported head dim / group size
    p = mcs.params(1, 2, 256, 96, 64, 40)
    assert L.mcs_dense_attn(ctypes.byref(p), 16, 16, 16, 16, None, None) == 2
    p = mcs.params(1, 2, 256, 128, 32, 40)
    assert L.mcs_sparse_attn(ctypes.byref(p), 16, 16, 16, 16, 16, None, 16, None) == 2
    # K out of range
    p = mcs.params(1, 2, 256, 128, 64, 0)
    assert L.mcs_sparse_attn(ctypes.byref(p), 16, 16, 16, 16, 16, None, 16, None) == 1
    p = mcs.params(1, 2, 256, 128, 64, 257)
    assert L.mcs_sparse_attn(ctypes.byref(p), 16, 16, 16, 16, 16, None, 16, None) == 1
    # null tensor pointer
    p = mcs.params(1, 2, 256, 128, 64, 40)
    assert L.mcs_sparse_attn(ctypes.byref(p), 16, 16, None, 16, 16, None, 16, None) == 1
    # misaligned bf16 pointer
    assert L.mcs_dense_attn(ctypes.byref(p), 16, 16, 24, 16, None, None) == 1
    # too many heads for the grid
    p = mcs.params(2, 40000, 64, 128, 64, 10)
    assert L.mcs_dense_attn(ctypes.byref(p), 16, 16, 16, 16, None, None) == 1
    # negative scale
    p = mcs.params(1, 1, 64, 128, 64, 10, scale=-1.0)
    assert L.mcs_dense_attn(ctypes.byref(p), 16, 16, 16, 16, None, None) == 1
    # workspace missing / too small
    p = mcs.params(1, 2, 2048, 128, 64, 410)
    assert L.mcs_group(ctypes.byref(p), 16, 16, None, 0, None) == 3
    assert L.mcs_anchor_select(ctypes.byref(p), 16, 16, 16, 16, 16, 16, 16, 16, None, 16, 64,
                               None) == 3


def test_workspace_queries(L):
    p = mcs.params(1, 2, 2048, 128, 64, 410)
    g = mcs.mcs_group_workspace(p)
    a = mcs.mcs_anchor_workspace(p)
    assert g > 0 and a >= g
    # at least one head of group masses (G x N fp32)
    assert a >= p.G * p.N * 4
    bad = mcs.params(1, 2, 2048, 96, 64, 410)
    assert mcs.mcs_group_workspace(bad) == 0


def test_meta_entry_layout(L):
    # one layer's cache entry: perm | idx | residual, 256-byte aligned sections
    p = mcs.params(1, 40, 75600, 128, 128, 15120)
    G = p.G
    po, io, ro = mcs.mcs_meta_offsets(p)
    total = mcs.mcs_meta_bytes(p)
    # the indices are stored as bitmaps of N bits per group
    perm_b, idx_b, res_b = 40 * G * 128 * 4, 40 * G * (-(-75600 // 32)) * 4, 40 * 75600 * 128 * 2
    assert po == 0 and io % 256 == 0 and ro % 256 == 0 and total % 256 == 0
    assert perm_b <= io < perm_b + 256
    assert idx_b <= ro - io < idx_b + 256
    assert res_b <= total - ro < res_b + 256
    # K outside [1, N]: no size, an error status
    bad = mcs.params(1, 1, 100, 128, 64, 0)
    assert L.mcs_meta_bytes(ctypes.byref(bad)) == 0
    assert L.mcs_meta_offsets(ctypes.byref(bad), None, None, None) == 1


def test_meta_pack_rejects_bad_arguments(L):
    p = mcs.params(1, 2, 256, 128, 64, 40)
    assert L.mcs_meta_pack(ctypes.byref(p), None, 256, None) == 1
    assert L.mcs_meta_pack(ctypes.byref(p), 256, 256 + 16, None) == 1   # entry not 256-aligned
    assert L.mcs_meta_unpack(ctypes.byref(p), 256, None, None) == 1
    bad = mcs.params(1, 2, 256, 128, 64, 0)
    assert L.mcs_meta_unpack(ctypes.byref(bad), 256, 256, None) == 1


def test_stager_rejects_bad_arguments(L):
    # every check here happens on the host before any CUDA call
    p = mcs.params(1, 2, 256, 128, 64, 40)
    h = ctypes.c_void_p()
    two = (ctypes.c_void_p * 2)(256, 512)
    assert L.mcs_stager_create(ctypes.byref(p), 2, two, None, None) == 1    # no out pointer
    assert L.mcs_stager_create(ctypes.byref(p), 0, two, None, ctypes.byref(h)) == 1  # no slots
    assert L.mcs_stager_create(ctypes.byref(p), 2, None, None, ctypes.byref(h)) == 1
    odd = (ctypes.c_void_p * 1)(256 + 16)                                   # not 256-aligned
    assert L.mcs_stager_create(ctypes.byref(p), 1, odd, None, ctypes.byref(h)) == 1
    bad = mcs.params(1, 2, 256, 96, 64, 40)                                 # unsupported D
    assert L.mcs_stager_create(ctypes.byref(bad), 2, two, None, ctypes.byref(h)) == 2
    assert not h.value
    assert L.mcs_stager_prefetch(None, 0, 16, None) == 1
    assert L.mcs_stager_offload(None, 0, 16, None) == 1
    assert L.mcs_stager_wait(None, 0, None) == 1
    L.mcs_stager_destroy(None)


def test_layout_field_is_checked_on_the_host(L):
    # layout 0 ([B,H,N,D]) and 1 ([B,N,H,D]) are accepted; anything else is
    # an invalid argument, reported before any CUDA call
    for layout, want in ((2, 1), (-1, 1)):
        p = mcs.params(1, 2, 256, 128, 64, 40, layout=layout)
        assert L.mcs_dense_attn(ctypes.byref(p), 16, 16, 16, 16, None, None) == want
        assert L.mcs_meta_bytes(ctypes.byref(p)) == 0
    assert ctypes.sizeof(mcs.Params) == 9 * 4


def test_pair_lists_host_checks(L):
    # sibling-pair lists: C = 64 only, K up to 16384; buffer of P = ceil(G/2)
    # lengths, then P rows of the union capacity (2K rounded up to 128)
    p = mcs.params(1, 2, 1000, 128, 64, 300)  # G = 16, P = 8
    n = mcs.mcs_pair_bytes(p)
    cap = -(-2 * 300 // 128) * 128
    off = -(-2 * 8 * 4 // 256) * 256
    assert n == off + 2 * 8 * cap * 4
    assert mcs.mcs_pair_bytes(mcs.params(1, 2, 1000, 128, 128, 300)) == 0  # C = 128
    assert mcs.mcs_pair_bytes(mcs.params(1, 1, 40000, 128, 64, 16385)) == 0  # K too large
    q = mcs.params(1, 2, 1000, 128, 128, 300)
    assert L.mcs_pair_lists(ctypes.byref(q), 256, 256, 1 << 20, None) == 2
    assert L.mcs_sparse_attn_pairs(ctypes.byref(q), 16, 16, 16, 16, 256, None, 16, None) == 2
    assert L.mcs_pair_lists(ctypes.byref(p), None, 256, n, None) == 1  # null idx
    assert L.mcs_pair_lists(ctypes.byref(p), 256, 16, n, None) == 1  # pairs not 256-aligned
    assert L.mcs_pair_lists(ctypes.byref(p), 256, 256, n - 4, None) == 3  # too small
    assert L.mcs_sparse_attn_pairs(ctypes.byref(p), 16, 16, 16, 16, None, None, 16, None) == 1
    assert L.mcs_sparse_attn_pairs_record(ctypes.byref(p), 16, 16, 16, 16, 256, None, 16,
                                          None) == 1  # record needs dense_out


def test_e4m3_entries_reject_bad_arguments(L):
    f = ctypes.c_float
    # quantize: null or misaligned buffers, bad scales; n = 0 launches nothing
    assert L.mcs_quantize_e4m3(None, 16, f(1.0), 16, None) == 1
    assert L.mcs_quantize_e4m3(16, 16, f(1.0), 24, None) == 1
    assert L.mcs_quantize_e4m3(16, 16, f(0.0), 16, None) == 1
    assert L.mcs_quantize_e4m3(16, 16, f(float("inf")), 16, None) == 1
    assert L.mcs_quantize_e4m3(None, 0, f(1.0), None, None) == 0
    # sparse attention over E4M3 K/V: the shape checks of mcs_sparse_attn,
    # then pointers, alignment and scales
    p = mcs.params(1, 2, 256, 96, 64, 40)
    assert L.mcs_sparse_attn_e4m3(ctypes.byref(p), 16, 16, 16, f(1), f(1), 16, 16, None, 16,
                                  None) == 2
    p = mcs.params(1, 2, 256, 128, 64, 0)
    assert L.mcs_sparse_attn_e4m3(ctypes.byref(p), 16, 16, 16, f(1), f(1), 16, 16, None, 16,
                                  None) == 1
    p = mcs.params(1, 2, 256, 128, 64, 40)
    assert L.mcs_sparse_attn_e4m3(ctypes.byref(p), 16, None, 16, f(1), f(1), 16, 16, None, 16,
                                  None) == 1
    assert L.mcs_sparse_attn_e4m3(ctypes.byref(p), 16, 16, 40, f(1), f(1), 16, 16, None, 16,
                                  None) == 1
    assert L.mcs_sparse_attn_e4m3(ctypes.byref(p), 16, 16, 16, f(0), f(1), 16, 16, None, 16,
                                  None) == 1
    assert L.mcs_sparse_attn_e4m3(ctypes.byref(p), 16, 16, 16, f(1), f(-2), 16, 16, None, 16,
                                  None) == 1
    assert L.mcs_sparse_attn_e4m3(ctypes.byref(p), 16, 16, 16, f(1), f(1), 16, 16, 24, 16,
                                  None) == 1

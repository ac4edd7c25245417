"""Thin Python binding of libmcs.so (the C ABI declared in include/mcs.h).

Argument marshalling only: every function takes torch tensors that already
live on a CUDA device, checks dtype/shape/contiguity, and passes raw device
pointers and the current CUDA stream to the C entry point of the same name.
Every step of the computation runs in the library's kernels; there is no
fallback of any kind.  If libmcs.so is missing or fails to load, the first
call raises.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

__all__ = [
    "McsError", "Params", "params", "lib", "library_path", "EXPORTED",
    "mcs_status_string", "mcs_last_cuda_error", "mcs_device_status",
    "mcs_group_workspace", "mcs_anchor_workspace", "mcs_group", "mcs_dense_attn",
    "mcs_group_mass", "mcs_topk", "mcs_select", "mcs_sparse_attn", "mcs_sparse_attn_record",
    "mcs_anchor_select", "mcs_group_noalloc", "mcs_meta_bytes", "mcs_meta_offsets",
    "meta_views", "mcs_meta_pack", "mcs_meta_unpack", "Stager", "mcs_block_workspace", "mcs_block_topk", "mcs_pooled_block_select",
    "mcs_gather_mass", "mcs_rel_l1", "mcs_pair_bytes", "empty_pairs", "mcs_pair_lists",
    "mcs_sparse_attn_pairs", "mcs_sparse_attn_pairs_record", "mcs_quantize_e4m3",
    "mcs_sparse_attn_e4m3",
]

# Every symbol include/mcs.h declares.
EXPORTED = (
    "mcs_status_string", "mcs_last_cuda_error", "mcs_device_status", "mcs_group_workspace",
    "mcs_anchor_workspace", "mcs_group", "mcs_dense_attn", "mcs_group_mass", "mcs_topk",
    "mcs_select", "mcs_sparse_attn", "mcs_sparse_attn_record", "mcs_anchor_select", "mcs_group_noalloc",
    "mcs_pair_bytes", "mcs_pair_lists", "mcs_sparse_attn_pairs", "mcs_sparse_attn_pairs_record",
    "mcs_meta_bytes", "mcs_meta_offsets", "mcs_meta_pack", "mcs_meta_unpack",
    "mcs_stager_create", "mcs_stager_destroy",
    "mcs_stager_prefetch", "mcs_stager_offload", "mcs_stager_wait", "mcs_block_workspace",
    "mcs_block_topk", "mcs_pooled_block_select", "mcs_gather_mass", "mcs_rel_l1",
    "mcs_quantize_e4m3", "mcs_sparse_attn_e4m3",
)

STATUS_NAMES = {0: "MCS_OK", 1: "MCS_ERR_INVALID_ARG", 2: "MCS_ERR_UNSUPPORTED",
                3: "MCS_ERR_WORKSPACE", 4: "MCS_ERR_CUDA", 5: "MCS_ERR_TIMEOUT",
                6: "MCS_ERR_BOUNDS"}


class McsError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{where}: {name}" + (f" ({detail})" if detail else ""))


class Params(ctypes.Structure):
    """mcs_params: B, H, N, D, C, K, scale (0 -> 1/sqrt(D)), pddp_iters (0 -> 32),
    layout (0: activations [B, H, N, D]; 1: [B, N, H, D])."""

    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int),
                ("D", ctypes.c_int), ("C", ctypes.c_int), ("K", ctypes.c_int),
                ("scale", ctypes.c_float), ("pddp_iters", ctypes.c_int), ("layout", ctypes.c_int)]

    @property
    def G(self) -> int:
        return -(-self.N // self.C)


LAYOUT_BHND, LAYOUT_BNHD = 0, 1


def params(B, H, N, D, C=128, K=None, scale=0.0, pddp_iters=0, layout=LAYOUT_BHND) -> Params:
    return Params(B, H, N, D, C, N if K is None else K, scale, pddp_iters, layout)


def library_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmcs.so")


_LIB = None
_vp, _sz, _i, _st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int
_pp = ctypes.POINTER(Params)

_SIGS = {
    "mcs_status_string": ([_st], ctypes.c_char_p),
    "mcs_last_cuda_error": ([], ctypes.c_char_p),
    "mcs_device_status": ([_vp], _st),
    "mcs_group_workspace": ([_pp], _sz),
    "mcs_anchor_workspace": ([_pp], _sz),
    "mcs_group": ([_pp, _vp, _vp, _vp, _sz, _vp], _st),
    "mcs_dense_attn": ([_pp, _vp, _vp, _vp, _vp, _vp, _vp], _st),
    "mcs_group_mass": ([_pp, _vp, _vp, _vp, _vp, _i, _i, _vp, _vp], _st),
    "mcs_topk": ([_pp, _vp, _i, _vp, _vp, _vp], _st),
    "mcs_select": ([_pp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _st),
    "mcs_sparse_attn": ([_pp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp], _st),
    "mcs_sparse_attn_record": ([_pp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp], _st),
    "mcs_pair_bytes": ([_pp], _sz),
    "mcs_pair_lists": ([_pp, _vp, _vp, _sz, _vp], _st),
    "mcs_sparse_attn_pairs": ([_pp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp], _st),
    "mcs_sparse_attn_pairs_record": ([_pp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp], _st),
    "mcs_anchor_select": ([_pp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _st),
    "mcs_group_noalloc": ([_pp, _vp, _vp, _vp], _st),
    "mcs_meta_bytes": ([_pp], _sz),
    "mcs_meta_offsets": ([_pp, ctypes.POINTER(_sz), ctypes.POINTER(_sz), ctypes.POINTER(_sz)], _st),
    "mcs_meta_pack": ([_pp, _vp, _vp, _vp], _st),
    "mcs_meta_unpack": ([_pp, _vp, _vp, _vp], _st),
    "mcs_stager_create": ([_pp, _i, ctypes.POINTER(_vp), _vp, ctypes.POINTER(_vp)], _st),
    "mcs_stager_destroy": ([_vp], None),
    "mcs_stager_prefetch": ([_vp, _i, _vp, _vp], _st),
    "mcs_stager_offload": ([_vp, _i, _vp, _vp], _st),
    "mcs_stager_wait": ([_vp, _i, _vp], _st),
    "mcs_block_workspace": ([_pp, _i], _sz),
    "mcs_block_topk": ([_pp, _vp, _i, _i, _vp, _vp, _vp, _sz, _vp], _st),
    "mcs_pooled_block_select": ([_pp, _vp, _vp, _vp, _i, _vp, _vp, _sz, _vp], _st),
    "mcs_gather_mass": ([_pp, _vp, _i, _vp, _vp, _vp], _st),
    "mcs_rel_l1": ([_pp, _vp, _vp, _vp, _i, _vp, _vp], _st),
    "mcs_quantize_e4m3": ([_vp, _sz, ctypes.c_float, _vp, _vp], _st),
    "mcs_sparse_attn_e4m3": ([_pp, _vp, _vp, _vp, ctypes.c_float, ctypes.c_float, _vp, _vp,
                              _vp, _vp, _vp], _st),
}


def lib() -> ctypes.CDLL:
    """Load libmcs.so (built in-tree by build.py).  Raises if absent."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built; run __graft_entry__.build() first")
        L = ctypes.CDLL(path)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _LIB = L
    return _LIB


# ---------------------------------------------------------------- helpers

def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t, dtype, shape=None, name="tensor", optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _check(status: int, where: str):
    if status != 0:
        detail = lib().mcs_last_cuda_error().decode() if status == 4 else ""
        raise McsError(status, where, detail)


def _qkv_shape(p: Params):
    return (p.B, p.N, p.H, p.D) if p.layout == LAYOUT_BNHD else (p.B, p.H, p.N, p.D)


# ---------------------------------------------------------------- entry points

def mcs_status_string(status: int) -> str:
    return lib().mcs_status_string(status).decode()


def mcs_last_cuda_error() -> str:
    return lib().mcs_last_cuda_error().decode()


def mcs_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return lib().mcs_device_status(_stream(stream))


def mcs_group_workspace(p: Params) -> int:
    return lib().mcs_group_workspace(ctypes.byref(p))


def mcs_anchor_workspace(p: Params) -> int:
    return lib().mcs_anchor_workspace(ctypes.byref(p))


def mcs_group(p: Params, q, perm, ws, stream=None):
    bf = torch.bfloat16
    _check(lib().mcs_group(ctypes.byref(p), _ptr(q, bf, _qkv_shape(p), "q"),
                           _ptr(perm, torch.int32, (p.B, p.H, p.G * p.C), "perm"),
                           _ptr(ws, torch.uint8, None, "ws"), ws.numel(), _stream(stream)),
           "mcs_group")


def mcs_group_noalloc(p: Params, q, perm, stream=None):
    """mcs_group for callers that cannot allocate: uses the library's built-in
    64 MiB scratch instead of a workspace (see include/mcs.h)."""
    bf = torch.bfloat16
    _check(lib().mcs_group_noalloc(ctypes.byref(p), _ptr(q, bf, _qkv_shape(p), "q"),
                                   _ptr(perm, torch.int32, (p.B, p.H, p.G * p.C), "perm"),
                                   _stream(stream)), "mcs_group_noalloc")


def mcs_dense_attn(p: Params, q, k, v, out, lse=None, stream=None):
    bf, s = torch.bfloat16, _qkv_shape(p)
    _check(lib().mcs_dense_attn(ctypes.byref(p), _ptr(q, bf, s, "q"), _ptr(k, bf, s, "k"),
                                _ptr(v, bf, s, "v"), _ptr(out, bf, s, "out"),
                                _ptr(lse, torch.float32, (p.B, p.H, p.N), "lse", optional=True),
                                _stream(stream)), "mcs_dense_attn")


def mcs_group_mass(p: Params, q, k, lse, perm, head_begin, head_count, mass, stream=None):
    bf, s = torch.bfloat16, _qkv_shape(p)
    _check(lib().mcs_group_mass(ctypes.byref(p), _ptr(q, bf, s, "q"), _ptr(k, bf, s, "k"),
                                _ptr(lse, torch.float32, (p.B, p.H, p.N), "lse"),
                                _ptr(perm, torch.int32, (p.B, p.H, p.G * p.C), "perm"),
                                int(head_begin), int(head_count),
                                _ptr(mass, torch.float32, (head_count, p.G, p.N), "mass"),
                                _stream(stream)), "mcs_group_mass")


def mcs_topk(p: Params, mass, idx, retained=None, stream=None):
    rows = mass.numel() // p.N
    _check(lib().mcs_topk(ctypes.byref(p), _ptr(mass, torch.float32, None, "mass"), rows,
                          _ptr(idx, torch.int32, None, "idx"),
                          _ptr(retained, torch.float32, None, "retained", optional=True),
                          _stream(stream)), "mcs_topk")
    if idx.numel() != rows * p.K:
        raise ValueError("idx must hold rows * K entries")


def mcs_sparse_attn(p: Params, q, k, v, perm, idx, residual, out, stream=None):
    bf, s = torch.bfloat16, _qkv_shape(p)
    _check(lib().mcs_sparse_attn(ctypes.byref(p), _ptr(q, bf, s, "q"), _ptr(k, bf, s, "k"),
                                 _ptr(v, bf, s, "v"),
                                 _ptr(perm, torch.int32, (p.B, p.H, p.G * p.C), "perm"),
                                 _ptr(idx, torch.int32, (p.B, p.H, p.G, p.K), "idx"),
                                 _ptr(residual, bf, s, "residual", optional=True),
                                 _ptr(out, bf, s, "out"), _stream(stream)), "mcs_sparse_attn")


def mcs_sparse_attn_record(p: Params, q, k, v, perm, idx, dense_out, residual, stream=None):
    bf, s = torch.bfloat16, _qkv_shape(p)
    _check(lib().mcs_sparse_attn_record(
        ctypes.byref(p), _ptr(q, bf, s, "q"), _ptr(k, bf, s, "k"), _ptr(v, bf, s, "v"),
        _ptr(perm, torch.int32, (p.B, p.H, p.G * p.C), "perm"),
        _ptr(idx, torch.int32, (p.B, p.H, p.G, p.K), "idx"),
        _ptr(dense_out, bf, s, "dense_out"), _ptr(residual, bf, s, "residual"),
        _stream(stream)), "mcs_sparse_attn_record")


def _bytes8(t, name, numel):
    """E4M3 tensors: torch.float8_e4m3fn or their uint8 view."""
    if isinstance(t, torch.Tensor) and t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    ptr = _ptr(t, torch.uint8, None, name)
    if t.numel() != numel:
        raise ValueError(f"{name} must hold {numel} bytes, got {t.numel()}")
    return ptr


def mcs_quantize_e4m3(x, scale: float, x8, stream=None):
    """x8 = E4M3(x / scale), elementwise (x bf16; x8 uint8 or float8_e4m3fn)."""
    n = x.numel()
    _check(lib().mcs_quantize_e4m3(_ptr(x, torch.bfloat16, None, "x"), n, float(scale),
                                   _bytes8(x8, "x8", n), _stream(stream)), "mcs_quantize_e4m3")


def mcs_sparse_attn_e4m3(p: Params, q, k8, v8, k_scale: float, v_scale: float, perm, idx,
                         residual, out, stream=None):
    bf, s = torch.bfloat16, _qkv_shape(p)
    n = math.prod(s)
    _check(lib().mcs_sparse_attn_e4m3(
        ctypes.byref(p), _ptr(q, bf, s, "q"), _bytes8(k8, "k8", n), _bytes8(v8, "v8", n),
        float(k_scale), float(v_scale),
        _ptr(perm, torch.int32, (p.B, p.H, p.G * p.C), "perm"),
        _ptr(idx, torch.int32, (p.B, p.H, p.G, p.K), "idx"),
        _ptr(residual, bf, s, "residual", optional=True), _ptr(out, bf, s, "out"),
        _stream(stream)), "mcs_sparse_attn_e4m3")


def mcs_pair_bytes(p: Params) -> int:
    """Bytes of the sibling-pair key-list buffer (0: unsupported for p)."""
    return lib().mcs_pair_bytes(ctypes.byref(p))


def empty_pairs(p: Params, device="cuda"):
    """A device buffer for mcs_pair_lists (uint8, 256-byte aligned)."""
    n = mcs_pair_bytes(p)
    if n == 0:
        raise ValueError("pair lists need C = 64, K <= 16384 and N < 2^28")
    return empty_workspace(n, device)


def mcs_pair_lists(p: Params, idx, pairs, stream=None):
    _check(lib().mcs_pair_lists(
        ctypes.byref(p), _ptr(idx, torch.int32, (p.B, p.H, p.G, p.K), "idx"),
        _ptr(pairs, torch.uint8, None, "pairs"), pairs.numel(), _stream(stream)),
        "mcs_pair_lists")


def mcs_sparse_attn_pairs(p: Params, q, k, v, perm, pairs, residual, out, stream=None):
    bf, s = torch.bfloat16, _qkv_shape(p)
    _check(lib().mcs_sparse_attn_pairs(
        ctypes.byref(p), _ptr(q, bf, s, "q"), _ptr(k, bf, s, "k"), _ptr(v, bf, s, "v"),
        _ptr(perm, torch.int32, (p.B, p.H, p.G * p.C), "perm"),
        _ptr(pairs, torch.uint8, None, "pairs"),
        _ptr(residual, bf, s, "residual", optional=True), _ptr(out, bf, s, "out"),
        _stream(stream)), "mcs_sparse_attn_pairs")


def mcs_sparse_attn_pairs_record(p: Params, q, k, v, perm, pairs, dense_out, residual,
                                 stream=None):
    bf, s = torch.bfloat16, _qkv_shape(p)
    _check(lib().mcs_sparse_attn_pairs_record(
        ctypes.byref(p), _ptr(q, bf, s, "q"), _ptr(k, bf, s, "k"), _ptr(v, bf, s, "v"),
        _ptr(perm, torch.int32, (p.B, p.H, p.G * p.C), "perm"),
        _ptr(pairs, torch.uint8, None, "pairs"),
        _ptr(dense_out, bf, s, "dense_out"), _ptr(residual, bf, s, "residual"),
        _stream(stream)), "mcs_sparse_attn_pairs_record")


def mcs_select(p: Params, q, k, lse, perm, idx, ws, retained=None, stream=None):
    bf, s = torch.bfloat16, _qkv_shape(p)
    _check(lib().mcs_select(
        ctypes.byref(p), _ptr(q, bf, s, "q"), _ptr(k, bf, s, "k"),
        _ptr(lse, torch.float32, (p.B, p.H, p.N), "lse"),
        _ptr(perm, torch.int32, (p.B, p.H, p.G * p.C), "perm"),
        _ptr(idx, torch.int32, (p.B, p.H, p.G, p.K), "idx"),
        _ptr(retained, torch.float32, (p.B, p.H, p.G), "retained", optional=True),
        _ptr(ws, torch.uint8, None, "ws"), ws.numel(), _stream(stream)), "mcs_select")


def mcs_anchor_select(p: Params, q, k, v, perm, idx, dense_out, lse, residual, ws,
                      retained=None, stream=None):
    bf, s = torch.bfloat16, _qkv_shape(p)
    _check(lib().mcs_anchor_select(
        ctypes.byref(p), _ptr(q, bf, s, "q"), _ptr(k, bf, s, "k"), _ptr(v, bf, s, "v"),
        _ptr(perm, torch.int32, (p.B, p.H, p.G * p.C), "perm"),
        _ptr(idx, torch.int32, (p.B, p.H, p.G, p.K), "idx"),
        _ptr(dense_out, bf, s, "dense_out"), _ptr(lse, torch.float32, (p.B, p.H, p.N), "lse"),
        _ptr(residual, bf, s, "residual"),
        _ptr(retained, torch.float32, (p.B, p.H, p.G), "retained", optional=True),
        _ptr(ws, torch.uint8, None, "ws"), ws.numel(), _stream(stream)), "mcs_anchor_select")


def mcs_meta_bytes(p: Params) -> int:
    return lib().mcs_meta_bytes(ctypes.byref(p))


def mcs_meta_offsets(p: Params) -> tuple[int, int, int]:
    o = [_sz(0), _sz(0), _sz(0)]
    _check(lib().mcs_meta_offsets(ctypes.byref(p), *[ctypes.byref(x) for x in o]),
           "mcs_meta_offsets")
    return tuple(x.value for x in o)


def meta_views(p: Params, entry: torch.Tensor):
    """(perm, bits, residual) views into a metadata entry (uint8, host or
    device); bits [B, H, G, ceil(N/32)] holds the index bitmaps (as int32)."""
    if entry.dtype != torch.uint8 or not entry.is_contiguous() or entry.dim() != 1:
        raise ValueError("entry must be a contiguous 1-D uint8 tensor")
    if entry.numel() < mcs_meta_bytes(p):
        raise ValueError("entry is smaller than mcs_meta_bytes(p)")
    po, io, ro = mcs_meta_offsets(p)
    n_perm = p.B * p.H * p.G * p.C * 4
    W = -(-p.N // 32)
    n_idx = p.B * p.H * p.G * W * 4
    n_res = p.B * p.H * p.N * p.D * 2
    perm = entry[po:po + n_perm].view(torch.int32).view(p.B, p.H, p.G * p.C)
    idx = entry[io:io + n_idx].view(torch.int32).view(p.B, p.H, p.G, W)
    res = entry[ro:ro + n_res].view(torch.bfloat16).view(*_qkv_shape(p))
    return perm, idx, res


def mcs_meta_pack(p: Params, idx, entry, stream=None):
    _check(lib().mcs_meta_pack(ctypes.byref(p),
                               _ptr(idx, torch.int32, (p.B, p.H, p.G, p.K), "idx"),
                               _ptr(entry, torch.uint8, None, "entry"), _stream(stream)),
           "mcs_meta_pack")


def mcs_meta_unpack(p: Params, entry, idx, stream=None):
    _check(lib().mcs_meta_unpack(ctypes.byref(p), _ptr(entry, torch.uint8, None, "entry"),
                                 _ptr(idx, torch.int32, (p.B, p.H, p.G, p.K), "idx"),
                                 _stream(stream)), "mcs_meta_unpack")


class Stager:
    """Moves metadata entries between host memory and device slots (mcs_stager_*)."""

    def __init__(self, p: Params, slots, copy_stream):
        for t in slots:
            _ptr(t, torch.uint8, None, "slot")
            if t.numel() < mcs_meta_bytes(p):
                raise ValueError("slot is smaller than mcs_meta_bytes(p)")
        self.slots = list(slots)
        self._h = _vp()
        arr = (_vp * len(slots))(*[t.data_ptr() for t in slots])
        _check(lib().mcs_stager_create(ctypes.byref(p), len(slots), arr, _stream(copy_stream),
                                       ctypes.byref(self._h)), "mcs_stager_create")

    @staticmethod
    def _host(t):
        if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.uint8 or \
                not t.is_contiguous():
            raise ValueError("host entry must be a contiguous uint8 CPU tensor (pinned)")
        return t.data_ptr()

    def prefetch(self, slot: int, host_entry, after=None):
        _check(lib().mcs_stager_prefetch(self._h, slot, self._host(host_entry), _stream(after)),
               "mcs_stager_prefetch")

    def offload(self, slot: int, host_entry, after=None):
        _check(lib().mcs_stager_offload(self._h, slot, self._host(host_entry), _stream(after)),
               "mcs_stager_offload")

    def wait(self, slot: int, stream=None):
        _check(lib().mcs_stager_wait(self._h, slot, _stream(stream)), "mcs_stager_wait")

    def close(self):
        if self._h:
            lib().mcs_stager_destroy(self._h)
            self._h = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def mcs_block_workspace(p: Params, block: int) -> int:
    return lib().mcs_block_workspace(ctypes.byref(p), block)


def mcs_block_topk(p: Params, mass, block: int, idx, ws, retained=None, stream=None):
    rows = mass.numel() // p.N
    _ptr(idx, torch.int32, None, "idx")
    if idx.numel() != rows * p.K:
        raise ValueError("idx must hold rows * K entries")
    _check(lib().mcs_block_topk(ctypes.byref(p), _ptr(mass, torch.float32, None, "mass"), rows,
                                block, idx.data_ptr(),
                                _ptr(retained, torch.float32, (rows,), "retained", optional=True),
                                _ptr(ws, torch.uint8, None, "ws"), ws.numel(), _stream(stream)),
           "mcs_block_topk")


def mcs_pooled_block_select(p: Params, q, k, perm, block: int, idx, ws, stream=None):
    bf, s = torch.bfloat16, _qkv_shape(p)
    _check(lib().mcs_pooled_block_select(
        ctypes.byref(p), _ptr(q, bf, s, "q"), _ptr(k, bf, s, "k"),
        _ptr(perm, torch.int32, (p.B, p.H, p.G * p.C), "perm"), block,
        _ptr(idx, torch.int32, (p.B, p.H, p.G, p.K), "idx"),
        _ptr(ws, torch.uint8, None, "ws"), ws.numel(), _stream(stream)), "mcs_pooled_block_select")


def mcs_gather_mass(p: Params, mass, idx, retained, stream=None):
    rows = mass.numel() // p.N
    _ptr(idx, torch.int32, None, "idx")
    if idx.numel() != rows * p.K:
        raise ValueError("idx must hold rows * K entries")
    _check(lib().mcs_gather_mass(ctypes.byref(p), _ptr(mass, torch.float32, None, "mass"), rows,
                                 idx.data_ptr(), _ptr(retained, torch.float32, (rows,), "retained"),
                                 _stream(stream)), "mcs_gather_mass")


def mcs_rel_l1(p: Params, got, want, rows=None, stream=None) -> tuple:
    """(sum |got - want|, sum |want|) over the listed rows (all when None);
    synchronises the stream to read the two sums."""
    bf, s = torch.bfloat16, _qkv_shape(p)
    sums = torch.empty(2, dtype=torch.float64, device=got.device)
    nrows = 0 if rows is None else rows.numel()
    _check(lib().mcs_rel_l1(ctypes.byref(p), _ptr(got, bf, s, "got"), _ptr(want, bf, s, "want"),
                            _ptr(rows, torch.int32, None, "rows", optional=True), nrows,
                            sums.data_ptr(), _stream(stream)), "mcs_rel_l1")
    v = sums.cpu()
    return float(v[0]), float(v[1])


def empty_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A device byte buffer of at least nbytes (256-byte aligned by torch)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)

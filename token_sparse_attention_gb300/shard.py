"""Head-range partitioning of the attention path over ranks (one process per
GPU).

Every attention head (b, h) is independent at every step of the path:
grouping, dense attention with LSE, exact selection, sparse attention and the
residual all work on one head's queries, keys and values only (the pages
group the queries of each head and select KV tokens per head: wispaper.ai,
"Token-level selection needs tile-aligned query groups").  So a job with
several GPUs gives each rank a contiguous range of the flattened B*H heads;
the rank keeps its heads' groups, index sets and residual in its own memory,
and nothing crosses ranks on the data path.

Host logic only: which heads a rank owns and how a head range maps onto the
library's parameters and onto views of [B, H, N, D] activations.
"""

from __future__ import annotations

from . import mcs

__all__ = ["head_range", "slice_params", "head_slice"]


def head_range(rank: int, world: int, n_heads: int) -> tuple[int, int]:
    """Flattened heads [start, stop) owned by `rank` of `world`: contiguous
    ranges in rank order that cover every head once, sizes differing by at
    most one (the first n_heads % world ranks take one more)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of world {world}")
    if n_heads < 0:
        raise ValueError("n_heads must be >= 0")
    base, extra = divmod(n_heads, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def slice_params(p: mcs.Params, start: int, stop: int) -> mcs.Params:
    """Parameters of the call that covers flattened heads [start, stop) of
    the problem `p`.  In the [B, H, N, D] layout consecutive flattened heads
    are consecutive in memory, so the range is one batch of (stop - start)
    heads whose tensors start at head `start`.  The [B, N, H, D] layout
    interleaves the heads of a token and has no such slice."""
    if p.layout != mcs.LAYOUT_BHND:
        raise ValueError("head ranges are contiguous only in the [B, H, N, D] layout")
    if not 0 <= start < stop <= p.B * p.H:
        raise ValueError(f"head range [{start}, {stop}) outside 0..{p.B * p.H}")
    return mcs.params(1, stop - start, p.N, p.D, p.C, p.K, p.scale, p.pddp_iters, p.layout)


def head_slice(t, start: int, stop: int):
    """View of heads [start, stop) of a contiguous [B, H, ...] tensor (q, k,
    v, outputs, lse, perm, idx, retained) as a [1, stop - start, ...] tensor
    sharing its memory (no copy)."""
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    flat = t.reshape(t.shape[0] * t.shape[1], *t.shape[2:])
    return flat[start:stop].unsqueeze(0)

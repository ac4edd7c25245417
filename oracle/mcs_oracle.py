"""Plain fp64 CPU oracle for MC-Sparse token-sparse attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library.

Every function works on ONE attention head at a time (arrays ``[N, D]``), in
float64, on inputs that are already bf16 values (the bytes the GPU receives).
The arithmetic follows the method step by step, in the order the pages give it;
library primitives (matmul, exp, sort) serve as single steps and nothing is
blocked, fused or reordered.

Sources.  All pages carry the title "MC-Sparse: Deconstructing and Closing the
Dense-Sparse Attention Gap in Diffusion Transformers".  Citations below name
the site and the section:

* [ai.info/Method]  ai.info AI summary, section "Methodology in Plain English".
* [ai.info/Contrib] ai.info AI summary, section "Key Contributions".
* [wisp/Tile]       wispaper.ai, section "Token-level selection needs
                    tile-aligned query groups".
* [wisp/Reuse]      wispaper.ai, section "Reused exact selection beats
                    recomputed mean pooling".
* [wisp/Residual]   wispaper.ai, section "Residual correction recovers the
                    discarded tail".
* [wisp/Gap]        wispaper.ai, section "The gap has three separable sources".
* [agihunt/Select]  agihunt.info summary, paragraph on the selection objective
                    (top-K KV tokens of largest group attention mass, two-pass
                    kernel).
* [agihunt/Group]   agihunt.info summary, paragraph on token-level gathering
                    and PDDP groups of exactly C queries.
* [wisp/Pool]       wispaper.ai, section "Mean-pooled block scoring misses
                    high-mass tokens".
* [ai.info/Find]    ai.info AI summary, section "Main Findings" (recall and
                    relative L1 of the selectors at matched density).
* [ai.info/Future]  ai.info AI summary, section "Future Directions" (a
                    comparison with low-precision attention left open).
* [OFP8]            the OCP 8-bit floating point specification, format E4M3
                    (not one of the pages: it defines the bytes of an fp8
                    K/V cache).

Readings taken where the pages are silent (each repeated at its function):
softmax scale 1/sqrt(D); natural-log LSE; PDDP centred covariance, power
iteration from (1,..,1)/sqrt(D) for ``iters`` steps, sign fixed by the largest
|component| (lowest index on ties); median split at rank C*floor(g/2) with ties
broken by token index; leaves in tree order (left first), ascending inside a
leaf, the one short leaf (when C does not divide N) last and padded with -1;
top-K ties to the lower KV index, result ascending; sparse softmax
renormalised over the selected K only; the residual is taken against the
stored bf16 dense output and stored as bf16.

Parity status: every function here is pinned by tests in
``tests/test_oracle_pins.py`` (closed forms, library routines, brute force,
invariants); none is "parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "round_to_bf16",
    "default_scale",
    "dense_attention",
    "principal_direction",
    "pddp_leaves",
    "pddp_perm",
    "group_members",
    "group_mass",
    "topk_select",
    "per_query_topk_mass",
    "sparse_attention",
    "sparse_attention_group",
    "anchor_step",
    "reuse_step",
    "block_topk_select",
    "pooled_block_select",
    "per_query_select",
    "retained_mass",
    "rel_l1",
    "e4m3_decode",
    "e4m3_encode",
    "sparse_attention_e4m3",
]


# ---------------------------------------------------------------------------
# bf16 storage rounding
# ---------------------------------------------------------------------------

def round_to_bf16(x) -> np.ndarray:
    """Round real values to the nearest bfloat16 (ties to even), as float64.

    bfloat16 keeps 8 significant bits and the float32 exponent range.  For
    x = m * 2**e with 0.5 <= |m| < 1 the spacing of bf16 values around x is
    2**(e-8); below the smallest normal (e < -125) the spacing stays 2**-133.
    ``np.rint`` rounds half-way cases to even.  Values beyond the bf16 range do
    not occur here and are not handled.
    """
    a = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(a)
    e = np.maximum(e, -125)
    ulp = np.ldexp(1.0, e - 8)
    return np.rint(a / ulp) * ulp


def default_scale(D: int) -> float:
    """Softmax temperature.  The pages do not state it; standard attention
    uses 1/sqrt(D), and that is the reading taken."""
    return 1.0 / math.sqrt(D)


# ---------------------------------------------------------------------------
# a2: dense attention with log-sum-exp  [ai.info/Method], [agihunt/Select]
# ---------------------------------------------------------------------------

def dense_attention(q, k, v, scale, rows=None):
    """Dense softmax attention of one head, plus the per-query log-sum-exp.

    The selector's first pass "computes the dense output and row-wise
    log-sum-exp values" [ai.info/Method].  With S = scale * q k^T:
        lse_i = log sum_j exp(S_ij)            (natural log; reading)
        O_i   = sum_j exp(S_ij - lse_i) v_j
    ``rows`` restricts the computation to some query rows (each row is
    independent of the others).  Returns (O [r, D], lse [r]).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    if rows is not None:
        q = q[np.asarray(rows)]
    S = scale * (q @ k.T)
    m = S.max(axis=1)
    lse = m + np.log(np.exp(S - m[:, None]).sum(axis=1))
    P = np.exp(S - lse[:, None])
    return P @ v, lse


# ---------------------------------------------------------------------------
# a1: Fast PDDP median-split grouping  [wisp/Tile], [ai.info/Method],
#     [ai.info/Contrib], [agihunt/Group]
# ---------------------------------------------------------------------------

def principal_direction(cov, iters: int):
    """Leading eigenvector of a covariance matrix by power iteration.

    The pages name batched power iteration as the way the principal direction
    is found [ai.info/Contrib]; start vector, step count and sign are not
    given.  Reading: start at (1,...,1)/sqrt(D), apply v <- Cv/|Cv| ``iters``
    times (stop early only if Cv is exactly zero, i.e. a degenerate node),
    then flip the sign so that the component of largest magnitude is
    positive (the lowest such index on ties).
    """
    cov = np.asarray(cov, np.float64)
    D = cov.shape[0]
    v = np.full(D, 1.0 / math.sqrt(D))
    for _ in range(iters):
        w = cov @ v
        norm = math.sqrt(float(w @ w))
        if norm == 0.0:
            break
        v = w / norm
    lead = int(np.argmax(np.abs(v)))  # argmax returns the first maximum
    if v[lead] < 0:
        v = -v
    return v


def pddp_leaves(x, C: int, iters: int = 32):
    """Median-split principal direction divisive partitioning of one head.

    Each node is projected onto its principal direction and the ordered
    queries are split at the median, recursively, until every group holds C
    queries [wisp/Tile], [agihunt/Group].  The pages assume C divides the
    node; for a node of n rows, g = ceil(n / C) groups, the reading taken is:
    the left child receives the C*floor(g/2) rows of smallest projection and
    the right child the rest, so the only short group is the right-most leaf.

    Per node: mu = mean, Cov = sum_i (x_i - mu)(x_i - mu)^T, v = leading
    direction (``principal_direction``), t_i = (x_i - mu).v, order rows by
    (t_i, token index) ascending, split, recurse left then right.

    Returns the leaves left to right, each an ascending int64 array of token
    indices.
    """
    x = np.asarray(x, np.float64)
    N = x.shape[0]
    leaves = []

    def split(members):
        n = members.shape[0]
        g = -(-n // C)
        if g <= 1:
            leaves.append(np.sort(members))
            return
        xs = x[members]
        mu = xs.mean(axis=0)
        xc = xs - mu
        cov = xc.T @ xc
        v = principal_direction(cov, iters)
        t = xc @ v
        order = np.lexsort((members, t))  # primary key t, then token index
        n_left = C * (g // 2)
        split(members[order[:n_left]])
        split(members[order[n_left:]])

    split(np.arange(N, dtype=np.int64))
    return leaves


def pddp_perm(x, C: int, iters: int = 32):
    """PDDP groups as the padded permutation array ``[G*C]`` (int64).

    Group g occupies positions [g*C, (g+1)*C); entry p holds the original
    token index at that position; unused slots of the short last group are
    -1.  G = ceil(N / C).
    """
    N = np.asarray(x).shape[0]
    G = -(-N // C)
    perm = np.full(G * C, -1, dtype=np.int64)
    for g, leaf in enumerate(pddp_leaves(x, C, iters)):
        perm[g * C: g * C + leaf.shape[0]] = leaf
    return perm


def group_members(perm, g: int, C: int):
    """Token indices of group g in a padded permutation (padding dropped)."""
    seg = np.asarray(perm)[g * C:(g + 1) * C]
    return seg[seg >= 0]


# ---------------------------------------------------------------------------
# a3 + a4: exact group mass and top-K  [agihunt/Select], [ai.info/Method]
# ---------------------------------------------------------------------------

def group_mass(q, k, lse, members, scale):
    """Attention mass a query group puts on every KV token.

    The second selector pass recomputes QK scores and recovers the exact
    attention probabilities from the first pass's LSE [ai.info/Method]:
        P_ij = exp(scale * q_i.k_j - lse_i)        (full-row softmax)
        mass[j] = sum_{i in group} P_ij
    Returns mass over all N KV tokens.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    lse = np.asarray(lse, np.float64)
    members = np.asarray(members)
    S = scale * (q[members] @ k.T)
    return np.exp(S - lse[members][:, None]).sum(axis=0)


def topk_select(mass, K: int):
    """The K KV tokens of largest group mass, returned ascending.

    The objective is the K KV tokens whose summed group attention weight is
    largest [agihunt/Select].  Ties (equal mass) go to the lower token index
    (reading).  Returns (idx ascending int64 [K], retained mass = sum of the
    selected masses).
    """
    mass = np.asarray(mass, np.float64)
    n = mass.shape[0]
    order = np.lexsort((np.arange(n), -mass))  # mass descending, then index
    idx = np.sort(order[:K])
    return idx, float(mass[idx].sum())


def per_query_topk_mass(q, k, lse, rows, K: int, scale):
    """The per-query oracle: each query keeps its own K most probable KV
    tokens; returns the kept probability mass per query.  Summed over a group
    it bounds from above what any shared selection of K tokens can retain
    [wisp/Gap], [ai.info/Method]."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    lse = np.asarray(lse, np.float64)
    rows = np.asarray(rows)
    P = np.exp(scale * (q[rows] @ k.T) - lse[rows][:, None])
    P.sort(axis=1)
    return P[:, -K:].sum(axis=1)


# ---------------------------------------------------------------------------
# a5: token-sparse attention  [wisp/Tile], [ai.info/Method], [agihunt/Group]
# ---------------------------------------------------------------------------

def sparse_attention_group(q, k, v, members, idx, scale):
    """Attention of one query group restricted to its selected KV tokens.

    The group's queries attend only to the gathered rows idx of K and V
    [wisp/Tile]; the softmax is renormalised over those K tokens (reading:
    the discarded tail is what the residual accounts for [wisp/Residual]).
    Returns O' [|group|, D].
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    members = np.asarray(members)
    idx = np.asarray(idx)
    S = scale * (q[members] @ k[idx].T)
    m = S.max(axis=1)
    P = np.exp(S - m[:, None])
    P /= P.sum(axis=1)[:, None]
    return P @ v[idx]


def sparse_attention(q, k, v, perm, idx, C: int, scale, groups=None):
    """Token-sparse attention of one head, in original token order.

    ``idx`` is ``[G, K]``.  Rows of tokens outside the requested ``groups``
    are left as NaN.  Returns O' [N, D].
    """
    q = np.asarray(q, np.float64)
    N, D = q.shape
    idx = np.asarray(idx)
    G = idx.shape[0]
    out = np.full((N, np.asarray(v).shape[1]), np.nan)
    for g in (range(G) if groups is None else groups):
        members = group_members(perm, g, C)
        if members.shape[0]:
            out[members] = sparse_attention_group(q, k, v, members, idx[g], scale)
    return out


# ---------------------------------------------------------------------------
# Anchor and reuse steps  [wisp/Reuse], [wisp/Residual]
# ---------------------------------------------------------------------------

def anchor_step(q, k, v, C: int, K: int, scale, iters: int = 32):
    """Everything one anchor step computes for one head.

    At an anchor the method groups the queries, selects KV tokens with exact
    probabilities, outputs dense attention, and records the residual between
    the dense and the sparse outputs [wisp/Reuse], [wisp/Residual].  Data
    flow (reading): the dense output is stored as bf16; the residual is
    ``bf16(dense_bf16 - O')`` with O' the sparse output under the new groups
    and indices.

    Returns a dict with perm [G*C], lse [N], dense (fp64), dense_bf16,
    mass [G, N], idx [G, K], retained [G], sparse (fp64 O'), residual (bf16
    values).
    """
    q = np.asarray(q, np.float64)
    N = q.shape[0]
    G = -(-N // C)
    perm = pddp_perm(q, C, iters)
    dense, lse = dense_attention(q, k, v, scale)
    mass = np.empty((G, N))
    idx = np.empty((G, K), dtype=np.int64)
    retained = np.empty(G)
    for g in range(G):
        mass[g] = group_mass(q, k, lse, group_members(perm, g, C), scale)
        idx[g], retained[g] = topk_select(mass[g], K)
    sparse = sparse_attention(q, k, v, perm, idx, C, scale)
    dense_bf16 = round_to_bf16(dense)
    residual = round_to_bf16(dense_bf16 - sparse)
    return dict(perm=perm, lse=lse, dense=dense, dense_bf16=dense_bf16,
                mass=mass, idx=idx, retained=retained, sparse=sparse,
                residual=residual)


def reuse_step(q, k, v, perm, idx, residual, C: int, scale, groups=None):
    """Output of a reuse step for one head: the current step's sparse
    attention under the cached groups and indices, plus the cached residual
    [wisp/Residual].  Returns the exact (fp64) sum; the stored output is its
    bf16 rounding.  ``groups`` restricts the work to some groups, as in
    ``sparse_attention`` (rows of other groups are NaN)."""
    sparse = sparse_attention(q, k, v, perm, idx, C, scale, groups=groups)
    return sparse + np.asarray(residual, np.float64)


# ---------------------------------------------------------------------------
# Diagnostic selectors  [wisp/Gap], [ai.info/Method], [wisp/Pool], [ai.info/Find]
# ---------------------------------------------------------------------------
# The pages separate the dense-sparse gap by comparing selectors that keep
# the same number of KV tokens: mean-pooled block-sparse attention (vanilla
# BSA), a block oracle (whole KV blocks, chosen with the exact probabilities),
# the token oracle (individual KV tokens shared by a query group: the exact
# group-mass selection above) and a per-query oracle (every query its own KV
# tokens).  Readings: KV blocks are the full blocks [b*block, (b+1)*block);
# the partial block at the end of the sequence (when block does not divide N)
# is never selected; K must be a multiple of block; ties go to the lower block
# (or token) index and results are ascending.

def _full_blocks(N: int, K: int, block: int) -> int:
    if block < 1 or K % block != 0 or K // block > N // block or K < 1:
        raise ValueError("K must be a positive multiple of block, at most N // block blocks")
    return N // block


def block_topk_select(mass, K: int, block: int):
    """Block oracle for one group: the K/block full KV blocks of largest
    summed group mass, expanded to their tokens (ascending).  Returns
    (idx [K], retained mass)  [wisp/Gap], [ai.info/Method]."""
    mass = np.asarray(mass, np.float64)
    nb = _full_blocks(mass.shape[0], K, block)
    bm = mass[:nb * block].reshape(nb, block).sum(axis=1)
    order = np.lexsort((np.arange(nb), -bm))
    blocks = np.sort(order[:K // block])
    idx = (blocks[:, None] * block + np.arange(block)[None, :]).ravel()
    return idx, float(mass[idx].sum())


def pooled_block_select(q, k, members, K: int, block: int, scale):
    """Vanilla BSA selection for one query group: each full KV block is
    scored by the dot product of the group's mean query with the block's mean
    key (times the softmax scale), and the K/block best blocks are kept,
    expanded to their tokens (ascending)  [wisp/Pool].  Returns (idx [K],
    scores [N // block])."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    N, D = k.shape
    nb = _full_blocks(N, K, block)
    qbar = q[np.asarray(members)].mean(axis=0)
    kbar = k[:nb * block].reshape(nb, block, D).mean(axis=1)
    score = scale * (kbar @ qbar)
    order = np.lexsort((np.arange(nb), -score))
    blocks = np.sort(order[:K // block])
    idx = (blocks[:, None] * block + np.arange(block)[None, :]).ravel()
    return idx, score


def per_query_select(q, k, lse, row: int, K: int, scale):
    """Per-query oracle for one query: its own K most probable KV tokens
    (ties to the lower index, ascending) and the probability mass they keep
    [wisp/Gap], [ai.info/Method].  Equivalent to topk_select on the
    probabilities of a one-query group."""
    p = np.exp(scale * (np.asarray(k, np.float64) @ np.asarray(q, np.float64)[row])
               - float(np.asarray(lse, np.float64)[row]))
    return topk_select(p, K)


def retained_mass(mass, idx) -> float:
    """Mass a selection keeps: the sum of the group masses at idx.  Divided
    by the group size it is the group's attention recall [ai.info/Find]."""
    return float(np.asarray(mass, np.float64)[np.asarray(idx)].sum())


def rel_l1(got, want) -> float:
    """Relative L1 error of an output, sum |got - want| / sum |want|
    [ai.info/Find]."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return float(np.abs(got - want).sum() / np.abs(want).sum())


# ---------------------------------------------------------------------------
# fp8 (E4M3) K/V cache  [ai.info/Future], [OFP8]
# ---------------------------------------------------------------------------
# The pages leave attention over low-precision K/V open [ai.info/Future].  The
# library can hold K and V as E4M3 bytes with one scale per tensor:
# k = k_scale * decode(k8).  E4M3 [OFP8]: sign bit, 4 exponent bits (bias 7),
# 3 mantissa bits; exponent field 0 holds the subnormals m * 2**-9; no
# infinities; S.1111.111 is NaN, so the largest finite magnitude is
# 1.75 * 2**8 = 448.  Readings: a value is divided by its scale in float32
# (one correctly rounded division), rounded to the nearest E4M3 value with
# ties to the even mantissa, and magnitudes above 448 saturate to 448; NaN
# becomes the code 0x7F.

def e4m3_decode(codes) -> np.ndarray:
    """Values of E4M3 codes (uint8), as float64 (NaN for the NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(x, scale: float) -> np.ndarray:
    """E4M3 codes of x / scale: the quotient taken in float32, then rounded to
    the nearest E4M3 value (ties to even), saturating at +-448."""
    r = np.asarray(x, dtype=np.float32) / np.float32(scale)
    a = np.abs(r).astype(np.float64)
    sign = np.signbit(r).astype(np.int64) << 7
    code = np.zeros(a.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    # subnormal range: multiples of 2**-9; 8 * 2**-9 is the smallest normal,
    # whose code (exponent 1, mantissa 0) is also 8
    code[sub] = np.rint(a[sub] / 2.0 ** -9).astype(np.int64)
    nrm = ~sub & (a < 448.0)
    _, e2 = np.frexp(a[nrm])            # a = f * 2**e2, 0.5 <= f < 1
    e = e2 - 1                          # a in [2**e, 2**(e+1))
    m = np.rint(a[nrm] / np.ldexp(1.0, e - 3)).astype(np.int64)  # 8 .. 16
    up = m == 16
    e = np.where(up, e + 1, e)
    m = np.where(up, 8, m)
    code[nrm] = np.minimum(((e + 7) << 3) | (m - 8), 0x7E)
    code[~sub & ~nrm] = 0x7E            # >= 448: saturate
    code = code | sign
    code[np.isnan(r)] = 0x7F
    return code.astype(np.uint8)


def sparse_attention_e4m3(q, k8, v8, k_scale: float, v_scale: float, perm, idx, C: int,
                          scale, groups=None):
    """Token-sparse attention of one head over an E4M3 K/V cache: the method's
    sparse attention [wisp/Tile] applied to the values the bytes stand for,
    k = k_scale * decode(k8) and v = v_scale * decode(v8) [ai.info/Future]."""
    k = k_scale * e4m3_decode(k8)
    v = v_scale * e4m3_decode(v8)
    return sparse_attention(q, k, v, perm, idx, C, scale, groups=groups)

"""Shared tolerances, error measures and input cases for the parity tests.

Tolerances (floating point) are the ones the target states: outputs within
max abs error 1e-2 and mean relative error 2e-3, group mass within 1e-4
relative, selected index sets equal except for ties within 1e-5 relative of
the K-th mass.  "Mean relative error" is read as sum|got - want| /
sum|want| over the compared elements.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import mcs_oracle as orc
from token_sparse_attention_gb300 import synth

MAX_ABS = 1e-2
MEAN_REL = 2e-3
MASS_REL = 1e-4
TIE_REL = 1e-5
LSE_ABS = 1e-3


def f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, np.float64)


def err(got, want):
    got, want = f64(got), f64(want)
    d = np.abs(got - want)
    return float(d.max()), float(d.sum() / max(np.abs(want).sum(), 1e-300))


def assert_close(got, want, what="output", max_abs=MAX_ABS, mean_rel=MEAN_REL):
    ma, mr = err(got, want)
    assert ma <= max_abs and mr <= mean_rel, f"{what}: max abs {ma:.3g}, mean rel {mr:.3g}"
    return ma, mr


def bf16_tensor(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).to(device)


def random_qkv(B, H, N, D, seed):
    """bf16 Q, K, V with the workloads' structure (Fourier features of token
    positions; see synth.make_qkv_like) for an arbitrary size.  Pure Gaussian
    V would make every output an average of unrelated vectors, so small that
    bf16 output rounding alone (~1.4e-3 mean relative) eats most of the
    2e-3 budget; the workloads' V does not behave like that."""
    return synth.make_qkv_like(B, H, N, D, seed)


def random_groups(N, C, seed):
    """A random grouping in the padded perm layout (ascending inside groups)."""
    rng = np.random.default_rng(seed)
    G = -(-N // C)
    order = rng.permutation(N)
    perm = np.full(G * C, -1, dtype=np.int64)
    for g in range(G):
        seg = np.sort(order[g * C:(g + 1) * C])
        perm[g * C:g * C + seg.shape[0]] = seg
    return perm


def random_idx(N, G, K, seed):
    rng = np.random.default_rng(seed)
    return np.stack([np.sort(rng.choice(N, size=K, replace=False)) for _ in range(G)])


def separated_clusters(N, C, D, seed, jitter=2e-3):
    """Points in ceil(N/C) tight clusters whose sizes follow the split rule
    (left child C*floor(g/2) rows, the short group right-most).  A node at
    depth d splits along its own axis with the smaller child at -s_d and the
    larger at +s_d, s_d = 4 * 0.6**d, so each node's principal direction is
    its split axis and the median split recovers the clusters exactly.
    Returns (x [N, D] float64 holding bf16 values, expected padded perm)."""
    rng = np.random.default_rng(seed)
    G = -(-N // C)
    axes = rng.permutation(D)
    centre_of = {}

    def walk(start, n, depth, centre):
        g = -(-n // C)
        if g <= 1:
            centre_of[start] = (n, centre)
            return
        nl = C * (g // 2)
        s = 4.0 * 0.6 ** depth
        a = axes[depth % D]
        cl, cr = centre.copy(), centre.copy()
        cl[a] -= s
        cr[a] += s
        walk(start, nl, depth + 1, cl)
        walk(start + nl, n - nl, depth + 1, cr)

    walk(0, N, 0, np.zeros(D))
    tokens = rng.permutation(N)
    x = np.empty((N, D))
    want = np.full(G * C, -1, dtype=np.int64)
    for g, start in enumerate(sorted(centre_of)):
        n, centre = centre_of[start]
        members = tokens[start:start + n]
        x[members] = centre + jitter * rng.standard_normal((n, D))
        want[g * C:g * C + n] = np.sort(members)
    return orc.round_to_bf16(x), want


def check_valid_perm(perm, N, C):
    """perm [G*C]: a permutation of 0..N-1 in groups of C (the short one last,
    padded with -1), ascending inside each group."""
    perm = np.asarray(perm)
    G = -(-N // C)
    assert perm.shape == (G * C,)
    real = perm[perm >= 0]
    assert np.array_equal(np.sort(real), np.arange(N)), "not a permutation"
    for g in range(G):
        seg = perm[g * C:(g + 1) * C]
        n_real = C if g < G - 1 else N - (G - 1) * C
        assert np.all(seg[:n_real] >= 0) and np.all(seg[n_real:] == -1), f"group {g} size"
        assert np.all(np.diff(seg[:n_real]) > 0), f"group {g} not ascending"


def assert_topk_within_ties(got_idx, want_idx, mass, K):
    """Index sets equal except where the differing tokens' masses lie within
    TIE_REL (relative) of the K-th largest mass."""
    got, want = set(np.asarray(got_idx).tolist()), set(np.asarray(want_idx).tolist())
    if got == want:
        return 0
    kth = np.sort(np.asarray(mass))[::-1][K - 1]
    diff = np.array(sorted(got ^ want))
    assert np.all(np.abs(mass[diff] - kth) <= TIE_REL * abs(kth) + 1e-30), \
        f"top-K differs beyond ties: {diff[:8]} masses {mass[diff][:8]} kth {kth}"
    return len(diff) // 2

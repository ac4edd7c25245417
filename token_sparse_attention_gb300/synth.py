"""Seeded synthetic inputs shaped like the workloads MC-Sparse is measured on.

The pages measure on activations of video and 3D-asset diffusion transformers
(Wan2.1, HunyuanVideo, HY3D-Internal); neither those models nor their
activations exist here.  This module stands in for them with queries, keys
and values of the same shapes built from random Fourier features of token
positions, so that nearby tokens attend to each other and the softmax is
peaked the way the pages' recall figures imply.

This module holds input generation only: no attention, selection or grouping
arithmetic.  The library, the tests, the benchmark and the oracle all draw
their inputs from here.

Recipe for one (config c, step t):

1. positions: a normalised (t, y, x) video grid, or, for the 3D workload,
   Fibonacci-sphere points pushed along the normal by 3 octaves of random
   sinusoidal noise;
2. features phi(p) = [cos(2 pi W p), sin(2 pi W p)] with W ~ N(0, 4^2),
   16 frequencies (32 features);
3. per head and per tensor X in {Q, K, V}: X = phi A_X + N(0, 0.3^2) noise,
   A_X ~ N(0, 1/32); Q and K are then standardised per head to unit
   per-element standard deviation (V is not);
4. drift: at step t >= 1 each of the three standardised tensors receives
   N(0, sigma_d^2) noise on top of step t-1 (a random walk);
5. peaking: Q is multiplied by alpha (a per-config constant, below).

Seeds: frequencies and projections use 1000*c + 7, the 3D surface noise
1000*c + 8; the noise of tensor
X (0, 1, 2 for Q, K, V) at step t uses 1000*c + 10*t + X; each head draws from
its own stream seeded ``seed * 4096 + head`` so that any subset of heads can
be generated on its own.
"""

from __future__ import annotations

import dataclasses
import math

import torch

__all__ = ["Workload", "WORKLOADS", "workload", "make_qkv", "make_qkv_like", "positions"]


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload.  ``index`` numbers it for the seed scheme."""

    name: str
    index: int
    B: int
    H: int
    D: int
    C: int
    densities: tuple
    drift: float
    steps: int
    anchors: tuple
    grid: tuple | None = None  # (T, Y, X) video grid
    points: int | None = None  # 3D surface points
    alpha: float = 1.0

    @property
    def N(self) -> int:
        if self.grid is not None:
            t, y, x = self.grid
            return t * y * x
        return int(self.points)

    @property
    def G(self) -> int:
        return -(-self.N // self.C)

    def K(self, density: float) -> int:
        """Selected KV tokens per group: round(density * N), at least 1."""
        return max(1, min(self.N, int(round(density * self.N))))


# alpha: the factor on Q that makes the mean per-query mass of the 20% most
# probable keys about 0.95 at step 0 (the per-query recall level the pages
# report at density 0.2).  Values were found by bisection with
# oracle/calibrate_alpha.py on 256 queries of heads 0 and 1 of each workload.
_ALPHA = {
    "tiny": 2.6637,
    "small": 2.7102,
    "large": 2.6979,
    "long": 2.6941,
    "asset3d": 2.6973,
}

WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny", 1, B=1, H=2, D=128, C=64, densities=(0.2,), drift=0.05,
                 steps=2, anchors=(0,), grid=(8, 16, 16)),
        Workload("small", 2, B=1, H=12, D=128, C=128, densities=(0.1, 0.2, 0.3),
                 drift=0.03, steps=5, anchors=(0,), grid=(21, 39, 40)),
        Workload("large", 3, B=1, H=40, D=128, C=128, densities=(0.2,), drift=0.03,
                 steps=1, anchors=(0,), grid=(21, 60, 60)),
        Workload("long", 4, B=1, H=24, D=128, C=128, densities=(0.15, 0.25),
                 drift=0.03, steps=10, anchors=(0, 5), grid=(33, 60, 60)),
        Workload("asset3d", 5, B=1, H=16, D=64, C=64, densities=(0.15,), drift=0.03,
                 steps=5, anchors=(0,), points=65536),
    )
}


def workload(name: str) -> Workload:
    w = WORKLOADS[name]
    return dataclasses.replace(w, alpha=_ALPHA[name])


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def positions(w: Workload, device="cpu") -> torch.Tensor:
    """Token positions [N, 3] in float32."""
    if w.grid is not None:
        T, Y, X = w.grid
        axes = [torch.linspace(0.0, 1.0, n, device=device) if n > 1
                else torch.zeros(1, device=device) for n in (T, Y, X)]
        t, y, x = torch.meshgrid(*axes, indexing="ij")
        return torch.stack([t, y, x], dim=-1).reshape(-1, 3)
    n = w.N
    g = _gen(1000 * w.index + 8, device)
    i = torch.arange(n, dtype=torch.float64, device=device) + 0.5
    z = 1.0 - 2.0 * i / n
    r = torch.sqrt(torch.clamp(1.0 - z * z, min=0.0))
    phi = math.pi * (3.0 - math.sqrt(5.0)) * i
    p = torch.stack([r * torch.cos(phi), r * torch.sin(phi), z], dim=-1)
    radius = torch.ones(n, dtype=torch.float64, device=device)
    for octave in range(3):
        freq = 4.0 * 2.0 ** octave
        dirs = torch.randn(8, 3, generator=g, device=device, dtype=torch.float64)
        dirs = dirs / dirs.norm(dim=1, keepdim=True)
        phase = 2 * math.pi * torch.rand(8, generator=g, device=device, dtype=torch.float64)
        noise = torch.sin(2 * math.pi * freq * (p @ dirs.T) + phase).mean(dim=1)
        radius = radius + 0.5 ** (octave + 1) * noise
    return (p * radius[:, None]).to(torch.float32)


def _features(w: Workload, device) -> tuple[torch.Tensor, torch.Generator]:
    g = _gen(1000 * w.index + 7, device)
    pos = positions(w, device)
    omega = 4.0 * torch.randn(16, 3, generator=g, device=device)
    ang = 2 * math.pi * (pos @ omega.T)
    return torch.cat([torch.cos(ang), torch.sin(ang)], dim=1), g


def make_qkv(w: Workload, step: int = 0, heads=None, device="cpu",
             dtype=torch.bfloat16, alpha: float | None = None):
    """Q, K, V of shape [B, H', N, D] for the given heads (default: all B*H,
    numbered b*H + h) at the given denoising step.

    ``alpha`` overrides the workload's Q scale (used by the calibration
    script, which needs pre-scaling queries).
    """
    BH = w.B * w.H
    heads = list(range(BH)) if heads is None else list(heads)
    a = w.alpha if alpha is None else alpha
    phi, g = _features(w, device)
    proj = torch.randn(BH, 3, 32, w.D, generator=g, device=device) / math.sqrt(32.0)
    out = [torch.empty(len(heads), w.N, w.D, dtype=dtype, device=device) for _ in range(3)]
    for slot, bh in enumerate(heads):
        for x in range(3):
            base = phi @ proj[bh, x]
            gn = _gen((1000 * w.index + x) * 4096 + bh, device)
            t = base + 0.3 * torch.randn(base.shape, generator=gn, device=device)
            if x < 2:
                t = t / t.std()
            for s in range(1, step + 1):
                gd = _gen((1000 * w.index + 10 * s + x) * 4096 + bh, device)
                t = t + w.drift * torch.randn(t.shape, generator=gd, device=device)
            if x == 0:
                t = t * a
            out[x][slot] = t.to(dtype)
    B = w.B if len(heads) == BH else 1
    return tuple(o.reshape(B, -1, w.N, w.D) for o in out)


def make_qkv_like(B: int, H: int, N: int, D: int, seed: int, alpha: float = 2.7,
                  device="cpu", dtype=torch.bfloat16):
    """Q, K, V [B, H, N, D] for an arbitrary token count, built like the
    workloads above (Fourier features of positions, per-head projections,
    N(0, 0.3^2) noise, Q and K standardised, Q scaled by alpha) but with the
    N positions drawn uniformly in the unit cube.  For small parity cases."""
    g = _gen(seed, device)
    pos = torch.rand(N, 3, generator=g, device=device)
    omega = 4.0 * torch.randn(16, 3, generator=g, device=device)
    ang = 2 * math.pi * (pos @ omega.T)
    phi = torch.cat([torch.cos(ang), torch.sin(ang)], dim=1)
    out = []
    for x in range(3):
        proj = torch.randn(B * H, 32, D, generator=g, device=device) / math.sqrt(32.0)
        t = phi[None] @ proj + 0.3 * torch.randn(B * H, N, D, generator=g, device=device)
        if x < 2:
            t = t / t.std(dim=(1, 2), keepdim=True)
        if x == 0:
            t = t * alpha
        out.append(t.reshape(B, H, N, D).to(dtype))
    return tuple(out)

"""Find each workload's Q scale alpha (test infrastructure).

alpha is chosen so that, at step 0, the mean over sampled queries of the
probability mass held by each query's own 20% most probable keys is 0.95: the
per-query recall level reported for density 0.2 (ai.info AI summary, "Main
Findings", token-granularity recall of the per-query oracle).  It calls only
the oracle and the input generator; the printed values are copied into
token_sparse_attention_gb300/synth.py.

Usage: python -m oracle.calibrate_alpha [workload ...]
"""

from __future__ import annotations

import math
import sys

import numpy as np
import torch

from oracle import mcs_oracle as orc
from token_sparse_attention_gb300 import synth

TARGET = 0.95


def mean_top20_mass(q, k, rows, alpha, scale):
    qa = orc.round_to_bf16(alpha * q)
    _, lse_rows = orc.dense_attention(qa, k, k, scale, rows=rows)
    lse = np.zeros(k.shape[0])
    lse[rows] = lse_rows
    K = max(1, int(round(0.2 * k.shape[0])))
    return float(orc.per_query_topk_mass(qa, k, lse, rows, K, scale).mean())


def calibrate(name: str, n_rows: int = 256) -> float:
    w = synth.workload(name)
    q, k, _ = synth.make_qkv(w, 0, heads=[0, 1], dtype=torch.float32, alpha=1.0)
    rng = np.random.default_rng(1234)
    scale = orc.default_scale(w.D)
    vals = []
    for h in range(2):
        qh = q[0, h].double().numpy()
        kh = orc.round_to_bf16(k[0, h].double().numpy())
        rows = np.sort(rng.choice(w.N, size=min(n_rows, w.N), replace=False))
        lo, hi = math.log(0.25), math.log(64.0)
        for _ in range(30):
            mid = 0.5 * (lo + hi)
            if mean_top20_mass(qh, kh, rows, math.exp(mid), scale) < TARGET:
                lo = mid
            else:
                hi = mid
        vals.append(math.exp(0.5 * (lo + hi)))
    return float(np.mean(vals))


if __name__ == "__main__":
    names = sys.argv[1:] or list(synth.WORKLOADS)
    for n in names:
        print(f'    "{n}": {calibrate(n):.4f},', flush=True)

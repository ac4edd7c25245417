#!/usr/bin/env python
"""Benchmark of the MC-Sparse hot path on GB300.

Metric: token-sparse attention effective TFLOP/s (4*B*H*N*K*D per pass,
real query rows only) and its speedup over this library's own dense
attention, on the large video workload: B=1, H=40, N=75600 (21x60x60 grid),
D=128, C=128, density 0.2 (K=15120), synthetic Fourier-feature inputs.

One timed step = the whole hot path on that workload: an anchor step on step-0
inputs (PDDP grouping, dense attention + LSE, exact group mass + top-K per
head chunk, sparse attention recording the residual) followed by a reuse step
on step-1 inputs (sparse attention + cached residual).  Inputs (0.77 GB per
tensor) are larger than L2, so no explicit flush is needed between steps.
`value` is the effective TFLOP/s of the reuse step's sparse attention, timed
with CUDA events around its launch inside every timed step; the dense time
that gives the speedup is timed the same way in the same steps.

`--impl reference` times the fp64 CPU oracle (the only reference that
exists for this method) on a bounded sample of the same workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mcs|reference]
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from token_sparse_attention_gb300 import synth  # noqa: E402

METRIC = "sparse-attn effective TFLOP/s & speedup vs own dense attn at N=75600, density 0.2"

# dram__bytes_read.sum + dram__bytes_write.sum per launch from ncu, with the
# sha1 of the kernel source it was measured on (traffic is reported only
# while the source is unchanged).
TRAFFIC = {
    # ncu dram bytes (read + write) of the sparse reuse launch, captured on the
    # 4-head large workload (the timed step's first reuse launch of `bench.py
    # --heads 4 --steps 1 --warmup 1 --no-e2e --no-cpu-baseline
    # --no-workloads --no-e4m3`), times 10 for the 40-head launch: heads are independent
    # and the grid scales with them
    "attn.cu": {"sha": "a02022ef129b", "bytes_per_launch": 7307924480},
}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


def reduce_max_over_ranks(vals, dist, device):
    """Max of each value over all ranks (every rank gets the result); the
    job's time is that of its slowest replica."""
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def depths_of(G: int) -> int:
    """Tree depths of the PDDP grouping: ceil(log2 G)."""
    return max(0, math.ceil(math.log2(G))) if G > 1 else 0


def pddp_launches(N: int, C: int) -> int:
    """Kernel launches of one mcs_group call: init, the table of splitting
    nodes (when there is a depth) and finalize, then per depth moments, power
    iteration, projection and the warp-per-node split, plus the chunk-partial
    reduction when a node has >= 4 chunks of 1024 rows and the block-per-node
    split when a node has > 1024 rows (pddp.cu)."""
    G = -(-N // C)
    nodes, count = [N], 2 + (1 if depths_of(G) > 0 else 0)
    for _ in range(depths_of(G)):
        mx = max(nodes)
        count += 4 + (1 if -(-mx // 1024) >= 4 else 0) + (1 if mx > 1024 else 0)
        nxt = []
        for n in nodes:
            g = -(-n // C)
            if g <= 1:
                nxt.append(n)
            else:
                nxt += [C * (g // 2), n - C * (g // 2)]
        nodes = nxt
    return count


def pddp_bytes(BH: int, N: int, D: int, G: int) -> float:
    """Algorithmic HBM bytes of the PDDP grouping: per depth, every head's
    rows read twice (moments and projection, bf16) plus the index traffic
    (positions read, keys written and read back, 4 bytes each)."""
    return depths_of(G) * (2 * 2.0 * BH * N * D + 3 * 4.0 * BH * N)


def sum_over_ranks(x, dist, device):
    """Sum of one number over all ranks (every rank gets the result)."""
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return t.item()


def job_tflops(world: int, flops_per_replica: float, ms: float) -> float:
    """Whole-job throughput of `world` independent replicas that each do
    flops_per_replica in `ms` (the max over ranks): weak scaling."""
    return world * flops_per_replica / (ms * 1e-3) / 1e12


def _src_sha(name: str) -> str:
    with open(os.path.join(ROOT, "token_sparse_attention_gb300", "csrc", name), "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()[:12]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        # nvidia-smi numbers GPUs physically; address ours by UUID
        try:
            self.index = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            self.index = vis.split(",")[device] if vis else str(device)
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- reference arm

def oracle_setup(w, K, n_groups=32, seed=99):
    """A bounded sample of the workload for the oracle: head 0, its oracle
    PDDP groups at step 0, the first, the last and random groups with their
    oracle top-K selections; the timed part runs on step-1 inputs."""
    import numpy as np

    from oracle import mcs_oracle as orc

    q0, k0, v0 = (t[0, 0].double().numpy() for t in synth.make_qkv(w, 0, heads=[0]))
    q1, k1, v1 = (t[0, 0].double().numpy() for t in synth.make_qkv(w, 1, heads=[0]))
    scale = orc.default_scale(w.D)
    perm = orc.pddp_perm(q0, w.C, 32)
    rng = np.random.default_rng(seed)
    G = w.G
    groups = [0, G - 1] + list(rng.choice(np.arange(1, G - 1), size=n_groups - 2, replace=False))
    sel = []
    for g in groups:
        m = orc.group_members(perm, g, w.C)
        _, l = orc.dense_attention(q0, k0, v0, scale, rows=m)
        lse = np.zeros(w.N)
        lse[m] = l
        sel.append((m, orc.topk_select(orc.group_mass(q0, k0, lse, m, scale), K)[0]))
    return dict(q=q1, k=k1, v=v1, sel=sel, scale=scale, K=K, D=w.D, seed=seed)


def oracle_time(s, min_seconds):
    """Time the oracle's token-sparse attention over the sample, in passes
    until min_seconds have elapsed.  Returns (TFLOP/s, seconds, description)."""
    from oracle import mcs_oracle as orc

    flops, t0, passes = 0.0, time.perf_counter(), 0
    while True:
        for m, idx in s["sel"]:
            orc.sparse_attention_group(s["q"], s["k"], s["v"], m, idx, s["scale"])
            flops += 4.0 * m.shape[0] * s["K"] * s["D"]
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    n = len(s["sel"])
    desc = (f"oracle sparse attention on {n} groups of head 0 (first, last, {n - 2} random, "
            f"seed {s['seed']}) x {passes} passes, fp64 numpy")
    return flops / dt / 1e12, dt, desc


def workload_label(w, density, K) -> str:
    """The `config.workload` both arms print for the same run."""
    return f"{w.name} B={w.B} H={w.H} N={w.N} D={w.D} C={w.C} density {density} K={K}"


def run_reference(args, w, K, rank):
    if rank != 0:
        return
    cores = len(os.sched_getaffinity(0))
    sample = oracle_setup(w, K)
    vals = []
    for i in range(args.warmup + args.steps):
        v, dt, desc = oracle_time(sample, min_seconds=2.0)
        if i >= args.warmup:
            vals.append((v, dt))
    value = statistics.mean(v for v, _ in vals)
    ms = statistics.mean(dt for _, dt in vals) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_label(w, args.density, K),
                   "sample": "bounded sample per step"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm

def rank_heads(w, rank, world, split):
    """The problem a rank works on and the flattened heads it owns.

    weak:   the job is `world` copies of the workload's batch (global batch
            world * B); rank r owns flattened heads [r*B*H, (r+1)*B*H), so
            every rank's work equals the single-GPU workload.
    strong: the job is the workload itself; its B*H heads are split into
            contiguous ranges (shard.head_range).
    Returns (global workload, start, stop)."""
    from token_sparse_attention_gb300 import shard

    wg = dataclasses.replace(w, B=w.B * world) if split == "weak" else w
    h0, h1 = shard.head_range(rank, world, wg.B * wg.H)
    return wg, h0, h1


def run_gpu(args, w, K, rank, world, dist):
    from token_sparse_attention_gb300 import mcs

    mcs.lib()
    dev = torch.device("cuda", torch.cuda.current_device())
    layout = mcs.LAYOUT_BNHD if args.layout == "bnhd" else mcs.LAYOUT_BHND
    wg, h0, h1 = rank_heads(w, rank, world, args.split)
    heads = list(range(h0, h1))

    def lay(t):  # the generator writes [B,H,N,D]; DiT blocks hold [B,N,H,D]
        return t.transpose(1, 2).contiguous() if layout == mcs.LAYOUT_BNHD else t

    # this rank's heads only: [B, H, N, D] when it owns the whole batch,
    # else one batch of h1 - h0 heads
    q0, k0, v0 = (lay(t) for t in synth.make_qkv(wg, 0, heads=heads, device=dev))
    Bl, Hl = (q0.shape[0], q0.shape[2]) if layout == mcs.LAYOUT_BNHD else q0.shape[:2]
    p = mcs.params(Bl, Hl, w.N, w.D, w.C, K, layout=layout)
    G = p.G
    BH = Bl * Hl
    # the anchor's metadata serves the next R denoising steps, each with its
    # own inputs (the generator's steps 1..R)
    R = args.reuse_per_anchor
    reuse_in = [tuple(lay(t) for t in synth.make_qkv(wg, s_, heads=heads, device=dev))
                for s_ in range(1, R + 1)]
    q1, k1, v1 = reuse_in[0]
    perm = torch.empty(Bl, Hl, G * w.C, dtype=torch.int32, device=dev)
    idx = torch.empty(Bl, Hl, G, K, dtype=torch.int32, device=dev)
    dense = torch.empty_like(q0)
    lse = torch.empty(Bl, Hl, w.N, dtype=torch.float32, device=dev)
    res = torch.empty_like(q0)
    out = torch.empty_like(q0)
    retained = torch.empty(Bl, Hl, G, dtype=torch.float32, device=dev)
    ws_bytes = mcs.mcs_anchor_workspace(p)
    ws = mcs.empty_workspace(ws_bytes, dev)
    stream = torch.cuda.current_stream()
    stages = ["pddp", "dense", "select", "record"] + [f"reuse{r}" for r in range(R)]

    def step(ev):
        ev[0].record(stream)
        mcs.mcs_group(p, q0, perm, ws)
        ev[1].record(stream)
        mcs.mcs_dense_attn(p, q0, k0, v0, dense, lse)
        ev[2].record(stream)
        mcs.mcs_select(p, q0, k0, lse, perm, idx, ws, retained)
        ev[3].record(stream)
        mcs.mcs_sparse_attn_record(p, q0, k0, v0, perm, idx, dense, res)
        ev[4].record(stream)
        for r, (qr, kr, vr) in enumerate(reuse_in):
            mcs.mcs_sparse_attn(p, qr, kr, vr, perm, idx, res, out)
            ev[5 + r].record(stream)

    def new_events():
        return [torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]

    for _ in range(args.warmup):
        step(new_events())
    torch.cuda.synchronize()
    st = mcs.mcs_device_status()
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {mcs.mcs_status_string(st)}")

    evs = [new_events() for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        end.record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    total_ms = start.elapsed_time(end)
    stage_ms = {s: statistics.mean(e[k].elapsed_time(e[k + 1]) for e in evs)
                for k, s in enumerate(stages)}
    reuse_launch_ms = [stage_ms.pop(f"reuse{r}") for r in range(R)]
    stage_ms["reuse"] = statistics.mean(reuse_launch_ms)  # the metric's kernel
    st = mcs.mcs_device_status()
    if st != 0:
        raise RuntimeError(f"device status after timing: {mcs.mcs_status_string(st)}")

    # ---- end to end: pinned host inputs -> device, reuse-step sparse attention, result -> host
    # Every step copies its inputs from pinned host memory and reads its result
    # back, as a serving loop would; the steps are pipelined like one: two
    # device input sets, step i+1's host->device copies on a copy stream while
    # step i's kernel and read-back run on the compute stream.  The layer's
    # metadata from the anchor (perm, idx, residual: 1.0 GB here, 60 GB for
    # a 60-layer model) stays resident in HBM; a second run also stages it
    # from pinned host memory every step (the offload scheme of mcs_stager).
    e2e = None
    e2e_staged = None
    staging = None
    if not args.no_e2e:
        # The reuse step's inputs: Q, K, V from pinned host memory, and the
        # layer's cached metadata (perm, idx as bitmaps, residual) as one
        # entry staged by mcs_stager from pinned host memory into two device
        # slots, each step's entry prefetched two steps ahead (one step ahead
        # of the step that runs while it copies) and its index lists unpacked
        # on the device before the step's sparse attention.
        hq, hk, hv = (t.cpu().pin_memory() for t in (q1, k1, v1))
        meta_bytes = mcs.mcs_meta_bytes(p)
        slots = [torch.empty(meta_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
        views = [mcs.meta_views(p, sl) for sl in slots]
        views[0][0].copy_(perm)
        views[0][2].copy_(res)
        mcs.mcs_meta_pack(p, idx, slots[0])
        hentry = torch.empty(meta_bytes, dtype=torch.uint8, pin_memory=True)
        hentry.copy_(slots[0])
        didx = torch.empty_like(idx)
        hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        sets = [[torch.empty_like(t) for t in (q1, k1, v1)] for _ in range(2)]
        douts = [torch.empty_like(out) for _ in range(2)]
        host_in = (hq, hk, hv)
        h2d = sum(t.numel() * t.element_size() for t in host_in) + meta_bytes
        d2h = hout.numel() * hout.element_size()
        copy_stream, meta_stream, d2h_stream = (torch.cuda.Stream() for _ in range(3))
        stager = mcs.Stager(p, slots, meta_stream)
        loaded = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        read_back = [torch.cuda.Event() for _ in range(2)]

        def staged_run(n, with_qkv, stage_meta=True):
            for i in range(min(2, n) if stage_meta else 0):
                stager.prefetch(i, hentry, after=stream)
            for i in range(n):
                s = i % 2
                if with_qkv:
                    with torch.cuda.stream(copy_stream):
                        if i >= 2:
                            copy_stream.wait_event(consumed[s])  # set s free again
                        for dst, src in zip(sets[s], host_in):
                            dst.copy_(src, non_blocking=True)
                        loaded[s].record(copy_stream)
                    stream.wait_event(loaded[s])
                    dq, dk, dv = sets[s]
                else:
                    dq, dk, dv = q1, k1, v1
                if stage_meta:
                    stager.wait(s, stream)
                    dperm, _, dres = views[s]
                    mcs.mcs_meta_unpack(p, slots[s], didx, stream=stream)
                    sidx = didx
                else:
                    dperm, sidx, dres = perm, idx, res  # resident since the anchor
                if with_qkv and i >= 2:
                    stream.wait_event(read_back[s])  # output buffer s read back
                mcs.mcs_sparse_attn(p, dq, dk, dv, dperm, sidx, dres, douts[s], stream=stream)
                consumed[s].record(stream)
                if stage_meta and i + 2 < n:
                    stager.prefetch(s, hentry, after=stream)  # after this step read slot s
                if with_qkv:
                    # the result goes back to the host on its own stream, over
                    # the link's other direction, while the next step runs
                    computed[s].record(stream)
                    with torch.cuda.stream(d2h_stream):
                        d2h_stream.wait_event(computed[s])
                        hout.copy_(douts[s], non_blocking=True)
                        read_back[s].record(d2h_stream)

        def timed(with_qkv, stage_meta=True):
            staged_run(max(2, args.warmup), with_qkv, stage_meta)
            torch.cuda.synchronize()
            if dist is not None:
                dist.barrier()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            copy_stream.wait_stream(stream)  # the first copies start after `a`
            meta_stream.wait_stream(stream)
            d2h_stream.wait_stream(stream)
            staged_run(args.steps, with_qkv, stage_meta)
            stream.wait_stream(d2h_stream)
            b.record(stream)  # after the last read-back, which follows every copy
            torch.cuda.synchronize()
            return a.elapsed_time(b) / args.steps

        h2d_qkv = sum(t.numel() * t.element_size() for t in host_in)
        e2e = {"ms": timed(True, stage_meta=False), "h2d": h2d_qkv, "d2h": d2h}
        e2e_staged = {"ms": timed(True), "h2d": h2d, "d2h": d2h}
        staging = {"ms": timed(False), "bytes": meta_bytes}
        stager.close()
        if mcs.mcs_device_status() != 0:
            raise RuntimeError("device status after the end-to-end runs")

    # ---- max over ranks; FLOPs summed over ranks (head ranges may differ by one)
    total_ms, t_sparse, t_dense, e2e_ms, e2e_staged_ms, staged_ms = reduce_max_over_ranks(
        [total_ms, stage_ms["reuse"], stage_ms["dense"], e2e["ms"] if e2e else 0.0,
         e2e_staged["ms"] if e2e_staged else 0.0, staging["ms"] if staging else 0.0], dist, dev)
    job_heads = sum_over_ranks(BH, dist, dev)
    extra = None
    if world == 1 and not args.no_workloads:
        extra = run_schedules(dev)
    e4m3 = None
    if world == 1 and not args.no_e4m3:
        e4m3 = e4m3_pass(mcs, p, reuse_in, perm, idx, res, out, stream)
    if rank != 0:
        return

    flops_sparse = 4.0 * BH * w.N * K * w.D  # this rank's heads
    flops_dense = 4.0 * BH * w.N * w.N * w.D
    job_flops_sparse = 4.0 * job_heads * w.N * K * w.D
    value = job_flops_sparse / (t_sparse * 1e-3) / 1e12
    speedup = t_dense / t_sparse
    peaks, peak_kind = _peaks()
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    achieved = flops_sparse / (t_sparse * 1e-3) / 1e12
    tr = TRAFFIC.get("attn.cu")
    traffic = tr["bytes_per_launch"] if tr and tr["sha"] == _src_sha("attn.cu") else None

    def tflops(fl, ms):
        return fl / (ms * 1e-3) / 1e12

    kernels = {
        "sparse_attn(reuse)": {"ms": t_sparse, "tflops": tflops(flops_sparse, t_sparse),
                               "frac": tflops(flops_sparse, t_sparse) / peak},
        "sparse_attn(record)": {"ms": stage_ms["record"],
                                "tflops": tflops(flops_sparse, stage_ms["record"])},
        "dense_attn": {"ms": t_dense, "tflops": tflops(flops_dense, t_dense),
                       "frac": tflops(flops_dense, t_dense) / peak},
        "group_mass+topk": {"ms": stage_ms["select"],
                            "tflops_qk": tflops(flops_dense / 2, stage_ms["select"])},
        # algorithmic bytes per depth: Q read twice (moments, projection) and
        # the index traffic (perm read, keys written and read), 2-D x 2 + 3 x 4
        # bytes per token and head
        # the same reuse launches over an E4M3 K/V cache (outside the timed
        # step; None with --no-e4m3 or on several ranks)
        "sparse_attn_e4m3(reuse)": (
            dict(e4m3, tflops=tflops(flops_sparse, e4m3["ms"]),
                 frac=tflops(flops_sparse, e4m3["ms"]) / peak) if e4m3 else None),
        "pddp": {"ms": stage_ms["pddp"], "depths": depths_of(G),
                 "algorithmic_gb": pddp_bytes(BH, w.N, w.D, G) / 1e9,
                 "gbs": pddp_bytes(BH, w.N, w.D, G) / (stage_ms["pddp"] * 1e-3) / 1e9,
                 "frac": pddp_bytes(BH, w.N, w.D, G) / (stage_ms["pddp"] * 1e-3) / 1e9
                 / float(peaks.get("hbm_gbs", 6800.0)),
                 "peak": "hbm_gbs (" + peak_kind + ")"},
    }
    # mcs_select passes the heads through the workspace in chunks; each chunk
    # is one group-mass and one top-K launch
    rup = lambda x: -(-x // 256) * 256  # noqa: E731
    chunk = max(1, min(BH, ws_bytes // (rup(G * w.N * 4) + rup(G * 1088 * 4))))
    n_chunks = -(-BH // chunk)
    launches = pddp_launches(w.N, w.C) + 1 + 2 * n_chunks + 1 + R
    cores = len(os.sched_getaffinity(0))
    cpu = None
    if not args.no_cpu_baseline:
        v, dt, desc = oracle_time(oracle_setup(w, K), min_seconds=10.0)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}
    clocks = clk.summary()
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True,
        "scaling": args.split,
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": workload_label(w, args.density, K),
            "step": f"anchor (pddp, dense+lse, mass+top-k, sparse record) + {R} reuse steps "
                    "(sparse+residual, each with its own step's inputs; anchor interval "
                    f"{R + 1})",
            "value_basis": "reuse-step sparse attention kernel time, CUDA events, mean over the "
                           "reuse launches of the timed steps",
            "l2": "inputs larger than L2 (0.77 GB per tensor); no flush",
            "parallelism": (f"heads{world}: each rank owns a contiguous range of the "
                            f"flattened heads ({args.split} scaling: "
                            + ("global batch = ranks x the workload's batch"
                               if args.split == "weak" else "the workload's heads split")
                            + "); no collective on the data path"),
            "layout": "[B,N,H,D]" if layout == mcs.LAYOUT_BNHD else "[B,H,N,D]",
        },
        "speedup_vs_dense": speedup,
        "efficiency_vs_ideal": speedup * args.density,
        "dense_equivalent_tflops": job_flops_sparse / K * w.N / (t_sparse * 1e-3) / 1e12,
        "stage_ms": stage_ms,
        "reuse_launch_ms": reuse_launch_ms,  # by position after the anchor
        "kernels": kernels,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "token-sparse attention (reuse step)",
                     "peak_source": f"bf16_tflops_sustained ({peak_kind})"},
        "cpu_baseline": cpu,
        "e2e": ({"value": job_flops_sparse / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                 "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                 "ms_per_step": e2e_ms,
                 "pipelining": "step i+1's host->device copies of Q, K, V and step i-1's "
                               "device->host read-back overlap step i's kernel; the "
                               "layer's metadata from the anchor (perm, idx, residual) "
                               "stays resident in HBM"}
                if e2e else None),
        # the same loop with the metadata entry also staged from pinned host
        # memory every step (mcs_stager's offload scheme, for models whose
        # layers' metadata does not fit in HBM)
        "e2e_staged_metadata": (
            {"value": job_flops_sparse / (e2e_staged_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
             "h2d_bytes_per_step": e2e_staged["h2d"], "d2h_bytes_per_step": e2e_staged["d2h"],
             "ms_per_step": e2e_staged_ms,
             "pipelining": "as e2e; the metadata entry (perm, idx bitmaps, residual) is staged "
                           "by mcs_stager into two device slots and its indices unpacked on "
                           "the device each step"}
            if e2e_staged else None),
        # Q, K, V resident; only the layer's metadata entry comes from pinned host
        # memory each step, prefetched ahead through mcs_stager (the cache offload
        # scheme): hidden when ms_per_step matches the resident reuse kernel time
        "metadata_staging": ({"ms_per_step": staged_ms, "resident_ms_per_step": t_sparse,
                              "bytes_per_step": staging["bytes"],
                              "copy_gbs_needed": staging["bytes"] / (t_sparse * 1e-3) / 1e9}
                             if staging else None),
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
    }
    if extra is not None:
        line["workloads"] = extra
    print(json.dumps(line), flush=True)


def e4m3_pass(mcs, p, reuse_in, perm, idx, res, out, stream, rounds=3):
    """The reuse launches with K and V held as E4M3 bytes (one amax scale per
    tensor), timed beside the bf16 launches on the same inputs and metadata,
    alternating, after one warm-up round.  Returns the mean launch times, the
    ratio, the quantisation time of one step's K and V, and the K/V bytes the
    gathers read per launch."""
    cached = []
    for q_, k_, v_ in reuse_in:
        ks = float(k_.float().abs().max().item()) / 448.0
        vs = float(v_.float().abs().max().item()) / 448.0
        k8 = torch.empty(k_.shape, dtype=torch.uint8, device=k_.device)
        v8 = torch.empty_like(k8)
        qa, qb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        qa.record(stream)
        mcs.mcs_quantize_e4m3(k_, ks, k8)
        mcs.mcs_quantize_e4m3(v_, vs, v8)
        qb.record(stream)
        cached.append((q_, k_, v_, k8, v8, ks, vs, qa, qb))
    pairs = []  # (e4m3 launch, bf16 launch) events per input set and round
    for rnd in range(rounds + 1):
        for q_, k_, v_, k8, v8, ks, vs, _, _ in cached:
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record(stream)
            mcs.mcs_sparse_attn_e4m3(p, q_, k8, v8, ks, vs, perm, idx, res, out)
            ev[1].record(stream)
            mcs.mcs_sparse_attn(p, q_, k_, v_, perm, idx, res, out)
            ev[2].record(stream)
            if rnd > 0:
                pairs.append(ev)
    torch.cuda.synchronize()
    st = mcs.mcs_device_status()
    if st != 0:
        raise RuntimeError(f"device status after the e4m3 pass: {mcs.mcs_status_string(st)}")
    ms8 = statistics.mean(e[0].elapsed_time(e[1]) for e in pairs)
    ms16 = statistics.mean(e[1].elapsed_time(e[2]) for e in pairs)
    quant_ms = statistics.mean(c[7].elapsed_time(c[8]) for c in cached)
    BH, G = p.B * p.H, p.G
    return {"ms": ms8, "bf16_ms_same_run": ms16, "vs_bf16": ms16 / ms8,
            "quantize_kv_ms": quant_ms,
            "kv_gather_gb_per_launch": 2.0 * BH * G * p.K * p.D * 1 / 1e9,
            "bf16_kv_gather_gb_per_launch": 2.0 * BH * G * p.K * p.D * 2 / 1e9,
            "launches": len(pairs), "scales": "one amax scale per tensor (K, V)"}


# The workloads' denoising schedules (single GPU), each density measured on its
# own: (workload, density, timed passes over the schedule).
SCHEDULES = [("small", 0.1, 3), ("small", 0.2, 3), ("small", 0.3, 3),
             ("long", 0.15, 2), ("long", 0.25, 2), ("asset3d", 0.15, 3)]


def schedule_pass(p, steps, anchors, inputs, bufs, stream, pairs=None):
    """One pass over a denoising schedule: an anchor step (grouping, dense
    attention + LSE, exact selection, sparse attention recording the
    residual) at each anchor, a reuse step (sparse attention + cached
    residual) otherwise, each on its own step's inputs.  With `pairs` (C = 64)
    the anchor also builds the sibling-pair key lists and the sparse passes
    run on them.  Returns the events bracketing every stage, in order."""
    from token_sparse_attention_gb300 import mcs

    perm, idx, dense, lse, res, out, retained, ws = bufs
    marks = []

    def mark(name):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        marks.append((name, e))

    mark("start")
    for t in range(steps):
        q, k, v = inputs[t]
        if t in anchors:
            mcs.mcs_group(p, q, perm, ws)
            mark("pddp")
            mcs.mcs_dense_attn(p, q, k, v, dense, lse)
            mark("dense")
            mcs.mcs_select(p, q, k, lse, perm, idx, ws, retained)
            if pairs is not None:
                mcs.mcs_pair_lists(p, idx, pairs)
            mark("select")
            if pairs is not None:
                mcs.mcs_sparse_attn_pairs_record(p, q, k, v, perm, pairs, dense, res)
            else:
                mcs.mcs_sparse_attn_record(p, q, k, v, perm, idx, dense, res)
            mark("record")
        elif pairs is not None:
            mcs.mcs_sparse_attn_pairs(p, q, k, v, perm, pairs, res, out)
            mark("reuse")
        else:
            mcs.mcs_sparse_attn(p, q, k, v, perm, idx, res, out)
            mark("reuse")
    return marks


def run_schedules(dev):
    """Per-workload measurements: each workload's schedule (anchors and reuse
    steps on drifting inputs) timed stage by stage with CUDA events.  Reports
    the reuse-step sparse kernel (effective TFLOP/s, speedup over this
    library's dense kernel on the same workload, efficiency against the ideal
    1/density, fraction of the measured sustained bf16 peak), the anchor's
    cost, and the schedule's time per step with the density it amounts to:
    equivalent density = time per step / dense attention time; the anchors'
    share of it, anchor_delta_s = anchors x (anchor step - reuse step) /
    (steps x dense), is what the pages express as points of density."""
    from token_sparse_attention_gb300 import mcs

    peaks, _ = _peaks()
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    stream = torch.cuda.current_stream()
    res_all = {}
    for name, density, reps in SCHEDULES:
        w = synth.workload(name)
        K = w.K(density)
        p = mcs.params(w.B, w.H, w.N, w.D, w.C, K)
        G = p.G
        inputs = [synth.make_qkv(w, t, device=dev) for t in range(w.steps)]
        q0 = inputs[0][0]
        bufs = (torch.empty(w.B, w.H, G * w.C, dtype=torch.int32, device=dev),
                torch.empty(w.B, w.H, G, K, dtype=torch.int32, device=dev),
                torch.empty_like(q0), torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev),
                torch.empty_like(q0), torch.empty_like(q0),
                torch.empty(w.B, w.H, G, dtype=torch.float32, device=dev),
                mcs.empty_workspace(mcs.mcs_anchor_workspace(p), dev))
        # C = 64: sibling pairs share one 128-row tile over their key union,
        # when the paired grid (two pairs per CTA) still fills the GPU twice
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        paired_ctas = w.B * w.H * (-(-G // 2)) / 2
        pairs = (mcs.empty_pairs(p, dev)
                 if mcs.mcs_pair_bytes(p) and paired_ctas >= 2 * sms else None)
        schedule_pass(p, w.steps, w.anchors, inputs, bufs, stream, pairs)  # warm-up
        torch.cuda.synchronize()
        unpaired_ms = None
        if pairs is not None:
            # the same reuse launch without pairing, for comparison
            q1, k1, v1 = inputs[1]
            perm_, idx_, _, _, res_, out_ = bufs[:6]
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            mcs.mcs_sparse_attn(p, q1, k1, v1, perm_, idx_, res_, out_)
            a_.record(stream)
            for _ in range(3):
                mcs.mcs_sparse_attn(p, q1, k1, v1, perm_, idx_, res_, out_)
            b_.record(stream)
            torch.cuda.synchronize()
            unpaired_ms = a_.elapsed_time(b_) / 3
        per = {}
        for _ in range(reps):
            marks = schedule_pass(p, w.steps, w.anchors, inputs, bufs, stream, pairs)
            torch.cuda.synchronize()
            for (_, a), (n, b) in zip(marks, marks[1:]):
                per.setdefault(n, []).append(a.elapsed_time(b))
        if mcs.mcs_device_status() != 0:
            raise RuntimeError(f"device status after the {name} schedule")
        n_anchor, n_reuse = len(w.anchors), w.steps - len(w.anchors)
        stage = {n: statistics.mean(v) for n, v in per.items()}
        anchor_ms = sum(stage[n] for n in ("pddp", "dense", "select", "record"))
        reuse_ms = stage["reuse"]
        total = sum(sum(v) for v in per.values()) / reps
        BH = w.B * w.H
        fl_sparse = 4.0 * BH * w.N * K * w.D
        tfl = fl_sparse / (reuse_ms * 1e-3) / 1e12
        speedup = stage["dense"] / reuse_ms
        res_all[f"{name} s={density}"] = {
            "workload": workload_label(w, density, K),
            "schedule": f"{w.steps} steps, anchors at {list(w.anchors)}, drift {w.drift} per step",
            "sparse_reuse_ms": reuse_ms,
            "sparse_tflops": tfl,
            "dense_ms": stage["dense"],
            "dense_tflops": 4.0 * BH * w.N * w.N * w.D / (stage["dense"] * 1e-3) / 1e12,
            "speedup_vs_dense": speedup,
            "efficiency_vs_ideal": speedup * density,
            "roofline_frac": tfl / peak,
            "anchor_ms": anchor_ms,
            "anchor_stage_ms": {n: stage[n] for n in ("pddp", "dense", "select", "record")},
            "ms_per_step": total / w.steps,
            "equivalent_density": total / w.steps / stage["dense"],
            "anchor_delta_s": n_anchor * (anchor_ms - reuse_ms) / (w.steps * stage["dense"]),
            "passes": reps,
            "n_anchor": n_anchor, "n_reuse": n_reuse,
        }
        if pairs is not None:
            r = res_all[f"{name} s={density}"]
            r["sibling_pairs"] = True
            r["sparse_reuse_ms_unpaired"] = unpaired_ms
            r["speedup_vs_dense_unpaired"] = stage["dense"] / unpaired_ms
        del inputs, bufs, q0, pairs
        torch.cuda.empty_cache()
    return res_all


def run_diagnostics(args, w):
    """Selector diagnostics: attention recall and output relative L1 of
    mean-pooled block selection, the block oracle, the token oracle (exact
    group mass) and the per-query oracle, at matched numbers of kept tokens,
    under raster (consecutive tiles) and PDDP query groups.  One JSON line."""
    from token_sparse_attention_gb300 import mcs

    mcs.lib()
    dev = torch.device("cuda", torch.cuda.current_device())
    block = 128
    H = w.H
    q, k, v = synth.make_qkv(w, 0, device=dev)
    G = -(-w.N // w.C)
    p0 = mcs.params(w.B, H, w.N, w.D, w.C, w.N)
    dense = torch.empty_like(q)
    lse = torch.empty(w.B, H, w.N, dtype=torch.float32, device=dev)
    mcs.mcs_dense_attn(p0, q, k, v, dense, lse)
    raster = torch.arange(G * w.C, dtype=torch.int32, device=dev)
    raster[w.N:] = -1
    groupings = {"raster": raster.expand(w.B, H, -1).contiguous()}
    pddp = torch.empty(w.B, H, G * w.C, dtype=torch.int32, device=dev)
    mcs.mcs_group(p0, q, pddp, mcs.empty_workspace(mcs.mcs_group_workspace(p0), dev))
    groupings["pddp"] = pddp
    # per-query oracle: G sampled queries per head, each alone in a group
    gen = torch.Generator().manual_seed(99)
    sample = torch.stack([torch.randperm(w.N, generator=gen)[:G].sort().values for _ in range(H)])
    one = torch.full((w.B, H, G * w.C), -1, dtype=torch.int32)
    one[..., ::w.C] = sample.to(torch.int32)
    one = one.to(dev)
    sample_rows = (torch.arange(H)[:, None] * w.N + sample).reshape(-1).to(torch.int32).to(dev)
    BH = w.B * H
    rows = []
    timings = {}

    def timed(name, fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        timings.setdefault(name, []).append(a.elapsed_time(b))

    masses = {}
    for name, perm in list(groupings.items()) + [("one-query", one)]:
        m = torch.empty(BH, G, w.N, dtype=torch.float32, device=dev)
        timed("group_mass", lambda: mcs.mcs_group_mass(p0, q, k, lse, perm, 0, BH, m))
        masses[name] = m
    sizes = torch.tensor([min(w.C, w.N - g * w.C) for g in range(G)], dtype=torch.float64)
    for s_ in (0.1, 0.2, 0.3):
        K = max(block, round(s_ * w.N / block) * block)
        p = mcs.params(w.B, H, w.N, w.D, w.C, K)
        ws = mcs.empty_workspace(mcs.mcs_block_workspace(p, block), dev)
        out = torch.empty_like(q)

        def record(grouping, selector, idx, kept, rows_sel=None, denom=None):
            perm = one if grouping == "one-query" else groupings[grouping]
            mcs.mcs_sparse_attn(p, q, k, v, perm, idx, None, out)
            e, d = mcs.mcs_rel_l1(p, out, dense, rows_sel)
            # attention recall: kept probability mass per query, averaged over queries
            recall = float(kept.double().sum().cpu() / (denom.sum() * BH))
            rows.append({"density": K / w.N, "K": K, "grouping": grouping, "selector": selector,
                         "recall": recall, "rel_l1": e / d})

        for gname, perm in groupings.items():
            mass = masses[gname]
            idx = torch.empty(w.B, H, G, K, dtype=torch.int32, device=dev)
            kept = torch.empty(BH * G, dtype=torch.float32, device=dev)
            timed("pooled_block_select", lambda: mcs.mcs_pooled_block_select(p, q, k, perm, block,
                                                                            idx, ws))
            timed("gather_mass", lambda: mcs.mcs_gather_mass(p, mass, idx, kept))
            record(gname, f"mean-pooled blocks of {block}", idx, kept, denom=sizes)
            timed("block_topk", lambda: mcs.mcs_block_topk(p, mass, block, idx, ws, retained=kept))
            record(gname, f"block oracle ({block})", idx, kept, denom=sizes)
            timed("topk", lambda: mcs.mcs_topk(p, mass, idx, kept))
            record(gname, "token oracle", idx, kept, denom=sizes)
        idx = torch.empty(w.B, H, G, K, dtype=torch.int32, device=dev)
        kept = torch.empty(BH * G, dtype=torch.float32, device=dev)
        mcs.mcs_topk(p, masses["one-query"], idx, kept)
        record("one-query", "per-query oracle (sampled queries)", idx, kept, sample_rows,
               denom=torch.ones(G, dtype=torch.float64))
    if mcs.mcs_device_status() != 0:
        raise RuntimeError("device status after the diagnostics")
    print(json.dumps({
        "diagnostics": "selector recall and output relative L1 (sparse output without the "
                       "residual against dense attention), matched numbers of kept tokens",
        "workload": f"{w.name} B={w.B} H={H} N={w.N} D={w.D} C={w.C}", "data": "synthetic",
        "block": block, "per_query_sample": f"{G} random queries per head (seed 99)",
        "rows": rows,
        "kernel_ms": {n: statistics.median(t) for n, t in timings.items()},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="mcs", choices=["mcs", "reference"])
    ap.add_argument("--workload", default="large")
    ap.add_argument("--density", type=float, default=0.2)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reuse-per-anchor", type=int, default=4,
                    help="reuse steps timed after each anchor (anchor interval - 1)")
    ap.add_argument("--layout", default="bhnd", choices=["bhnd", "bnhd"],
                    help="activation layout: [B,H,N,D] or [B,N,H,D]")
    ap.add_argument("--diagnostics", action="store_true",
                    help="print the selector diagnostics line instead of the bench line")
    ap.add_argument("--split", default="weak", choices=["weak", "strong"],
                    help="several GPUs: weak = each rank a full copy of the workload's heads "
                         "(global batch grows), strong = the workload's heads split over ranks")
    ap.add_argument("--no-e4m3", action="store_true",
                    help="skip the reuse launches over an E4M3 K/V cache")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload schedule measurements (single GPU only)")
    ap.add_argument("--heads", type=int, default=0,
                    help="override the head count (smaller cases for profiling; not a bench number)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = synth.workload(args.workload)
    if args.heads:
        w = dataclasses.replace(w, H=args.heads)
    K = w.K(args.density)

    if args.impl == "reference":
        run_reference(args, w, K, rank)
        return

    torch.cuda.set_device(local)
    if args.diagnostics:
        run_diagnostics(args, w)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist_mod.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = dist_mod
    try:
        run_gpu(args, w, K, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

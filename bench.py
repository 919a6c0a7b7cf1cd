#!/usr/bin/env python
"""Benchmark of the VSA hot path on the Wan2.2 attention shape.

One step = one pass of the whole hot path over one batch of synthetic input
(21 x 30 x 52 latent grid, 40 heads, D = 128): tile k and v and mean-pool the
cubes of q and k -> coarse select (topk = 78 of 624 cubes) -> query-cube
pairing -> block-sparse attention reading q and writing the output in raster
order (the tiling of q and the untiling of the output are part of that pass).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is effective TFLOPS over the whole
step, using the fine-stage effective FLOP count 4 * S_pad * k * 64 * D * H * B
(the work the selected blocks need, not the dense work avoided); the fine
kernel's own time and roofline fraction are reported beside it.  Inputs
(q, k, v: 3 x 335 MB, plus 0.8 GB of tiled intermediates) exceed the 126 MB
L2, so no explicit flush is used between steps.

--impl reference times the CPU oracle (the only other implementation there is)
on a bounded sample of the same workload.  Under torchrun every rank runs its
own replica (the op shards by heads with no collective; this build runs one
replica per GPU) and rank 0 reports the aggregate.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)

METRIC = "VSA sparse-attn fwd ms/call and effective TFLOPS; % of GB300 bf16 TC peak"
UNIT = "TFLOPS (effective)"
WORKLOAD = "wan"

# DRAM traffic of one fine_fwd_kernel launch, from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum) of the Wan grid with 8 heads, scaled by 40/8 (traffic grows with
# the (batch, head, query-cube pair) units processed).  Valid only for the kernel source it
# was taken from: if fine.cu no longer hashes to `source_sha256`, the traffic is reported
# as null.
FINE_TRAFFIC = {
    "bytes_per_launch": (233.117696e6 + 55.445504e6) * 40 / 8,
    "capture": "ncu, fine_fwd_kernel on the Wan2.2 grid with 8 heads (one launch), scaled x5",
    "source_sha256": "6e7173ac74a9415274dd98393d31250459216f88c902b2f30282065ec3321514",
}
# The same for the 128-token-block workload, from a capture of one whole
# 12-head launch (no scaling).
FINE_TRAFFIC_BLOCKS = {
    "bytes_per_launch": 309.088768e6 + 86.803200e6,
    "capture": "ncu, fine_fwd_kernel on the 128-token-block workload (one whole launch)",
    "source_sha256": "6e7173ac74a9415274dd98393d31250459216f88c902b2f30282065ec3321514",
}


def load_peaks():
    path = os.path.join(HERE, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), float(p["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []        # (host monotonic time, csv line)
        self.window = None     # (t0, t1) of the timed region, host monotonic time

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        """Clocks seen inside the timed window; if the sampler produced no
        sample there (a very short timed region), the samples taken while the
        warm-up and timed steps ran, marked as such."""
        lines = self.lines
        where = "timed region"
        if self.window is not None:
            t0, t1 = self.window
            inside = [(t, ln) for t, ln in lines if t0 <= t <= t1 + 0.05]
            if inside:
                lines = inside
            else:
                where = "warm-up and timed steps (timed region shorter than the sampling period)"
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "sampled_over": where}


# ------------------------------------------------------------ CPU oracle
def host_cores():
    """Logical CPUs listed in /proc/cpuinfo (None where it is unreadable)."""
    try:
        with open("/proc/cpuinfo") as f:
            return sum(1 for line in f if line.startswith("processor"))
    except OSError:
        return None


def cpu_oracle_sample(wl, inputs, budget_s: float = 15.0, seed: int = 0):
    """The oracle pipeline on the host cores: tile (q, k, v) and the coarse
    selection in full, the fine stage (>99.9% of the work) on random query
    cubes for about `budget_s` seconds with every thread, then on a fixed
    subset with one thread.  Returns the cpu_baseline object."""
    import oracle
    t0 = time.perf_counter()
    qt, vbs = oracle.tile(inputs["q"], wl.grid)
    kt, _ = oracle.tile(inputs["k"], wl.grid)
    vt, _ = oracle.tile(inputs["v"], wl.grid)
    t_tile = time.perf_counter() - t0
    t0 = time.perf_counter()
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    t_coarse = time.perf_counter() - t0
    rng = np.random.default_rng(seed)
    nthreads = oracle.default_threads()
    units_total = wl.B * wl.heads * wl.ncubes
    flops_per_unit = wl.fine_flops() / units_total
    done_units, elapsed, used = 0, 0.0, 0
    batch = max(nthreads, 8)
    while elapsed < budget_s and done_units < units_total:
        units = rng.choice(units_total, size=batch, replace=False).astype(np.int64)
        t0 = time.perf_counter()
        _, _, used = oracle.fine(qt, kt, vt, idx, vbs, wl.sm_scale, units)
        elapsed += time.perf_counter() - t0
        done_units += batch
    per_unit = elapsed / done_units
    tflops = done_units * flops_per_unit / elapsed / 1e12
    one = np.arange(8, dtype=np.int64)  # fixed subset: the first 8 query cubes of head 0
    t0 = time.perf_counter()
    oracle.fine(qt, kt, vt, idx, vbs, wl.sm_scale, one, nthreads=1)
    t_one = time.perf_counter() - t0
    fine_full_s = per_unit * units_total
    desc = (f"tile of q, k, v and the coarse selection in full; the fine stage on {done_units} random "
            f"query cubes of {units_total} ({elapsed:.1f} s, {used} threads), its whole-call time "
            f"extrapolated from that sample")
    return {"value": tflops, "unit": UNIT, "cores": used, "kind": "oracle", "sample": desc,
            "host_cpus": host_cores(),
            "stage_seconds": {"tile_qkv": t_tile, "coarse_select": t_coarse,
                              "fine_extrapolated": fine_full_s,
                              "whole_call_extrapolated": t_tile + t_coarse + fine_full_s},
            "one_thread": {"units": int(one.size), "seconds": t_one,
                           "tflops": one.size * flops_per_unit / t_one / 1e12,
                           "subset": "the first 8 query cubes of head 0"}}


def reference_arm(args, wl, inputs):
    """--impl reference: the CPU oracle as it stands, one bounded sample per step."""
    import oracle
    qt, vbs = oracle.tile(inputs["q"], wl.grid)
    kt, _ = oracle.tile(inputs["k"], wl.grid)
    vt, _ = oracle.tile(inputs["v"], wl.grid)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    nthreads = oracle.default_threads()
    units_total = wl.B * wl.heads * wl.ncubes
    per_step = 2 * nthreads
    rng = np.random.default_rng(1)
    flops_per_unit = wl.fine_flops() / units_total
    used = 0
    for _ in range(args.warmup):
        _, _, used = oracle.fine(qt, kt, vt, idx, vbs, wl.sm_scale,
                                 rng.choice(units_total, size=per_step, replace=False))
    times = []
    for _ in range(args.steps):
        units = rng.choice(units_total, size=per_step, replace=False)
        t0 = time.perf_counter()
        _, _, used = oracle.fine(qt, kt, vt, idx, vbs, wl.sm_scale, units)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = args.steps * per_step * flops_per_unit / total / 1e12
    desc = f"fine stage on {per_step} random query cubes of {units_total} per step"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(wl),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def fine_traffic(record=None):
    """DRAM bytes per launch of the fine kernel from its ncu capture, or None
    once fine.cu no longer hashes to the source the capture was taken from."""
    import hashlib
    record = FINE_TRAFFIC if record is None else record
    path = os.path.join(HERE, "block_sparse_video_vsa_gb300", "csrc", "fine.cu")
    with open(path, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()
    return record["bytes_per_launch"] if digest == record["source_sha256"] else None


def stage_bytes(wl):
    """Algorithmic HBM bytes per call of the memory-bound stages."""
    real = wl.B * wl.tokens * wl.heads * wl.D * 2
    tiled = wl.B * wl.s_pad * wl.heads * wl.D * 2
    cubes = wl.B * wl.heads * wl.ncubes
    pooled = 16 * cubes * wl.D + 8 * cubes              # means + residuals of q, k (fp32), norms
    return {
        "tile_k_pool_qk": 2 * real + tiled + pooled,        # read raster q, k; write tiled k + statistics
        "tile_v": real + tiled,                              # side stream, beside the coarse selection
        "coarse_select": 8 * cubes * wl.D + 8 * cubes + 4 * cubes * wl.topk,  # read means, norms; write idx
    }


LABELS = {"wan": "Wan2.2-shape VSA", "wan_outlier": "Wan2.2-shape VSA with an outlier head (logits ~1e3)",
          "hunyuan": "HunyuanVideo-shape VSA",
          "blocks128": "Wan2.1-shape sequence in 128-token blocks (mean-pool CDF selector + fine stage)"}

# Cumulative-share threshold of the block selector for the blocks128 workload:
# with tau = 0.4608 the oracle's selector keeps 30.0% of the key blocks of the
# synthetic 32,768-token, 12-head call (found by bisection on the oracle), the
# 70% sparsity point of the pages' kernel-time sweep.
BLOCKS_TAU = 0.4608


def config_of(wl):
    label = LABELS.get(wl.name.split("-")[0], wl.name)
    return {"workload": f"{label}: grid {wl.T}x{wl.H}x{wl.W}, {wl.heads} heads, D={wl.D}, "
                        f"topk={wl.topk} of {wl.ncubes} cubes",
            "B": wl.B, "grid": [wl.T, wl.H, wl.W], "heads": wl.heads, "head_dim": wl.D,
            "topk": wl.topk, "ncubes": wl.ncubes, "s_padded": wl.s_pad,
            "fine_flops": wl.fine_flops(),
            "l2": f"inputs and intermediates ({step_bytes(wl) / 1e9:.2f} GB touched per step) exceed the "
                  f"126 MB L2; no flush"}


def step_bytes(wl):
    """Bytes of the step's big tensors: q, k, v and out raster; k and v tiled."""
    untiled = wl.B * wl.T * wl.H * wl.W * wl.heads * wl.D * 2
    tiled = wl.B * wl.s_pad * wl.heads * wl.D * 2
    return 4 * untiled + 2 * tiled


def executed_tensor_flops(idx, pairs, D: int) -> float:
    """Tensor-core FLOPs the paired fine kernel issues for a selection.

    A unit (query cubes i and j, 128 query rows) walks the union U of the two
    selections two key cubes per step: each step runs Q.K^T over 128 rows x
    128 keys, and P.V over the step's keys (64 per cube), so a unit costs
    ceil(|U| / 2) * 2*128*128*D + |U| * 2*128*64*D FLOPs.  idx: [B, heads, N,
    k] int32 (every entry in [0, N)); pairs: [B, heads, ceil(N / 2)] as
    i | (j << 16), j = 0xFFFF for a single cube."""
    idx = np.asarray(idx)
    pr = np.asarray(pairs).astype(np.int64) & 0xFFFFFFFF
    B, H, N, k = idx.shape
    steps = cubes = 0
    for b in range(B):
        for h in range(H):
            sel = np.zeros((N + 1, N), dtype=bool)  # row N: no cube
            sel[np.repeat(np.arange(N), k), idx[b, h].reshape(-1)] = True
            i0 = np.minimum(pr[b, h] & 0xFFFF, N)
            i1 = np.minimum(pr[b, h] >> 16, N)
            u = (sel[i0] | sel[i1]).sum(axis=1)
            steps += int(((u + 1) // 2).sum())
            cubes += int(u.sum())
    return float(steps) * 2 * 128 * 128 * D + float(cubes) * 2 * 128 * 64 * D


# --------------------------------------------------------- blocks128
def blocks_flops(counts, D: int) -> float:
    """Effective fine-stage FLOPs of a cube table: 4 * 64 * 64 * D per (query
    cube, listed key cube), i.e. 4 * S * k * 64 * D * heads for uniform k."""
    return 4.0 * 64 * 64 * D * float(np.asarray(counts, np.int64).sum())


def run_blocks(args, rank, world, dist):
    """One step = the block selector (pool + select) and the fine stage on its
    table, for q, k, v [1, 32768, 12, 128] in 128-token blocks."""
    import torch

    import block_sparse_video_vsa_gb300 as vsa
    from block_sparse_video_vsa_gb300 import synth

    wl, s_len = synth.SEQUENCE_WORKLOADS["blocks128"]
    inputs = synth.make_sequence_inputs("blocks128")
    dev = torch.device("cuda", torch.cuda.current_device())

    def dev_bf16(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)

    q, k, v = (dev_bf16(inputs[n]) for n in ("q", "k", "v"))
    vbs = torch.from_numpy(inputs["vbs"]).to(dev)
    B, S, H, D = q.shape
    nc = S // 64
    ws = torch.empty((vsa.block_select_workspace_bytes(B, S, H, D),), dtype=torch.uint8, device=dev)
    tbl = torch.empty((B, H, nc, nc), dtype=torch.int32, device=dev)
    cnt = torch.empty((B, H, nc), dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def step(marks=None, qin=None, kin=None, vin=None, oout=None):
        qin = q if qin is None else qin
        kin = k if kin is None else kin
        vin = v if vin is None else vin
        oout = out if oout is None else oout
        if marks is not None:
            marks[0].record(stream)
        vsa.block_select(qin, kin, BLOCKS_TAU, wl.sm_scale, workspace=ws, out=tbl, counts=cnt)
        if marks is not None:
            marks[1].record(stream)
        vsa.sparse_attn_fwd(qin, kin, vin, tbl, vbs, wl.sm_scale, out=oout, lse=lse, counts=cnt)
        if marks is not None:
            marks[2].record(stream)

    clk = ClockSampler(torch.cuda.current_device())
    with clk:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        if vsa.device_error(reset=True):
            raise RuntimeError("device error word set during warm-up")
        counts_host = cnt.cpu().numpy()
        marks = [[ev() for _ in range(3)] for _ in range(args.steps)]
        start, end = ev(), ev()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.monotonic()
        n0 = vsa.kernel_launches()
        start.record(stream)
        for s in range(args.steps):
            step(marks[s])
        end.record(stream)
        launches = vsa.kernel_launches() - n0
        torch.cuda.synchronize()
        clk.window = (t0, time.monotonic())
    if dist:
        dist.barrier()
    if vsa.device_error(reset=True):
        raise RuntimeError("device error word set during the timed run")
    ms_step = max_over_ranks(start.elapsed_time(end), dist, dev) / args.steps
    stage = {"block_select": [m[0].elapsed_time(m[1]) for m in marks],
             "sparse_attn_fwd": [m[1].elapsed_time(m[2]) for m in marks]}
    e2e = None
    if not args.no_e2e:
        e2e = e2e_leg(step, inputs, q, k, v, out, args, stream, dist, dev)
    flops = blocks_flops(counts_host, D)
    burst, sustained, hbm, peak_kind = load_peaks()
    fine_ms = statistics.mean(stage["sparse_attn_fwd"])
    fine_tflops = flops / (fine_ms * 1e-3) / 1e12
    sparsity = 1.0 - counts_host.mean() / nc
    sel_bytes = 2 * B * S * H * D * 2  # q and k read once by the pooling pass
    result = {
        "metric": METRIC, "value": whole_job_throughput(world, flops, ms_step), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{LABELS['blocks128']}: q, k, v [{B}, {S}, {H}, {D}], tau={BLOCKS_TAU} "
                               f"(sparsity {sparsity:.3f})",
                   "B": B, "seq_len": S, "heads": H, "head_dim": D, "block_tokens": 128, "tau": BLOCKS_TAU,
                   "sparsity": sparsity, "fine_flops": flops,
                   "l2": f"q, k, v, out ({4 * B * S * H * D * 2 / 1e9:.2f} GB) exceed the 126 MB L2; no flush"},
        "fine_kernel": {"ms_per_call_mean": fine_ms, "ms_per_call_median": statistics.median(stage["sparse_attn_fwd"]),
                        "effective_tflops": fine_tflops, "frac_of_burst_peak": fine_tflops / burst,
                        "frac_of_sustained_peak": fine_tflops / sustained},
        "stages_ms_median": {k2: statistics.median(v2) for k2, v2 in stage.items()},
        "stages_hbm_gbs": {"block_select": sel_bytes / (statistics.median(stage["block_select"]) * 1e-3) / 1e9},
        "hbm_peak_gbs": hbm,
        "roofline": {"bound": "tensor", "achieved": fine_tflops, "peak": burst, "unit": "TFLOP/s",
                     "frac": fine_tflops / burst, "traffic": fine_traffic(FINE_TRAFFIC_BLOCKS),
                     "peak_kind": f"{peak_kind} dense bf16 burst",
                     "kernel": "fine_fwd_kernel (vsa_sparse_attn_fwd with the selector's counts)"},
        "e2e": None if e2e is None else {
            "value": whole_job_throughput(world, flops, e2e[0]), "unit": UNIT, "ms_per_step": e2e[0],
            "h2d_bytes_per_step": e2e[1], "d2h_bytes_per_step": e2e[2], **e2e[3]},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_blocks_sample(inputs, tbl.cpu().numpy(), counts_host, wl, args.cpu_budget)
    return result


def cpu_blocks_sample(inputs, table, counts, wl, budget_s):
    """The oracle's fine stage on random query cubes of the blocks128 table."""
    import oracle
    rng = np.random.default_rng(0)
    nthreads = oracle.default_threads()
    total = counts.size
    flat = counts.reshape(-1)
    done, flops, elapsed, used = 0, 0.0, 0.0, 0
    while elapsed < budget_s and done < total:
        units = rng.choice(total, size=max(nthreads, 8), replace=False).astype(np.int64)
        t0 = time.perf_counter()
        _, _, used = oracle.fine_counts(inputs["q"], inputs["k"], inputs["v"], table, counts, inputs["vbs"],
                                        wl.sm_scale, units)
        elapsed += time.perf_counter() - t0
        done += units.size
        flops += blocks_flops(flat[units], wl.D)
    return {"value": flops / elapsed / 1e12, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"fine stage on {done} random query cubes of {total} ({elapsed:.1f} s, {used} threads)"}


# ------------------------------------------------------------------ ours
def run_ours(args, wl, inputs, rank, world, dist):
    import torch

    import block_sparse_video_vsa_gb300 as vsa

    dev = torch.device("cuda", torch.cuda.current_device())

    def dev_bf16(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)

    q, k, v = (dev_bf16(inputs[n]) for n in ("q", "k", "v"))
    grid = wl.grid
    N = wl.ncubes
    kt = torch.empty((wl.B, wl.s_pad, wl.heads, wl.D), dtype=torch.bfloat16, device=dev)
    vt = torch.empty_like(kt)
    vbs = torch.empty((N,), dtype=torch.int32, device=dev)
    vbs2 = torch.empty_like(vbs)
    idx = torch.empty((wl.B, wl.heads, N, wl.topk), dtype=torch.int32, device=dev)
    ws = torch.empty((vsa.coarse_workspace_bytes(wl.B, wl.heads, N, wl.D),), dtype=torch.uint8, device=dev)
    lse = torch.empty((wl.B, wl.heads, wl.s_pad), dtype=torch.float32, device=dev)
    pws = torch.empty((vsa.pair_workspace_bytes(wl.B, wl.heads, N, wl.topk),), dtype=torch.uint8, device=dev)
    pairs = torch.empty((wl.B, wl.heads, (N + 1) // 2), dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    # Tiling v needs neither the coarse selection nor the pairing, so it runs on
    # a side stream beside the coarse selection (a latency-bound GEMM and
    # per-row selection, which leave HBM bandwidth to spare); the pairing
    # kernels (one CTA per head) then run alone.
    side = torch.cuda.Stream()
    ev_qk, ev_v = torch.cuda.Event(), torch.cuda.Event()

    def step(marks=None, qin=None, kin=None, vin=None, oout=None):
        qin = q if qin is None else qin
        kin = k if kin is None else kin
        vin = v if vin is None else vin
        oout = out if oout is None else oout
        if marks is not None:
            marks[0].record(stream)
        # k is tiled and q, k pooled in one pass (q needs no tiled copy: the
        # fine stage reads it in raster order); the selection starts from the
        # pooled statistics the pass left in the workspace.
        vsa.tile_pool(qin, kin, grid, kt=kt, vbs=vbs, workspace=ws, want_qt=False)
        ev_qk.record(stream)
        side.wait_event(ev_qk)
        with torch.cuda.stream(side):
            if marks is not None:
                marks[6].record(side)
            vsa.tile(vin, grid, out=vt, vbs=vbs2)
            if marks is not None:
                marks[7].record(side)
            ev_v.record(side)
        if marks is not None:
            marks[1].record(stream)
        vsa.coarse_select_pooled(ws, vbs, wl.B, wl.heads, wl.D, wl.topk, wl.sm_scale, out=idx)
        if marks is not None:
            marks[2].record(stream)
        vsa.pair_cubes(idx, workspace=pws, out=pairs)
        if marks is not None:
            marks[3].record(stream)
        stream.wait_event(ev_v)
        # Raster q in, raster output out: no tiling of q, no untiling pass.
        vsa.sparse_attn_fwd_raster(qin, kt, vt, idx, vbs, grid, wl.sm_scale, out=oout, lse=lse, pairs=pairs)
        if marks is not None:
            marks[4].record(stream)

    clk = ClockSampler(torch.cuda.current_device())
    with clk:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        if vsa.device_error(reset=True):
            raise RuntimeError("device error word set during warm-up")

        marks = [[ev() for _ in range(8)] for _ in range(args.steps)]
        start, end = ev(), ev()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.monotonic()
        n0 = vsa.kernel_launches()
        start.record(stream)
        for s in range(args.steps):
            step(marks[s])
        end.record(stream)
        launches = vsa.kernel_launches() - n0  # every kernel the library enqueued in the timed region
        torch.cuda.synchronize()
        clk.window = (t0, time.monotonic())
    if dist:
        dist.barrier()
    ms_total = max_over_ranks(start.elapsed_time(end), dist, dev)
    ms_step = ms_total / args.steps
    stage = {name: [marks[s][i].elapsed_time(marks[s][i + 1]) for s in range(args.steps)]
             for i, name in enumerate(["tile_k_pool_qk", "coarse_select", "pair_cubes", "sparse_attn_fwd"])}
    stage["tile_v"] = [marks[s][6].elapsed_time(marks[s][7]) for s in range(args.steps)]  # side stream, beside coarse
    if vsa.device_error(reset=True):
        raise RuntimeError("device error word set during the timed run")

    e2e_ms, h2d, d2h, copy_ms = ((None, 0, 0, None) if args.no_e2e
                                 else e2e_leg(step, inputs, q, k, v, out, args, stream, dist, dev))
    # The next rows are timed last, after the end-to-end leg, on the step's
    # tensors (plus a tiled q and a tiled output buffer, which the step itself
    # does not need).
    qt, _ = vsa.tile(q, grid, vbs=vbs2)
    ot = torch.empty_like(qt)
    nxt = time_next_rows(vsa, torch, wl, qt, kt, vt, idx, vbs, pairs, ot, lse, stream)
    try:  # the tensor-core work the step's fine launch issued (host-side count, outside every timing)
        executed = executed_tensor_flops(idx.cpu().numpy(), pairs.cpu().numpy(), wl.D)
    except Exception:  # context only: never let it cost the result line
        executed = None
    return ms_step, stage, clk.summary(), (e2e_ms, h2d, d2h, copy_ms), launches, nxt, executed


def e2e_leg(step, inputs, q, k, v, out, args, stream, dist, dev):
    """End to end through host buffers (pinned), copies inside the timed region.

    Every step copies its q, k, v from pinned host memory and reads its output
    back; the copies run on their own streams, double-buffered, so the upload of
    step i + 1 and the read-back of step i - 1 overlap the compute of step i.
    `step(qin=, kin=, vin=, oout=)` enqueues one step on `stream`.  Returns
    (median ms per step over the runs, host-to-device bytes per step,
    device-to-host bytes per step, {copies-only ms per step, every run's ms
    per step, steps per run})."""
    import torch
    qh, kh, vh = (torch.from_numpy(inputs[n].view(np.int16)).view(torch.bfloat16).pin_memory()
                  for n in ("q", "k", "v"))
    ohs = [torch.empty(tuple(out.shape), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dq = [q, torch.empty_like(q)]
    dk = [k, torch.empty_like(k)]
    dv = [v, torch.empty_like(v)]
    douts = [out, torch.empty_like(out)]
    s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()
    # Up to 30 steps per run: the first upload (about 5 ms for 1 GB at the
    # ~210 GB/s host link) fills the pipeline once per run.  Five runs; the
    # median is reported with every run's figure (a run now and then holds
    # one stall of tens of ms while copies and kernels overlap).
    e2e_steps = max(3, min(args.steps, 30))
    e2e_repeats = 5

    def e2e_run(n, first=None, compute=True):
        up = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        down = [torch.cuda.Event() for _ in range(2)]
        if first is not None:
            s_up.wait_event(first)
        fin = []
        for i in range(n):
            bb = i & 1
            if i >= 4:
                # Keep the host at most four steps ahead: a full launch queue
                # blocks the enqueuing thread, and its wake-up has left the
                # GPU idle for tens of ms.
                fin[i - 4].synchronize()
            if i >= 2:
                s_up.wait_event(done[bb])  # step i - 2 has finished reading this input set
            with torch.cuda.stream(s_up):
                dq[bb].copy_(qh, non_blocking=True)
                dk[bb].copy_(kh, non_blocking=True)
                dv[bb].copy_(vh, non_blocking=True)
                up[bb].record(s_up)
            stream.wait_event(up[bb])
            if i >= 2:
                stream.wait_event(down[bb])  # the read-back of step i - 2 has left this output set
            if compute:
                step(qin=dq[bb], kin=dk[bb], vin=dv[bb], oout=douts[bb])
            done[bb].record(stream)
            fin.append(torch.cuda.Event())
            fin[-1].record(stream)
            s_down.wait_event(done[bb])
            with torch.cuda.stream(s_down):
                ohs[bb].copy_(douts[bb], non_blocking=True)
                down[bb].record(s_down)
        for bb in range(min(n, 2)):
            stream.wait_event(down[bb])

    e2e_run(2)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    runs = []
    for _ in range(e2e_repeats):
        torch.cuda.synchronize()
        e0.record(stream)
        e2e_run(e2e_steps, first=e0)
        e1.record(stream)
        torch.cuda.synchronize()
        runs.append(e0.elapsed_time(e1) / e2e_steps)
        last = (e2e_steps - 1) & 1
        if not torch.equal(ohs[last], douts[last].cpu()):
            raise RuntimeError("end-to-end read-back differs from the device result")
    e2e_ms = statistics.median(runs)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    # The same copies with no compute: the floor the host link sets.
    torch.cuda.synchronize()
    e0.record(stream)
    e2e_run(e2e_steps, first=e0, compute=False)
    e1.record(stream)
    torch.cuda.synchronize()
    copy_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)
    return e2e_ms, 3 * qh.numel() * 2, ohs[0].numel() * 2, {"copies_only_ms_per_step": copy_ms,
                                                            "runs_ms_per_step": runs, "steps_per_run": e2e_steps}


def max_over_ranks(x: float, dist, device) -> float:
    """The slowest rank's time (every rank gets it); x itself with one process."""
    if not dist:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(world: int, flops_per_rank: float, ms: float) -> float:
    """Effective TFLOP/s of all ranks together: every rank processed `flops_per_rank`
    in at most `ms` milliseconds (weak scaling: per-rank work is fixed)."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def time_next_rows(vsa, torch, wl, qt, kt, vt, idx, vbs, pairs, ot, lse, stream, calls=20):
    """CUDA-event medians of the coarse-stage attention output and of the fine
    stage with the gated combine, on the step's own tiled tensors (outside the
    timed step; gates are seeded uniform [0, 1) bf16)."""
    ws = torch.empty((vsa.coarse_attn_workspace_bytes(wl.B, wl.heads, wl.ncubes, wl.D),), dtype=torch.uint8,
                     device=qt.device)
    oc = torch.empty((wl.B, wl.heads, wl.ncubes, wl.D), dtype=torch.float32, device=qt.device)
    gen = torch.Generator(device=qt.device)
    gen.manual_seed(1234)
    gc = torch.rand(qt.shape, generator=gen, device=qt.device).to(torch.bfloat16)
    gf = torch.rand(qt.shape, generator=gen, device=qt.device).to(torch.bfloat16)

    def median_ms(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(calls):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    ca_ms = median_ms(lambda: vsa.coarse_attn(qt, kt, vt, vbs, wl.sm_scale, workspace=ws, out=oc))
    quality = selection_quality(vsa, torch, wl, qt, kt, vt, idx, vbs, pairs, stream)
    fg_ms = median_ms(lambda: vsa.sparse_attn_fwd(qt, kt, vt, idx, vbs, wl.sm_scale, out=ot, lse=lse, pairs=pairs,
                                                  coarse_out=oc, gate_c=gc, gate_f=gf))
    if vsa.device_error(reset=True):
        raise RuntimeError("device error word set while timing the coarse output / gated fine stage")
    n, real = wl.ncubes, wl.tokens
    pool_bytes = 3 * wl.B * real * wl.heads * wl.D * 2   # the real tokens of q, k, v, read once
    attn_flops = 4.0 * wl.B * wl.heads * n * n * wl.D   # scores and weighted sum, fp32 FMA
    return {
        "coarse_attn": {"ms_median": ca_ms, "algorithmic_bytes": pool_bytes, "fp32_flops": attn_flops,
                        "note": "pooled means of q, k, v (HBM) + cube-level attention (fp32 FMA)"},
        "sparse_attn_fwd_gated": {"ms_median": fg_ms, "effective_tflops": wl.fine_flops() / (fg_ms * 1e-3) / 1e12,
                                  "extra_hbm_bytes": 2 * wl.B * wl.s_pad * wl.heads * wl.D * 2,
                                  "note": "fine stage + gate_c * coarse + gate_f * fine in the epilogue"},
        "quality": quality,
    }


def selection_quality(vsa, torch, wl, qt, kt, vt, idx, vbs, pairs, stream):
    """Quality of the coarse selection against dense attention, measured with
    the fine stage itself: the dense reference selects every cube (topk = N).
    recall = mean over real query rows of exp(lse_selected - lse_dense), the
    share of each row's dense softmax mass its selection captures; rel_l1 =
    mean |o_sparse - o_dense| / mean |o_dense| over real rows; max_prob = the
    mean largest softmax weight of the selected rows."""
    N = wl.ncubes
    if N > 1024:
        return None  # the fine stage takes at most 1024 cubes per row
    dense = vsa.all_cubes(wl.B, wl.heads, N, device=qt.device)
    o_s, lse_s, mp = vsa.sparse_attn_fwd_peak(qt, kt, vt, idx, vbs, wl.sm_scale, pairs=pairs)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    o_d, lse_d = vsa.sparse_attn_fwd(qt, kt, vt, dense, vbs, wl.sm_scale)  # warm-up
    a.record(stream)
    o_d, lse_d = vsa.sparse_attn_fwd(qt, kt, vt, dense, vbs, wl.sm_scale, out=o_d, lse=lse_d)
    b.record(stream)
    torch.cuda.synchronize()
    if vsa.device_error(reset=True):
        raise RuntimeError("device error word set during the dense reference run")
    real = (torch.arange(64, device=qt.device)[None, :] < vbs[:, None]).reshape(-1)  # [S_pad] real slots
    cm = torch.exp(lse_s.double() - lse_d.double())[..., real]
    diff = (o_s.float() - o_d.float()).abs()[:, real]
    dense_flops = 4.0 * wl.B * wl.s_pad * N * 64 * wl.D * wl.heads
    return {"recall_captured_mass_mean": float(cm.mean()), "recall_captured_mass_p05": float(cm.quantile(0.05)),
            "rel_l1_vs_dense": float(diff.mean() / o_d.float().abs()[:, real].mean()),
            "max_prob_mean": float(mp[..., real].double().mean()),
            "dense_reference_ms": a.elapsed_time(b),
            "dense_reference_tflops": dense_flops / (a.elapsed_time(b) * 1e-3) / 1e12,
            "note": "dense reference = the fine stage with every cube selected; real query rows only"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffer) leg")
    ap.add_argument("--workload", choices=sorted(LABELS), default=WORKLOAD,
                    help="the Wan2.2 shape (default; the benchmark workload) or another configuration")
    ap.add_argument("--topk", type=int, default=0, help="override the workload's topk")
    ap.add_argument("--heads", type=int, default=0,
                    help="profiling only: run the Wan grid with this many heads instead of 40")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    from block_sparse_video_vsa_gb300 import synth
    if args.workload == "blocks128":
        return main_blocks(args, rank, world, local_rank)
    wl = synth.WORKLOADS[args.workload]
    if args.topk > 0:
        wl = wl.with_topk(args.topk)
    if args.heads > 0:
        wl = dataclasses.replace(wl, heads=args.heads)

    if args.impl == "reference":
        if rank != 0:
            return 0
        inputs = synth.make_inputs(wl)
        print(json.dumps(reference_arm(args, wl, inputs)), flush=True)
        return 0

    import torch
    dist = None
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl")
        dist = tdist
    from block_sparse_video_vsa_gb300 import build as vbuild
    if not vbuild.up_to_date() and rank == 0:
        vbuild.build()
    if dist:
        dist.barrier()

    inputs = synth.make_inputs(wl)
    ms_step, stage, clocks, (e2e_ms, h2d, d2h, copy_ms), launches, nxt, executed = run_ours(args, wl, inputs, rank,
                                                                                            world, dist)

    burst, sustained, hbm, peak_kind = load_peaks()
    flops = wl.fine_flops()
    fine_ms = statistics.mean(stage["sparse_attn_fwd"])
    fine_tflops = flops / (fine_ms * 1e-3) / 1e12
    value = whole_job_throughput(world, flops, ms_step)
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_of(wl),
        "fine_kernel": {
            "ms_per_call_mean": fine_ms, "ms_per_call_median": statistics.median(stage["sparse_attn_fwd"]),
            "effective_tflops": fine_tflops, "frac_of_burst_peak": fine_tflops / burst,
            "frac_of_sustained_peak": fine_tflops / sustained,
            # The pair tiles also compute the keys of the other cube's selection
            # (the union walk): the tensor-core work issued, its rate, and the
            # selected share of it.
            "executed_tensor_flops": executed,
            "executed_tflops": None if executed is None else executed / (fine_ms * 1e-3) / 1e12,
            "executed_frac_of_burst_peak": None if executed is None else executed / (fine_ms * 1e-3) / 1e12 / burst,
            "selected_share_of_executed": None if executed is None else flops / executed},
        "stages_ms_median": {k: statistics.median(v) for k, v in stage.items()},
        "stages_hbm_gbs": {k: b / (statistics.median(stage[k]) * 1e-3) / 1e9
                           for k, b in stage_bytes(wl).items()},
        "hbm_peak_gbs": hbm,
        "roofline": {"bound": "tensor", "achieved": fine_tflops, "peak": burst, "unit": "TFLOP/s",
                     "frac": fine_tflops / burst,
                     "traffic": fine_traffic() if wl.heads == 40 else None,
                     "peak_kind": f"{peak_kind} dense bf16 burst",
                     "kernel": "fine_fwd_kernel (vsa_sparse_attn_fwd_raster)"},
        "e2e": None if e2e_ms is None else {
            "value": whole_job_throughput(world, flops, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            # copies_only_ms_per_step: the same uploads and read-backs with no
            # compute (the host link's floor); runs_ms_per_step: every run
            **copy_ms},
        "gpu_launches": launches,
        "next_rows": nxt,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_oracle_sample(wl, inputs, args.cpu_budget)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main_blocks(args, rank, world, local_rank):
    """--workload blocks128 (the reference arm times the oracle's fine stage on it)."""
    if args.impl == "reference":
        if rank != 0:
            return 0
        from block_sparse_video_vsa_gb300 import synth
        import oracle
        wl, s_len = synth.SEQUENCE_WORKLOADS["blocks128"]
        inputs = synth.make_sequence_inputs("blocks128")
        idx, cnt, _ = oracle.block_select_cdf(inputs["q"], inputs["k"], 128, BLOCKS_TAU, wl.sm_scale)
        table, counts = oracle.blocks_to_cube_lut(idx, cnt)
        times, flops, used = [], 0.0, 0
        rng = np.random.default_rng(1)
        per_step = 2 * oracle.default_threads()
        for s in range(args.warmup + args.steps):
            units = rng.choice(counts.size, size=per_step, replace=False).astype(np.int64)
            t0 = time.perf_counter()
            _, _, used = oracle.fine_counts(inputs["q"], inputs["k"], inputs["v"], table, counts, inputs["vbs"],
                                            wl.sm_scale, units)
            if s >= args.warmup:
                times.append(time.perf_counter() - t0)
                flops += blocks_flops(counts.reshape(-1)[units], wl.D)
        value = flops / sum(times) / 1e12
        desc = f"fine stage on {per_step} random query cubes of {counts.size} per step"
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{LABELS['blocks128']}: tau={BLOCKS_TAU}"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)
        return 0
    import torch
    dist = None
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl")
        dist = tdist
    from block_sparse_video_vsa_gb300 import build as vbuild
    if not vbuild.up_to_date() and rank == 0:
        vbuild.build()
    if dist:
        dist.barrier()
    result = run_blocks(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

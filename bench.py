#!/usr/bin/env python3
"""Benchmark: causal SWA forward band-only useful TFLOP/s at the Mistral-7B shape on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--all] [--no-cpu-baseline] [--no-e2e]

One step = one forward call of the hot path over one batch of synthetic, seeded bf16
input (i.i.d. N(0,1), layout [B, H, N, d]) that is already resident in HBM.  The default
workload is the Mistral-7B-shaped causal SWA layer (B=1, Hq=32, Hkv=8, N=16384, d=128,
W=4096).  Its inputs plus output (320 MiB) exceed the 126 MB L2, so no flush is needed
between steps.  Useful FLOPs count only allowed (query, key) pairs: 4 d per pair per
query head.

Rank 0 prints one JSON line.  Under torchrun (N > 1) every rank runs its own replica of
the workload (weak scaling, no data-path collective); the timed region is bracketed by a
barrier and device synchronisation, and the time is the maximum over ranks.

``--impl reference`` times the fp64 CPU oracle (the only reference this method has) on
the host cores over bounded row samples of the same workload.

Other workloads (``--workload``, or ``--all`` for one line each): the Gemma-3-shaped layers
and ``gemma_group`` (one step = the 5:1 group: five W=1024 layers and one full-causal layer),
local + strided, window plus a global prefix, the differential forms, decode against a
rolling cache, and the backward calls: ``mistral_swa_bwd`` (one step = one swa_attn_bwd call of
the Mistral-shaped layer), ``strided_bwd`` (strided_attn_bwd at the strided workload's shape)
and ``diff_swa_bwd`` (diff_attn_bwd at the windowed differential workload's shape), each with
the forward's outputs and log-sum-exps computed once beforehand.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import swa_inputs  # noqa: E402
from sparse_causal_attention_swa_b300 import flops as flopcount  # noqa: E402

METRIC = "causal SWA fwd band-only TFLOP/s (Mistral shape, 1 B300) and % of BF16 peak"
DEFAULT_WORKLOAD = "mistral_swa"
_CSRC = "sparse_causal_attention_swa_b300/csrc/"
# device sources of each kernel family (a traffic figure is valid while they are unchanged)
KERNEL_SOURCES = {
    "attn_fwd": [_CSRC + "attn_fwd.cuh", _CSRC + "ptx.cuh"],
    "decode": [_CSRC + "decode.cuh", _CSRC + "ptx.cuh"],
    "attn_bwd": [_CSRC + "attn_bwd.cuh", _CSRC + "attn_fwd.cuh", _CSRC + "ptx.cuh"],
}
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
L2_BYTES = 126 * 2**20
FLUSH_BYTES = 256 * 2**20  # written between timed launches when a workload fits in twice L2
PREFILL_CYCLES = 20e6  # about 10 ms of device spin ahead of the timed launches (see below)

# DRAM traffic per launch of the dominant kernel, from one ncu capture (dram__bytes_read.sum
# + dram__bytes_write.sum), keyed by workload, with the hash of that kernel's device sources
# (KERNEL_SOURCES of its family) when it was taken.  A changed kernel invalidates the figure
# (reported as null).
TRAFFIC = {
    "mistral_swa": (326.28e6, "b2c86708711f2362"),
    "gemma_swa": (860.15e6, "b2c86708711f2362"),
    "strided": (112.13e6, "b2c86708711f2362"),
    "diff": (94.26e6, "b2c86708711f2362"),
    "diff_swa": (190.63e6, "b2c86708711f2362"),
    "global": (113.54e6, "b2c86708711f2362"),
    "swa_small": (0.48e6, "b2c86708711f2362"),
    # the backward calls: every kernel of one call (delta, dk/dv, dq, and the compact-key and
    # differential extras); Q, dO, K and V are read by both the dk/dv and the dq kernel
    "mistral_swa_bwd": (1124.93e6, "14ee695434112f38"),
    "strided_bwd": (481.59e6, "14ee695434112f38"),
    "diff_swa_bwd": (886.35e6, "14ee695434112f38"),
    # both decode kernels of one step
    "mistral_decode": (501.19e6, "795ae1706564fbfa"),
}


BWD_KINDS = ("bwd", "strided_bwd", "diff_bwd")


def kernel_family(w: swa_inputs.Workload) -> str:
    if w.kind in BWD_KINDS:
        return "attn_bwd"
    return {"decode": "decode"}.get(w.kind, "attn_fwd")


def kernel_hash(family: str = "attn_fwd") -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def workload_units(w: swa_inputs.Workload):
    if w.kind == "decode":
        pos = swa_inputs.make_inputs(w)["pos"]
        return (flopcount.decode_flops(pos, w.Hq, w.d, w.W),
                flopcount.decode_bytes(pos, w.Hq, w.Hkv, w.d, w.W))
    fl = flopcount.useful_flops(w.kind, w.B, w.Hq, w.N, w.d, w.W, w.stride)
    by = flopcount.algorithmic_bytes(w.kind, w.B, w.Hq, w.Hkv, w.N, w.d,
                                     layers=w.stride + 1 if w.kind == "group" else 1)
    return fl, by


def group_layers(w: swa_inputs.Workload):
    """The layers of a "group" step: `stride` W-window layers and one full-causal layer."""
    return [w.replace(kind="swa")] * w.stride + [w.replace(kind="swa", W=w.N)]


# ------------------------------------------------------------------------------ distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, ws: int, device=None) -> float:
    """Maximum of a per-rank float over the process group (identity when ws == 1)."""
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int, device=None):
    if ws > 1:
        import torch.distributed as dist

        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None, period_ms: int = 50):
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               f"-lms={period_ms}"]
        if uuid:
            cmd.insert(1, f"--id={uuid}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "power_w_max": float(max(power)), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------ CPU oracle
def oracle_sample_rows(w: swa_inputs.Workload, n_rows: int, seed: int) -> np.ndarray:
    """A bounded, seeded sample of query rows spread over the sequence."""
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(w.N, size=min(n_rows, w.N), replace=False)).astype(np.int64)


def sample_flops(w: swa_inputs.Workload, rows: np.ndarray) -> float:
    i = rows.astype(np.int64)
    if w.kind == "group":
        return sum(sample_flops(lw, rows) for lw in group_layers(w))
    if w.kind == "swa":
        per = np.minimum(i + 1, w.W)
        return 4.0 * w.d * float(per.sum()) * w.B * w.Hq
    if w.kind == "strided":
        lo = np.maximum(0, i - w.W + 1)
        per = np.minimum(i + 1, w.W) + np.where(lo > 0, (lo - 1) // w.stride + 1, 0)
        return 4.0 * w.d * float(per.sum()) * w.B * w.Hq
    if w.kind == "global":
        lo = np.maximum(0, i - w.W + 1)
        per = np.minimum(i + 1, w.W) + np.minimum(lo, w.stride)
        return 4.0 * w.d * float(per.sum()) * w.B * w.Hq
    return 8.0 * w.d * float(np.minimum(i + 1, w.W).sum()) * w.B * w.Hq


def run_oracle_rows(w, inp, rows, nthreads: int = 0):
    import oracle

    if w.kind == "group":  # every layer of the group, each one really computed
        out = None
        for lw in group_layers(w):
            out = run_oracle_rows(lw, inp, rows, nthreads)
        return out
    if w.kind == "diff":
        return oracle.diff(inp["q1"], inp["k1"], inp["q2"], inp["k2"], inp["v"], w.lam, w.scale,
                           rows=rows, W=w.W, nthreads=nthreads)
    kind = {"swa": "window", "strided": "strided", "global": "global"}[w.kind]
    return oracle.attn(inp["q"], inp["k"], inp["v"], w.W, w.scale, kind=kind, stride=w.stride,
                       rows=rows, nthreads=nthreads)


def oracle_inputs_f64(inp):
    """Widen the bf16 inputs once, so the timed oracle calls measure its arithmetic."""
    return {n: swa_inputs.bf16_bits_to_f64(a) for n, a in inp.items()}


def cpu_baseline_decode(w, inp, budget_s: float = 15.0):
    """The oracle's decode on the host cores over a bounded sample of the sequences."""
    import oracle

    oracle.build()
    t0 = time.perf_counter()
    oracle.decode(inp["q"][:1], inp["kc"][:1], inp["vc"][:1], inp["pos"][:1], w.W, w.scale)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(max(1, min(w.B, budget_s / dt)))
    t0 = time.perf_counter()
    oracle.decode(inp["q"][:n], inp["kc"][:n], inp["vc"][:n], inp["pos"][:n], w.W, w.scale)
    dt = time.perf_counter() - t0
    fl = flopcount.decode_flops(inp["pos"][:n], w.Hq, w.d, w.W)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"the first {n} of {w.B} sequences of {w.name} ({fl:.3e} useful FLOPs, "
                      f"{dt:.1f} s, fp64, one thread)"}


def bwd_prefix(w, inp, n_rows: int):
    """The backward restricted to the first n_rows positions of the first batch entry (all
    heads): with causal windows those rows and keys form a complete problem of their own."""
    return {n: np.ascontiguousarray(a[:1, :, :n_rows]) for n, a in inp.items()}


def run_oracle_bwd(w, inp, n_rows: int) -> float:
    """Run the oracle's gradients on a prefix sub-problem; returns its useful FLOPs."""
    import oracle

    sub = bwd_prefix(w, inp, n_rows)
    if w.kind == "diff_bwd":
        oracle.diff_bwd(sub["q1"], sub["k1"], sub["q2"], sub["k2"], sub["v"], w.lam, sub["dout"],
                        w.W, w.scale)
    elif w.kind == "strided_bwd":
        oracle.attn_bwd(sub["q"], sub["k"], sub["v"], sub["dout"], w.W, w.scale, kind="strided",
                        stride=w.stride)
    else:
        oracle.attn_bwd(sub["q"], sub["k"], sub["v"], sub["dout"], w.W, w.scale)
    return flopcount.useful_flops(w.kind, 1, w.Hq, n_rows, w.d, w.W, w.stride)


def bwd_sample_rows(w, inp, budget_s: float) -> int:
    """Prefix length whose oracle backward takes about budget_s seconds."""
    n = min(w.N, 1024)  # large enough that thread start-up does not dominate the probe
    t0 = time.perf_counter()
    fl = run_oracle_bwd(w, inp, n)
    dt = max(time.perf_counter() - t0, 1e-3)
    # cost grows with the useful work (the allowed pairs) of the prefix
    per_flop = dt / fl

    def work(m):
        return flopcount.useful_flops(w.kind, 1, w.Hq, m, w.d, w.W, w.stride)

    while n < w.N and work(min(w.N, 2 * n)) * per_flop < budget_s:
        n = min(w.N, 2 * n)
    return n


def cpu_baseline_bwd(w, inp, budget_s: float = 15.0):
    import oracle

    oracle.build()
    inp = oracle_inputs_f64(inp)
    n = bwd_sample_rows(w, inp, budget_s)
    t0 = time.perf_counter()
    fl = run_oracle_bwd(w, inp, n)
    dt = time.perf_counter() - t0
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": min(oracle.max_threads(), w.Hkv),
            "kind": "oracle",
            "sample": f"the first {n} positions of all {w.Hq} heads of {w.name} ({fl:.3e} useful "
                      f"FLOPs, {dt:.1f} s, fp64, one thread per KV head)"}


def cpu_baseline(w, inp, budget_s: float = 15.0):
    """Time the oracle as it stands on the host cores over a bounded row sample."""
    import oracle

    if w.kind == "decode":
        return cpu_baseline_decode(w, inp, budget_s)
    if w.kind in BWD_KINDS:
        return cpu_baseline_bwd(w, inp, budget_s)
    oracle.build()
    inp = oracle_inputs_f64(inp)
    probe = oracle_sample_rows(w, 4, seed=w.seed)
    t0 = time.perf_counter()
    run_oracle_rows(w, inp, probe)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(max(4, min(w.N, 4 * budget_s / dt)))
    rows = oracle_sample_rows(w, n, seed=w.seed + 1)
    t0 = time.perf_counter()
    run_oracle_rows(w, inp, rows)
    dt = time.perf_counter() - t0
    fl = sample_flops(w, rows)
    res = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
           "kind": "oracle",
           "sample": f"{rows.size} seeded random query rows x all {w.B * w.Hq} heads of "
                     f"{w.name} ({fl:.3e} useful FLOPs, {dt:.1f} s, fp64)"}
    if w.N * w.Hq * w.B <= 4096:  # the small workload: the whole of it on one core as well
        every = np.arange(w.N, dtype=np.int64)
        nt = oracle.max_threads()
        t0 = time.perf_counter()
        run_oracle_rows(w, inp, every, nthreads=1)
        dt1 = time.perf_counter() - t0
        run_oracle_rows(w, inp, every[:1], nthreads=nt)  # OpenMP keeps the last thread count
        res["one_core"] = {"value": sample_flops(w, every) / dt1 / 1e12, "unit": "TFLOP/s",
                           "seconds": dt1, "sample": "every row, one thread"}
    return res


def reference_arm(args, w, ws, rank):
    """--impl reference: the fp64 oracle on host cores, same metric and workload."""
    if rank != 0:
        return
    import oracle

    oracle.build()
    inp = oracle_inputs_f64(swa_inputs.make_inputs(w))
    fl_full, _ = workload_units(w)
    if w.kind in BWD_KINDS:
        reference_arm_bwd(args, w, ws, inp, fl_full)
        return
    # size every step so warmup + steps stay within about two minutes
    probe = oracle_sample_rows(w, 4, seed=w.seed)
    t0 = time.perf_counter()
    run_oracle_rows(w, inp, probe)
    dt = max(time.perf_counter() - t0, 1e-3)
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(w.N, 4 * per_step_budget / dt)))
    samples = [oracle_sample_rows(w, n, seed=w.seed + 10 + s)
               for s in range(args.steps + args.warmup)]
    for s in range(args.warmup):
        run_oracle_rows(w, inp, samples[s])
    fl = 0.0
    t0 = time.perf_counter()
    for s in range(args.warmup, args.warmup + args.steps):
        run_oracle_rows(w, inp, samples[s])
        fl += sample_flops(w, samples[s])
    dt = time.perf_counter() - t0
    value = fl / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, fl_full),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": f"{n} seeded random query rows x {w.B * w.Hq} heads per "
                                   f"step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def reference_arm_bwd(args, w, ws, inp, fl_full):
    import oracle

    n = bwd_sample_rows(w, inp, 120.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        run_oracle_bwd(w, inp, n)
    fl = 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fl += run_oracle_bwd(w, inp, n)
    dt = time.perf_counter() - t0
    value = fl / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, fl_full),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s",
                         "cores": min(oracle.max_threads(), w.Hkv), "kind": "oracle",
                         "sample": f"the first {n} positions of all {w.Hq} heads per step "
                                   f"(one thread per KV head)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w, fl, flush=False):
    cfg = {"workload": w.name, "kind": w.kind, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N,
           "d": w.d, "W": w.W, "scale": w.scale, "useful_flops_per_step": fl,
           "l2": ("L2 flushed (256 MiB write) before every timed launch; step time = sum of "
                  "the launches' CUDA-event durations") if flush else
                 "inputs+output larger than twice the 126 MB L2; no flush between steps"}
    if w.kind == "strided":
        cfg["stride"] = w.stride
    if w.kind == "global":
        cfg["n_global"] = w.stride
    if w.kind == "group":
        cfg["layers"] = (f"{w.stride} causal SWA layers with W={w.W} and one full-causal layer "
                         f"(W=N), each a swa_attn_fwd call on the same inputs")
        cfg["flop_convention"] = "4 d per allowed (row, key) pair, summed over the group's layers"
    if w.kind == "strided_bwd":
        cfg["stride"] = w.stride
        cfg["flop_convention"] = ("10 d per allowed (row, key) pair: the products S, dP, dV, dK, "
                                  "dQ (2.5 x the forward)")
    if w.kind == "diff_bwd":
        cfg["lambda"] = w.lam
        cfg["flop_convention"] = ("20 d per (row, key) pair in the window: the five products of "
                                  "each of the two maps")
    if w.kind == "bwd":
        cfg["flop_convention"] = ("10 d per (row, key) pair in the window: the products S, dP, "
                                  "dV, dK, dQ (2.5 x the forward)")
    if w.kind == "diff":
        cfg["lambda"] = w.lam
        cfg["flop_convention"] = "8 d per (row, key) pair in the window (two attention maps)"
    return cfg


# ------------------------------------------------------------------------------ GPU arm
def to_device(inp, dev):
    import torch

    return {n: (torch.from_numpy(a).to(dev) if a.dtype == np.int32 else
                torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev))
            for n, a in inp.items()}


_WORKSPACES = {}


def decode_workspace(pkg, w, dev):
    import torch

    key = (w.name, str(dev))
    if key not in _WORKSPACES:
        n = pkg.swa_decode_workspace_bytes(w.B, w.Hq, w.W, w.d)
        _WORKSPACES[key] = torch.empty(n, dtype=torch.uint8, device=dev)
    return _WORKSPACES[key]


def launch(pkg, w, t, out, stream):
    if w.kind == "decode":
        ws = decode_workspace(pkg, w, t["q"].device)
        pkg.swa_decode_fwd(t["q"], t["kc"], t["vc"], t["pos"], out, w.B, w.Hq, w.Hkv, w.W, w.d,
                           w.scale, ws, ws.numel(), stream)
    elif w.kind == "swa":
        pkg.swa_attn_fwd(t["q"], t["k"], t["v"], out, w.B, w.Hq, w.Hkv, w.N, w.d, w.W, w.scale,
                         stream)
    elif w.kind == "group":  # the window layers, then the full-causal layer
        for lw in group_layers(w):
            pkg.swa_attn_fwd(t["q"], t["k"], t["v"], out, lw.B, lw.Hq, lw.Hkv, lw.N, lw.d, lw.W,
                             lw.scale, stream)
    elif w.kind == "strided":
        pkg.strided_attn_fwd(t["q"], t["k"], t["v"], out, w.B, w.Hq, w.Hkv, w.N, w.d, w.W,
                             w.stride, w.scale, stream)
    elif w.kind == "global":
        pkg.global_attn_fwd(t["q"], t["k"], t["v"], out, w.B, w.Hq, w.Hkv, w.N, w.d, w.W,
                            w.stride, w.scale, stream)
    elif w.kind == "bwd":  # out receives dq
        pkg.swa_attn_bwd(t["q"], t["k"], t["v"], t["out_fwd"], t["lse"], t["dout"], out, t["dk"],
                         t["dv"], w.B, w.Hq, w.Hkv, w.N, w.d, w.W, w.scale, t["ws"],
                         t["ws"].numel(), stream)
    elif w.kind == "strided_bwd":  # out receives dq
        pkg.strided_attn_bwd(t["q"], t["k"], t["v"], t["out_fwd"], t["lse"], t["dout"], out,
                             t["dk"], t["dv"], w.B, w.Hq, w.Hkv, w.N, w.d, w.W, w.stride, w.scale,
                             t["ws"], t["ws"].numel(), stream)
    elif w.kind == "diff_bwd":  # out receives dq1
        pkg.diff_attn_bwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], w.lam, None, t["out1"],
                          t["lse1"], t["out2"], t["lse2"], t["dout"], out, t["dk1"], t["dq2"],
                          t["dk2"], t["dv"], t["dlam"], w.B, w.Hq, w.Hkv, w.N, w.d, w.W, w.scale,
                          t["ws"], t["ws"].numel(), stream)
    elif w.W < w.N:
        pkg.diff_swa_attn_fwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], w.lam, None, out, w.B,
                              w.Hq, w.Hkv, w.N, w.d, w.W, w.scale, stream)
    else:
        pkg.diff_attn_fwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], w.lam, out, w.B, w.Hq,
                          w.Hkv, w.N, w.d, w.scale, stream)


def bwd_buffers(pkg, w, t, stream):
    """Device buffers of a backward step besides its inputs: the forward's outputs and row
    log-sum-exps (computed here, once, by the forward calls), the workspace and the gradients
    other than the first (which the step's `out` receives).  Returns the names of the tensors
    a step writes, besides `out`."""
    import torch

    if w.kind == "diff_bwd":
        q1 = t["q1"]
        for m, (qq, kk) in enumerate(((q1, t["k1"]), (t["q2"], t["k2"])), start=1):
            t[f"out{m}"] = torch.empty_like(qq)
            t[f"lse{m}"] = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=q1.device)
            pkg.swa_attn_fwd_lse(qq, kk, t["v"], t[f"out{m}"], t[f"lse{m}"], w.B, w.Hq, w.Hkv, w.N,
                                 w.d, w.W, w.scale, stream)
        nb = pkg.diff_attn_bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.d)
        t["ws"] = torch.empty(nb, dtype=torch.uint8, device=q1.device)
        t["dq2"] = torch.empty_like(q1)
        t["dk1"] = torch.empty_like(t["k1"])
        t["dk2"] = torch.empty_like(t["k2"])
        t["dv"] = torch.empty_like(t["v"])
        t["dlam"] = torch.empty(w.Hq, dtype=torch.float32, device=q1.device)
        return ["dk1", "dq2", "dk2", "dv", "dlam"]
    q = t["q"]
    t["out_fwd"] = torch.empty_like(q)
    t["lse"] = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=q.device)
    if w.kind == "strided_bwd":
        pkg.strided_attn_fwd_lse(q, t["k"], t["v"], t["out_fwd"], t["lse"], w.B, w.Hq, w.Hkv,
                                 w.N, w.d, w.W, w.stride, w.scale, stream)
        nb = pkg.strided_attn_bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.d, w.W, w.stride)
    else:
        pkg.swa_attn_fwd_lse(q, t["k"], t["v"], t["out_fwd"], t["lse"], w.B, w.Hq, w.Hkv, w.N,
                             w.d, w.W, w.scale, stream)
        nb = pkg.swa_attn_bwd_workspace_bytes(w.B, w.Hq, w.N)
    t["ws"] = torch.empty(nb, dtype=torch.uint8, device=q.device)
    t["dk"] = torch.empty_like(t["k"])
    t["dv"] = torch.empty_like(t["v"])
    return ["dk", "dv"]


def bench_workload(args, w, ws, rank, dev, want_cpu, want_e2e):
    import torch

    import sparse_causal_attention_swa_b300 as pkg

    pkg.load()
    inp = swa_inputs.make_inputs(w)
    t = to_device(inp, dev)
    first = t["q1"] if w.kind in ("diff", "diff_bwd") else t["q"]
    out = torch.empty_like(first)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    if w.kind in BWD_KINDS:
        bwd_buffers(pkg, w, t, sh)
    fl, algo_bytes = workload_units(w)

    for _ in range(args.warmup):
        launch(pkg, w, t, out, sh)
    torch.cuda.synchronize(dev)
    if pkg.swa_device_status(sh) != 0:
        raise RuntimeError("kernel watchdog fired during warm-up")

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if uuid and not uuid.startswith("GPU-"):
            uuid = "GPU-" + uuid
    except Exception:
        uuid = None
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(uuid)
    time.sleep(0.3)  # let the sampler start
    barrier(ws, dev)
    torch.cuda.synchronize(dev)
    flush = algo_bytes < 2 * L2_BYTES
    scratch = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev) if flush else None
    # keep host time out of the events: a device-side spin of a few ms holds the stream while
    # the host enqueues every timed launch, so no launch waits for its host-side call
    torch.cuda._sleep(int(PREFILL_CYCLES))
    t_begin.record(stream)
    for s in range(args.steps):
        if flush:
            scratch.fill_(s)  # evict the previous step's lines from L2
        starts[s].record(stream)
        launch(pkg, w, t, out, sh)
        ends[s].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws, dev)
    clk = clocks.stop()
    if pkg.swa_device_status(sh) != 0:
        raise RuntimeError("kernel watchdog fired during the timed region")
    per_launch = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    launch_ms = float(np.mean(per_launch))
    # with a flush between launches the step time is the sum of the launches alone
    total_ms = float(np.sum(per_launch)) if flush else t_begin.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, ws, dev)
    launch_ms = max_over_ranks(launch_ms, ws, dev)
    ms_per_step = total_ms / args.steps
    value = fl * ws / (ms_per_step * 1e-3) / 1e12

    peaks, peak_src = load_peaks()
    bf16_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved_tf = fl / (launch_ms * 1e-3) / 1e12
    tkey = TRAFFIC.get(w.name)
    traffic = tkey[0] if (tkey and tkey[1] == kernel_hash(kernel_family(w))) else None
    # the bound is whichever floor is higher: the tensor time of the useful FLOPs or the
    # HBM time of the algorithmic bytes (below the ridge, e.g. local + strided, it is HBM)
    t_tensor = fl / (bf16_peak * 1e12)
    t_hbm = algo_bytes / (hbm_peak * 1e9)
    mode = {"swa": 0, "group": 0, "strided": 1, "global": 1, "diff": 2}.get(w.kind)
    if w.kind == "bwd":
        kname = (f"bwd_delta_kernel<{w.d}> + attn_bwd_kernel<{w.d},0> (dk, dv) + "
                 f"attn_bwd_kernel<{w.d},1> (dq), one call")
    elif w.kind == "strided_bwd":
        kname = (f"bwd_delta_kernel<{w.d}> + attn_bwd_kernel<{w.d},2> (dk, dv of the strided "
                 f"keys) + bwd_compact_reduce_kernel + attn_bwd_kernel<{w.d},0> + "
                 f"attn_bwd_kernel<{w.d},1>, one call")
    elif w.kind == "diff_bwd":
        kname = (f"2 x bwd_delta_kernel<{w.d}> + 2 x attn_bwd_kernel<{w.d},0> + 2 x "
                 f"attn_bwd_kernel<{w.d},1> + bwd_dlam_kernel, one call")
    elif w.kind == "decode":
        kname = (f"decode_mma_kernel<{w.Hq // w.Hkv}> + decode_combine_kernel<{w.d}>" if w.d == 128
                 else f"decode_split_kernel<{w.d}> + decode_combine_kernel<{w.d}>")
    elif w.kind == "group":
        kname = (f"attn_fwd_kernel<{w.d},0>, {w.stride} launches with W={w.W} and one with "
                 f"W=N per step")
    else:
        kname = f"attn_fwd_kernel<{w.d},{mode}>"
    gbs = algo_bytes / (launch_ms * 1e-3) / 1e9
    if t_tensor >= t_hbm:
        roofline = {"bound": "tensor", "achieved": achieved_tf, "peak": bf16_peak,
                    "unit": "TFLOP/s", "frac": achieved_tf / bf16_peak, "traffic": traffic,
                    "peak_source": f"{peak_src} bf16_tflops (burst, kernel timed alone)",
                    "kernel": kname, "algorithmic_flops_per_launch": fl,
                    "hbm_gbs_algorithmic": gbs}
    else:
        roofline = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                    "frac": gbs / hbm_peak, "traffic": traffic,
                    "peak_source": f"{peak_src} hbm_gbs",
                    "kernel": kname, "algorithmic_bytes_per_launch": algo_bytes,
                    "tflops_useful": achieved_tf,
                    "tensor_frac": achieved_tf / bf16_peak}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": workload_config(w, fl, flush),
        "pct_of_bf16_peak": 100.0 * achieved_tf / bf16_peak,
        "roofline": roofline,
        "gpu_launches": args.steps * {"decode": 2, "bwd": 3, "strided_bwd": 5, "diff_bwd": 7,
                                      "group": w.stride + 1}.get(w.kind, 1),
        "clocks": clk,
    }
    if ws > 1:
        line["config"]["parallelism"] = f"replicas x{ws} (independent problems per rank)"

    if want_e2e:
        line["e2e"] = e2e_measure(args, w, inp, pkg, dev, ws)
    if want_cpu and rank == 0 and ws == 1:
        line["cpu_baseline"] = cpu_baseline(w, inp)
    return line


def e2e_measure(args, w, inp, pkg, dev, ws):
    """Same metric through the public API with host buffers: every step copies its inputs in
    from pinned host memory, makes the C-ABI call and copies its result back, all inside the
    timed region.  The steps are pipelined as a serving loop would run them: two device buffer
    sets, the uploads on one stream and the downloads on another, so step s+1's upload and step
    s-1's download overlap step s's kernels (the two PCIe directions run at once)."""
    import torch

    host = {n: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
            for n, a in inp.items()}
    sets = [{n: torch.empty_like(h, device=dev) for n, h in host.items()} for _ in range(2)]
    cs = torch.cuda.current_stream(dev)
    sh = cs.cuda_stream
    first = "q1" if w.kind in ("diff", "diff_bwd") else "q"
    outs = [torch.empty_like(t[first]) for t in sets]
    results = [[o] for o in outs]
    if w.kind in BWD_KINDS:
        # the forward's outputs and log-sum-exps are inputs of the backward: made once on the
        # device, then copied from pinned host buffers every step like the inputs and dout
        for t in sets:
            for n in host:
                t[n].copy_(host[n])
        written = [bwd_buffers(pkg, w, t, sh) for t in sets]
        torch.cuda.synchronize(dev)
        fwd_names = ("out1", "lse1", "out2", "lse2") if w.kind == "diff_bwd" else ("out_fwd", "lse")
        for n in fwd_names:
            host[n] = sets[0][n].cpu().pin_memory()
        results = [[outs[b]] + [sets[b][n] for n in written[b]] for b in range(2)]
    res_host = [[torch.empty(r.shape, dtype=r.dtype).pin_memory() for r in results[b]]
                for b in range(2)]
    h2d = sum(h.numel() * h.element_size() for h in host.values())
    d2h = sum(r.numel() * r.element_size() for r in results[0])
    steps = max(3, min(args.steps, 20))
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_k = [torch.cuda.Event() for _ in range(2)]    # a set's kernels are done
    ev_out = [torch.cuda.Event() for _ in range(2)]  # a set's results have been read back
    started = [False, False]

    def step(k):
        b = k % 2
        with torch.cuda.stream(up):
            if started[b]:
                up.wait_event(ev_k[b])  # the kernels of step k-2 have read this set
            for n in host:
                sets[b][n].copy_(host[n], non_blocking=True)
        ev_in = torch.cuda.Event()
        ev_in.record(up)
        cs.wait_event(ev_in)
        if started[b]:
            cs.wait_event(ev_out[b])  # step k-2's results have left this set
        launch(pkg, w, sets[b], outs[b], sh)
        ev_k[b].record(cs)
        with torch.cuda.stream(down):
            down.wait_event(ev_k[b])
            for r, rh in zip(results[b], res_host[b]):
                rh.copy_(r, non_blocking=True)
        ev_out[b].record(down)
        started[b] = True

    for k in range(2):
        step(k)
    torch.cuda.synchronize(dev)
    barrier(ws, dev)
    a = torch.cuda.Event(enable_timing=True)
    bend = torch.cuda.Event(enable_timing=True)
    a.record(cs)
    up.wait_event(a)
    for k in range(steps):
        step(k)
    cs.wait_event(ev_out[(steps - 1) % 2])
    cs.wait_event(ev_out[(steps - 2) % 2])
    bend.record(cs)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(a.elapsed_time(bend) / steps, ws, dev)
    fl, _ = workload_units(w)
    return {"value": fl * ws / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "steps": steps,
            "pipeline": "two device buffer sets; uploads and downloads on their own streams "
                        "overlap the neighbouring steps' kernels"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(swa_inputs.WORKLOADS))
    ap.add_argument("--all", action="store_true",
                    help="one line per workload (measurement sweep, not the headline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    ws, rank, local = dist_env()
    w = swa_inputs.WORKLOADS[args.workload]

    if args.impl == "reference":
        reference_arm(args, w, ws, rank)
        return 0

    import torch

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    names = sorted(swa_inputs.WORKLOADS) if args.all else [args.workload]
    for name in names:
        line = bench_workload(args, swa_inputs.WORKLOADS[name], ws, rank, dev,
                              want_cpu=not args.no_cpu_baseline and not args.all,
                              want_e2e=not args.no_e2e)
        if rank == 0:
            print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds no attention arithmetic.  It only knows the workload shapes
and how to draw their inputs: i.i.d. N(0, 1) samples in fp32 from
``numpy.random.default_rng(seed)``, drawn in the order the tensors are listed
(q, k, v; or q1, k1, q2, k2, v), then rounded to bf16 with round-to-nearest-
even.  Both sides consume the *same* bf16 bytes (as uint16 bit patterns), so a
parity difference can only come from the arithmetic.

Tensors use the layout ``[B, H, N, d]`` contiguous; q / out carry ``Hq`` heads
and k / v carry ``Hkv`` heads.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

SEED_BASE = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: the sizes of one call of the hot path."""

    name: str
    kind: str  # "swa" | "strided" | "diff" | "decode" | "global" | "group" | "bwd" |
    #            "strided_bwd" | "diff_bwd"
    # (for "strided" the stride field is the stride; for "global" it is the number of global
    # prefix tokens; for "group" it is the number of W-window layers per full-causal layer)
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    W: int
    stride: int = 0
    lam: float = 0.0
    sink_shift: float = 0.0  # added to K1[:, :, 0, :] before rounding (diff only)
    seed_index: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def seed(self) -> int:
        return SEED_BASE + self.seed_index

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The workloads of the measurements (and the full-size parity cases).  Index = the seed offset.
WORKLOADS = {
    # small causal SWA case: B=1, H=2, N=512, d=64, W=64
    "swa_small": Workload("swa_small", "swa", 1, 2, 2, 512, 64, 64, seed_index=1),
    # Mistral-7B-shaped causal SWA: GQA 32/8, N=16384, d=128, W=4096
    "mistral_swa": Workload("mistral_swa", "swa", 1, 32, 8, 16384, 128, 4096, seed_index=2),
    # Gemma-3-shaped pair: W=1024 layer and a global (full causal, W=N) layer
    "gemma_swa": Workload("gemma_swa", "swa", 2, 16, 8, 32768, 128, 1024, seed_index=3),
    "gemma_global": Workload("gemma_global", "swa", 2, 16, 8, 32768, 128, 32768, seed_index=3),
    # the Gemma-3 5:1 group: five W=1024 layers and one full-causal layer on the same inputs
    "gemma_group": Workload("gemma_group", "group", 2, 16, 8, 32768, 128, 1024, stride=5,
                            seed_index=3),
    # local + strided sparse causal attention
    "strided": Workload("strided", "strided", 1, 16, 16, 16384, 64, 256, stride=128, seed_index=4),
    # differential causal attention with an attention sink on key 0 of K1
    "diff": Workload("diff", "diff", 1, 16, 16, 8192, 64, 8192, lam=0.8, sink_shift=3.0,
                     seed_index=5),
    # a differential head inside an SWA layer: both maps under a W=1024 window
    "diff_swa": Workload("diff_swa", "diff", 1, 16, 16, 16384, 64, 1024, lam=0.8, sink_shift=3.0,
                         seed_index=8),
    # backward pass of the Mistral-shaped SWA layer: q, k, v as the forward, plus dL/dout
    "mistral_swa_bwd": Workload("mistral_swa_bwd", "bwd", 1, 32, 8, 16384, 128, 4096,
                                seed_index=9),
    # backward of local + strided attention at the strided workload's shape, plus dL/dout
    "strided_bwd": Workload("strided_bwd", "strided_bwd", 1, 16, 16, 16384, 64, 256, stride=128,
                            seed_index=10),
    # backward of the windowed differential workload (both maps, lambda 0.8), plus dL/dout
    "diff_swa_bwd": Workload("diff_swa_bwd", "diff_bwd", 1, 16, 16, 16384, 64, 1024, lam=0.8,
                             sink_shift=3.0, seed_index=11),
    # window plus a global prefix (Longformer-style [CLS] / question tokens): W=512, 64 global
    "global": Workload("global", "global", 1, 16, 16, 16384, 64, 512, stride=64, seed_index=7),
    # decode against a W-slot rolling KV cache, Mistral-7B heads: one new query per
    # sequence, 32 sequences at positions drawn from [0, N); N = 4 W, so most windows
    # are full (W cache rows) and some are still filling
    "mistral_decode": Workload("mistral_decode", "decode", 32, 32, 8, 16384, 128, 4096,
                               seed_index=6),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    return r


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    return bf16_bits_to_f32(h).astype(np.float64)


def _normal_bf16(rng: np.random.Generator, shape, shift_row0: float = 0.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if shift_row0:
        x[:, :, 0, :] += np.float32(shift_row0)
    return f32_to_bf16_bits(x)


def tensor_names(kind: str) -> tuple[str, ...]:
    if kind == "decode":
        return ("q", "kc", "vc")
    if kind == "diff_bwd":
        return ("q1", "k1", "q2", "k2", "v", "dout")
    if kind in ("bwd", "strided_bwd"):
        return ("q", "k", "v", "dout")
    return ("q1", "k1", "q2", "k2", "v") if kind == "diff" else ("q", "k", "v")


def make_inputs(w: Workload, seed: int | None = None) -> dict[str, np.ndarray]:
    """Draw the workload's inputs as bf16 bit patterns (uint16), layout [B, H, N, d]."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    if w.kind == "decode":
        # q: [B, Hq, d]; the W-slot caches kc, vc: [B, Hkv, W, d] hold i.i.d. N(0, 1)
        # entries (whatever history filled them); pos: [B] absolute query positions
        return {
            "q": f32_to_bf16_bits(rng.standard_normal(size=(w.B, w.Hq, w.d), dtype=np.float32)),
            "kc": _normal_bf16(rng, (w.B, w.Hkv, w.W, w.d)),
            "vc": _normal_bf16(rng, (w.B, w.Hkv, w.W, w.d)),
            "pos": rng.integers(0, w.N, size=w.B, dtype=np.int64).astype(np.int32),
        }
    qs = (w.B, w.Hq, w.N, w.d)
    ks = (w.B, w.Hkv, w.N, w.d)
    if w.kind in ("diff", "diff_bwd"):
        d = {
            "q1": _normal_bf16(rng, qs),
            "k1": _normal_bf16(rng, ks, w.sink_shift),
            "q2": _normal_bf16(rng, qs),
            "k2": _normal_bf16(rng, ks),
            "v": _normal_bf16(rng, ks),
        }
        if w.kind == "diff_bwd":  # then the upstream gradient dL/dout
            d["dout"] = _normal_bf16(rng, qs)
        return d
    if w.kind in ("bwd", "strided_bwd"):  # the forward's inputs, then dL/dout
        return {
            "q": _normal_bf16(rng, qs),
            "k": _normal_bf16(rng, ks),
            "v": _normal_bf16(rng, ks),
            "dout": _normal_bf16(rng, qs),
        }
    return {
        "q": _normal_bf16(rng, qs),
        "k": _normal_bf16(rng, ks),
        "v": _normal_bf16(rng, ks),
    }


def sample_rows(N: int, n_random: int, seed: int, tile: int = 128) -> np.ndarray:
    """Rows to check at full size: the first two and the last tile, every tile
    boundary (both sides), and ``n_random`` seeded random rows.  Sorted, unique."""
    rows = set(range(0, min(N, 2 * tile)))
    rows.update(range(max(0, N - tile), N))
    for b in range(tile, N, tile):
        rows.update((b - 1, b))
    rng = np.random.default_rng(seed)
    if n_random > 0:
        rows.update(int(x) for x in rng.integers(0, N, size=n_random))
    return np.array(sorted(r for r in rows if 0 <= r < N), dtype=np.int64)

"""Closed-form counts of allowed (query, key) pairs and the useful FLOPs built on them.

The pair counts follow the SWA note ("SWA：滑动窗口注意力与跨层信息传递", §4.1):
a full causal head of length T has T(T+1)/2 allowed pairs and a window of W
positions (counting the current one) has sum_i min(i, W) = T W - W(W-1)/2 for
T >= W.  The strided count adds, for every row i, the multiples of the stride
that lie before the row's window (the local+strided mask of the attention-
variants lesson, "Build it" step 3).

Useful FLOPs count only the allowed pairs: 2 d for q.k plus 2 d for p.v, i.e.
4 d per pair per query head; the differential variant has two attention maps
and counts 8 d per causal pair.
"""
from __future__ import annotations

import numpy as np


def pairs_window(N: int, W: int) -> int:
    """Allowed pairs of one head under the causal window of W positions."""
    if W >= N:
        return N * (N + 1) // 2
    return N * W - W * (W - 1) // 2


def pairs_causal(N: int) -> int:
    return N * (N + 1) // 2


def pairs_strided(N: int, W: int, stride: int) -> int:
    """Window pairs plus, per row, the keys 0, s, 2s, ... that precede the window."""
    i = np.arange(N, dtype=np.int64)
    lo = np.maximum(0, i - W + 1)
    win = np.minimum(i + 1, W)
    extra = np.where(lo > 0, (lo - 1) // stride + 1, 0)
    return int(win.sum() + extra.sum())


def pairs_global(N: int, W: int, n_global: int) -> int:
    """Window pairs plus, per row, the global prefix keys j < n_global that precede the window."""
    i = np.arange(N, dtype=np.int64)
    lo = np.maximum(0, i - W + 1)
    win = np.minimum(i + 1, W)
    return int(win.sum() + np.minimum(lo, n_global).sum())


def useful_flops(kind: str, B: int, Hq: int, N: int, d: int, W: int, stride: int = 0) -> float:
    """Band-only useful FLOPs of one forward call."""
    if kind == "swa":
        p = pairs_window(N, W)
        return 4.0 * d * p * B * Hq
    if kind == "strided":
        p = pairs_strided(N, W, stride)
        return 4.0 * d * p * B * Hq
    if kind == "global":  # stride carries the number of global prefix tokens
        p = pairs_global(N, W, stride)
        return 4.0 * d * p * B * Hq
    if kind == "group":  # `stride` window-W layers plus one full-causal layer
        return 4.0 * d * (stride * pairs_window(N, W) + pairs_causal(N)) * B * Hq
    if kind == "bwd":  # S, dP, dV, dK, dQ: five products of 2 d per pair (2.5 x forward)
        p = pairs_window(N, W)
        return 10.0 * d * p * B * Hq
    if kind == "strided_bwd":  # the same five products per pair of the local + strided mask
        return 10.0 * d * pairs_strided(N, W, stride) * B * Hq
    if kind == "diff_bwd":  # five products per pair for each of the two maps
        return 20.0 * d * pairs_window(N, W) * B * Hq
    if kind == "diff":  # both maps under the window W (W >= N: causal)
        p = pairs_window(N, W)
        return 8.0 * d * p * B * Hq
    raise ValueError(kind)


def decode_keys(pos, W: int) -> int:
    """Cache rows a decode step reads per (sequence, KV head): the window of position t holds
    min(t + 1, W) keys (SWA note §3.1 and §4.2)."""
    p = np.asarray(pos, dtype=np.int64)
    return int(np.minimum(p + 1, W).sum())


def decode_flops(pos, Hq: int, d: int, W: int) -> float:
    """Useful FLOPs of a decode step: 4 d per (query head, window key)."""
    return 4.0 * d * Hq * decode_keys(pos, W)


def decode_bytes(pos, Hq: int, Hkv: int, d: int, W: int) -> int:
    """HBM bytes a decode step must move: the K and V rows of every window once, the
    queries read and the outputs written (bf16)."""
    B = int(np.asarray(pos).size)
    return 2 * Hkv * d * 2 * decode_keys(pos, W) + 2 * B * Hq * d * 2


def algorithmic_bytes(kind: str, B: int, Hq: int, Hkv: int, N: int, d: int,
                      layers: int = 1) -> int:
    """HBM bytes that every correct implementation must move: inputs read once, output written
    once (bf16); a "group" of `layers` calls moves them once per call."""
    q = B * Hq * N * d * 2
    kv = B * Hkv * N * d * 2
    if kind == "group":
        return layers * (q + 2 * kv + q)
    if kind == "diff":
        return 2 * q + 3 * kv + q  # q1, q2, k1, k2, v, out
    if kind in ("bwd", "strided_bwd"):  # q, out, dout, lse (fp32), k, v read; dq, dk, dv written
        return 4 * q + 4 * kv + B * Hq * N * 4
    if kind == "diff_bwd":  # q1, q2, out1, out2, dout, lse1, lse2, k1, k2, v; dq1, dq2, dk1, dk2, dv
        return 7 * q + 6 * kv + 2 * B * Hq * N * 4
    return q + 2 * kv + q  # q, k, v, out

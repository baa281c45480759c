"""fp64 CPU oracle for causal SWA, local+strided and differential attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
CUDA product path never imports it and it never imports the product package.

The arithmetic lives in ``swa_oracle.c`` (plain C, fp64, OpenMP over rows);
this module compiles it with gcc on first use and marshals numpy arrays.
Inputs may be fp64 arrays or bf16 bit patterns (uint16, widened exactly).

Parity status per function (what pins it is listed in the tests):
  attn(kind="window")  pinned: worked example of the SWA note §3.2, pair counts
                       of §4.1, the W=4 window figure of the attention-variants
                       lesson, W >= N, W = 1, uniform-key mean, brute force.
  attn(kind="strided") pinned: brute force of the lesson's strided mask,
                       stride = 1, stride >= N, W >= N special cases, closed-form
                       pair count.
  attn(kind="causal")  pinned: worked example (full causal 38/8), brute force.
  diff                 pinned: lambda = 0, (Q2, K2) = (Q1, K1), affinity in
                       lambda, brute force of the dense (A1 - lambda A2) V.
  attn(kind="global")  pinned: n_g = 0 is the window bitwise, n_g >= N or W >= N is
                       causal, n_g = 1 equals strided with stride >= N (window plus
                       key 0), brute force of the dense mask, closed-form pair count.
                       For this kind the ``stride`` argument carries n_g.
  diff_heads           pinned: equal lambdas reproduce diff bitwise; a head with
                       lambda = 0 is that head's causal attention.
  lse                  pinned: the worked example's exponentials 1, 2, 3 (ln 6) and
                       the full causal denominator 8 (ln 8); W = 1 (the row's own
                       score); exp(lse) equals the softmax denominator used by attn
                       (weights_row); brute force on tiny inputs.
  diff_bwd             pinned: central differences of sum(dout * diff_heads(...)) for
                       every entry of dq1, dk1, dq2, dk2, dv and every head's lambda;
                       lambda = 0 gives attn_bwd for map 1 and no gradient to map 2;
                       equal maps give dq2 = -lambda dq1 and dv = (1 - lambda) x attn_bwd's.
  decode, cache_slot   pinned: the SWA note's W = 3 slot walk-through (§4.2),
                       equality with row t of attn(kind="window") over the whole
                       sequence when the cache was filled by rolling writes,
                       W > t (full causal row), W = 1 (returns v_t).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swa_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None

KINDS = {"window": 0, "strided": 1, "causal": 2, "global": 3}

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_liboracle.so`` (gcc, -O2, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c99", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_attn.restype = ctypes.c_int
            lib.oracle_attn.argtypes = [ctypes.c_int, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                        _I64, _I64, _I64, ctypes.c_double, _P, _I64,
                                        ctypes.c_int]
            lib.oracle_diff.restype = ctypes.c_int
            lib.oracle_diff.argtypes = [_P, _P, _P, _P, _P, ctypes.c_double, _P, _I64, _I64,
                                        _I64, _I64, _I64, _I64, ctypes.c_double, _P, _I64,
                                        ctypes.c_int]
            lib.oracle_weights_row.restype = ctypes.c_int
            lib.oracle_weights_row.argtypes = [ctypes.c_int, _P, _P, _I64, _I64, _I64, _I64,
                                               _I64, _I64, _I64, ctypes.c_double, _I64, _I64,
                                               _I64, _P]
            lib.oracle_pair_count.restype = ctypes.c_int64
            lib.oracle_pair_count.argtypes = [ctypes.c_int, _I64, _I64, _I64]
            lib.oracle_mask_row.restype = ctypes.c_int
            lib.oracle_mask_row.argtypes = [ctypes.c_int, _I64, _I64, _I64, _I64, _P]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64,
                                          ctypes.c_double]
            lib.oracle_lse.restype = ctypes.c_int
            lib.oracle_lse.argtypes = [ctypes.c_int, _P, _P, _P, _I64, _I64, _I64, _I64, _I64,
                                       _I64, _I64, ctypes.c_double, _P, _I64]
            lib.oracle_attn_bwd.restype = ctypes.c_int
            lib.oracle_attn_bwd.argtypes = [ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _I64,
                                            _I64, _I64, _I64, _I64, _I64, _I64,
                                            ctypes.c_double, ctypes.c_int]
            lib.oracle_attn_bwd_rows.restype = ctypes.c_int
            lib.oracle_attn_bwd_rows.argtypes = [ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _I64,
                                                 _I64, _I64, _I64, _I64, _I64, _I64,
                                                 ctypes.c_double, _P, _I64, ctypes.c_int]
            lib.oracle_diff_bwd.restype = ctypes.c_int
            lib.oracle_diff_bwd.argtypes = [_P] * 13 + [_I64] * 6 + [ctypes.c_double,
                                                                    ctypes.c_int]
            lib.oracle_cache_slot.restype = ctypes.c_int64
            lib.oracle_cache_slot.argtypes = [_I64, _I64]
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:  # bf16 bit patterns: widen exactly
        x = (x.astype(np.uint32) << 16).view(np.float32)
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _rows_arg(rows, N):
    if rows is None:
        return None, N
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r, int(r.size)


def attn(q, k, v, W: int, scale: float, kind: str = "window", stride: int = 0,
         rows=None, nthreads: int = 0) -> np.ndarray:
    """Masked attention in fp64.  q: [B, Hq, N, d]; k, v: [B, Hkv, N, d].

    Returns [B, Hq, nrows, d] (nrows = N when ``rows`` is None)."""
    lib = _load()
    q64, k64, v64 = _f64(q), _f64(k), _f64(v)
    B, Hq, N, d = q64.shape
    Hkv = k64.shape[1]
    r, nrows = _rows_arg(rows, N)
    out = np.empty((B, Hq, nrows, d), dtype=np.float64)
    rc = lib.oracle_attn(KINDS[kind], _ptr(q64), _ptr(k64), _ptr(v64), _ptr(out), B, Hq, Hkv,
                         N, d, int(W), int(stride), float(scale),
                         None if r is None else _ptr(r), nrows, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attn rejected its arguments (code {rc})")
    return out


def diff(q1, k1, q2, k2, v, lam: float, scale: float, rows=None, nthreads: int = 0,
         W: int = 0):
    """Differential attention (A1 - lam A2) V in fp64, both maps under the window mask of
    width W (0 or W >= N: the causal mask)."""
    lib = _load()
    a = [_f64(x) for x in (q1, k1, q2, k2, v)]
    B, Hq, N, d = a[0].shape
    Hkv = a[1].shape[1]
    r, nrows = _rows_arg(rows, N)
    out = np.empty((B, Hq, nrows, d), dtype=np.float64)
    Wm = N if W == 0 else int(W)
    rc = lib.oracle_diff(*[_ptr(x) for x in a], float(lam), _ptr(out), B, Hq, Hkv, N, d, Wm,
                         float(scale), None if r is None else _ptr(r), nrows, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_diff rejected its arguments (code {rc})")
    return out


def diff_heads(q1, k1, q2, k2, v, lams, scale: float, rows=None, nthreads: int = 0,
               W: int = 0):
    """Differential causal attention with one lambda per query head (the attention-variants
    lesson's exercise 4, a learnable lambda per head): head h uses lams[h].  Computed head by
    head with ``diff``."""
    q1, q2 = np.asarray(q1), np.asarray(q2)
    k1, k2, v = np.asarray(k1), np.asarray(k2), np.asarray(v)
    lams = np.asarray(lams, dtype=np.float64)
    B, Hq, N, d = q1.shape
    Hkv = k1.shape[1]
    if lams.shape != (Hq,):
        raise ValueError("one lambda per query head expected")
    g = Hq // Hkv
    nrows = N if rows is None else len(rows)
    out = np.empty((B, Hq, nrows, d), dtype=np.float64)
    for h in range(Hq):
        hk = h // g
        out[:, h] = diff(q1[:, h:h + 1], k1[:, hk:hk + 1], q2[:, h:h + 1], k2[:, hk:hk + 1],
                         v[:, hk:hk + 1], float(lams[h]), scale, rows=rows,
                         nthreads=nthreads, W=W)[:, 0]
    return out


def weights_row(q, k, W: int, scale: float, b: int, h: int, i: int, kind: str = "window",
                stride: int = 0) -> np.ndarray:
    """Softmax weights of query row i (length N; keys after i are 0)."""
    lib = _load()
    q64, k64 = _f64(q), _f64(k)
    B, Hq, N, d = q64.shape
    Hkv = k64.shape[1]
    w = np.empty(N, dtype=np.float64)
    rc = lib.oracle_weights_row(KINDS[kind], _ptr(q64), _ptr(k64), B, Hq, Hkv, N, d, int(W),
                                int(stride), float(scale), b, h, i, _ptr(w))
    if rc != 0:
        raise ValueError(f"oracle_weights_row rejected its arguments (code {rc})")
    return w


def pair_count(N: int, W: int, kind: str = "window", stride: int = 0) -> int:
    """Allowed (i, j) pairs of one head, counted from the mask rows."""
    n = _load().oracle_pair_count(KINDS[kind], N, W, stride)
    if n < 0:
        raise ValueError("bad pair_count arguments")
    return int(n)


def mask_row(N: int, W: int, i: int, kind: str = "window", stride: int = 0) -> np.ndarray:
    """Row i of the mask as a bool array (True = allowed)."""
    a = np.zeros(N, dtype=np.uint8)
    rc = _load().oracle_mask_row(KINDS[kind], N, W, stride, i, _ptr(a))
    if rc != 0:
        raise ValueError("bad mask_row arguments")
    return a.astype(bool)


def decode(q, kc, vc, pos, W: int, scale: float) -> np.ndarray:
    """Decode against a rolling W-slot cache in fp64.  q: [B, Hq, d]; kc, vc: [B, Hkv, W, d];
    pos: [B] absolute positions.  Returns [B, Hq, d]."""
    lib = _load()
    q64, k64, v64 = _f64(q), _f64(kc), _f64(vc)
    B, Hq, d = q64.shape
    Hkv = k64.shape[1]
    if k64.shape[2] != W:
        raise ValueError("cache slot count does not match W")
    p = np.ascontiguousarray(pos, dtype=np.int64)
    out = np.empty((B, Hq, d), dtype=np.float64)
    rc = lib.oracle_decode(_ptr(q64), _ptr(k64), _ptr(v64), _ptr(p), _ptr(out), B, Hq, Hkv,
                           int(W), d, float(scale))
    if rc != 0:
        raise ValueError(f"oracle_decode rejected its arguments (code {rc})")
    return out


def lse(q, k, W: int, scale: float, kind: str = "window", stride: int = 0, rows=None):
    """Log-sum-exp of every row's masked scores, fp64 [B, Hq, nrows]."""
    lib = _load()
    q64, k64 = _f64(q), _f64(k)
    B, Hq, N, d = q64.shape
    Hkv = k64.shape[1]
    r, nrows = _rows_arg(rows, N)
    out = np.empty((B, Hq, nrows), dtype=np.float64)
    rc = lib.oracle_lse(KINDS[kind], _ptr(q64), _ptr(k64), _ptr(out), B, Hq, Hkv, N, d, int(W),
                        int(stride), float(scale), None if r is None else _ptr(r), nrows)
    if rc != 0:
        raise ValueError(f"oracle_lse rejected its arguments (code {rc})")
    return out


def attn_bwd(q, k, v, dout, W: int, scale: float, kind: str = "window", stride: int = 0,
             nthreads: int = 0, rows=None):
    """Gradients (dq, dk, dv) in fp64 of the masked attention forward for an upstream
    gradient ``dout`` = dL/dout ([B, Hq, N, d]).  dk and dv sum over the query heads that
    share a KV head.

    ``rows`` (optional): only the terms of these query rows are taken; dq is zero on the
    other rows and dk, dv are sums over these rows only (complete for every key whose
    readers all lie in the subset)."""
    lib = _load()
    q64, k64, v64, g64 = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, N, d = q64.shape
    Hkv = k64.shape[1]
    dq = np.empty_like(q64)
    dk = np.empty_like(k64)
    dv = np.empty_like(v64)
    r, nrows = _rows_arg(rows, N)
    rc = lib.oracle_attn_bwd_rows(KINDS[kind], _ptr(q64), _ptr(k64), _ptr(v64), _ptr(g64),
                                  _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, int(W),
                                  int(stride), float(scale), None if r is None else _ptr(r),
                                  nrows, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attn_bwd rejected its arguments (code {rc})")
    return dq, dk, dv


def diff_bwd(q1, k1, q2, k2, v, lams, dout, W: int, scale: float, nthreads: int = 0):
    """Gradients of differential attention (A1 - lambda_h A2) V, both maps under the window W
    (0 or W >= N: causal), one lambda per query head (``lams`` [Hq]; a scalar lambda is the
    same value for every head).  Returns (dq1, dk1, dq2, dk2, dv, dlam) with dlam [Hq] the
    gradient of each head's lambda (summed over batches)."""
    lib = _load()
    a = [_f64(x) for x in (q1, k1, q2, k2, v)]
    g64 = _f64(dout)
    B, Hq, N, d = a[0].shape
    Hkv = a[1].shape[1]
    lam = np.ascontiguousarray(np.broadcast_to(np.asarray(lams, dtype=np.float64), (Hq,)))
    dq1, dq2 = np.empty_like(a[0]), np.empty_like(a[0])
    dk1, dk2, dv = np.empty_like(a[1]), np.empty_like(a[1]), np.empty_like(a[1])
    dlam = np.empty(Hq, dtype=np.float64)
    Wm = N if W == 0 else int(W)
    rc = lib.oracle_diff_bwd(*[_ptr(x) for x in a], _ptr(lam), _ptr(g64), _ptr(dq1), _ptr(dk1),
                             _ptr(dq2), _ptr(dk2), _ptr(dv), _ptr(dlam), B, Hq, Hkv, N, d, Wm,
                             float(scale), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_diff_bwd rejected its arguments (code {rc})")
    return dq1, dk1, dq2, dk2, dv, dlam


def cache_slot(j: int, W: int) -> int:
    """Cache slot that holds absolute position j (0-indexed) in a W-slot rolling cache."""
    r = int(_load().oracle_cache_slot(int(j), int(W)))
    if r < 0:
        raise ValueError("bad cache_slot arguments")
    return r


def max_threads() -> int:
    return int(_load().oracle_max_threads())

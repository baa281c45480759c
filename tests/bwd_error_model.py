"""Per-element tolerances for the backward pass of causal sliding-window attention, from a
first-order model of the roundings the GPU kernels make, plus a numpy emulation of those
roundings that the CPU tests use to check the model.

What is rounded.  The backward kernels take bf16 operands, multiply on the tensor cores and
accumulate in fp32.  Four quantities are rounded to bf16 on the way (u = 2^-8 is the unit
roundoff of bf16: 8 significant bits, round to nearest even):
  1. in the forward, the weights p_ij (the A operand of O += P V) and the output out_i, which
     the backward reads to form delta_i = dout_i . out_i;
  2. the weights a_ij in dV += P^T dO;
  3. ds_ij = a_ij (dp_ij - delta_i) in dK += dS^T Q and dQ += dS K;
  4. the gradients themselves.
Every other step (the products S and dP, the exponentials, the fp32 sums, the forward's
log-sum-exp) is exact to a few fp32 ulps, i.e. 2^16 times finer.

The model.  A rounding multiplies a value by (1 + e) with |e| <= u; the errors of different
terms are independent and have mean zero (the standard model of probabilistic rounding-error
analysis, Higham and Mary, "A new approach to probabilistic rounding error analysis", SIAM J.
Sci. Comput. 2019).  A sum of terms t_k each carrying such an error then errs by at most
LAM * u * sqrt(sum_k t_k^2), except with probability 2 exp(-LAM^2 / 2) (Hoeffding's
inequality).  LAM = 6 puts that at 3e-8 per element for errors as wide as the bound allows;
real RNE errors are narrower still.  Per element of a gradient g with exact value ref:

  |g_gpu - ref| <= u |ref| + (1 + u) (LAM u sigma + D + 2^-14 A)

  dv_j[c]:  sigma^2 = sum a_ij^2 dout_i[c]^2                    (rounding 2)
            A = sum a_ij |dout_i[c]|,  D = 0
  dk_j[c]:  sigma^2 = sum (scale ds_ij q_i[c])^2                  (rounding 3)
            D = scale sum_i a_ij e_i |q_i[c]|                      (rounding 1, through delta)
            A = scale sum_i a_ij (|dp_ij| + |delta_i|) |q_i[c]|
  dq_i[c]:  sigma^2 = sum (scale ds_ij k_j[c])^2
            D = scale e_i sum_j a_ij |k_j[c]|
            A = scale sum_j a_ij (|dp_ij| + |delta_i|) |k_j[c]|
  e_i = LAM u (sqrt(sum_c dout_i[c]^2 out_i[c]^2) + sqrt(sum_j a_ij^2 dp_ij^2))
        + 2^-14 sum_c |dout_i[c]| |out_i[c]|
where the sums run over the allowed pairs (and, for dk and dv, over the query heads that
share the KV head).  e_i bounds the error of delta_i: the forward rounds out_i to bf16 (first
square root: delta = sum_c dout_c out_c with each out_c off by at most u |out_c|) and rounds
the weights it sums V with (second square root: sum_c dout_c (sum_j a_ij e_j v_j[c]) =
sum_j a_ij e_j dp_ij).  The u |ref| term is rounding 4; 2^-14 A covers every fp32-level error,
including cancellation in dp_ij - delta_i, with a wide margin.

All of the model's quantities are the exact (fp64) softmax weights and gradients of the
problem, computed here block by block over the band; the GPU tests compare with the oracle's
gradients, and this module only supplies the bound.
"""
from __future__ import annotations

import numpy as np

U_BF16 = 2.0 ** -8
LAM = 6.0
FP32_SLACK = 2.0 ** -14


def _widen(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:
        x = (x.astype(np.uint32) << 16).view(np.float32)
    return np.ascontiguousarray(x, dtype=np.float64)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round to bf16 (through fp32, ties to even) and widen back to fp64."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


def _row_chunks(rows: np.ndarray, block: int):
    """Split sorted rows into chunks of at most `block` rows spanning at most `block` positions."""
    start = 0
    n = rows.size
    while start < n:
        end = start + 1
        while end < n and end - start < block and rows[end] - rows[start] < block:
            end += 1
        yield rows[start:end]
        start = end


def _allowed(rows, keys, W, kind, stride, widen=0):
    """The mask on (rows x keys): the causal window of W positions (W + widen, for the planted
    mistake), plus, for "strided", the multiples of `stride` and, for "global", the keys below
    `stride` (the number of global tokens), each only where j <= i."""
    i, j = rows[:, None], keys[None, :]
    m = (j >= i - W + 1 - widen) & (j <= i)
    if kind == "strided":
        m |= (j % stride == 0) & (j <= i)
    elif kind == "global":
        m |= (j < stride) & (j <= i)
    return m


def _band(qi, rows, kk, W, scale, kind="window", stride=0, widen=0):
    """Scores of `rows` over the keys any of them may read (a sorted index array `keys`),
    masked to -inf outside the mask."""
    lo = max(0, int(rows[0]) - W + 1 - widen)
    hi = int(rows[-1])
    keys = np.arange(lo, hi + 1)
    if kind == "strided":
        keys = np.union1d(np.arange(0, lo, stride), keys)
    elif kind == "global":
        keys = np.union1d(np.arange(0, min(lo, stride)), keys)
    allowed = _allowed(rows, keys, W, kind, stride, widen)
    s = scale * (qi @ kk[keys].T)
    s = np.where(allowed, s, -np.inf)
    return keys, allowed, s


def bwd_bounds(q, k, v, dout, W: int, scale: float, rows=None, block: int = 256,
               kind: str = "window", stride: int = 0):
    """Exact gradients and their per-element bounds for causal SWA with window W (kind
    "window"), or its local + strided ("strided", stride = the stride) or global-prefix
    ("global", stride = the number of global tokens) extensions.

    q, dout: [B, Hq, N, d]; k, v: [B, Hkv, N, d] (fp64 or bf16 bit patterns).
    rows: the query rows whose terms are taken (default all); dq is zero on the other rows and
    dk, dv hold the sums over these rows (as the oracle's row-subset form).
    Returns {"dq": (ref, bound), "dk": (ref, bound), "dv": (ref, bound),
    "delta": (delta_i, e_i)}, the last the rows' delta = dout_i . out_i and the bound e_i on
    the error of the delta the kernels form ([B, Hq, N]; zero on rows not taken)."""
    q, k, v, g = _widen(q), _widen(k), _widen(v), _widen(dout)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    grp = Hq // Hkv
    W = min(int(W), N)
    rows = np.arange(N) if rows is None else np.unique(np.asarray(rows, dtype=np.int64))
    u = U_BF16
    dq, dq_s2, dq_D, dq_A = (np.zeros_like(q) for _ in range(4))
    dk, dk_s2, dk_D, dk_A = (np.zeros_like(k) for _ in range(4))
    dv, dv_s2, dv_A = (np.zeros_like(v) for _ in range(3))
    dl_ref, dl_e = np.zeros(q.shape[:3]), np.zeros(q.shape[:3])
    for b in range(B):
        for h in range(Hq):
            hk = h // grp
            kk, vv = k[b, hk], v[b, hk]
            for rr in _row_chunks(rows, block):
                keys, allowed, s = _band(q[b, h, rr], rr, kk, W, scale, kind, stride)
                a = np.exp(s - s.max(axis=1, keepdims=True))
                a /= a.sum(axis=1, keepdims=True)
                kb, vb, gr, qr = kk[keys], vv[keys], g[b, h, rr], q[b, h, rr]
                out = a @ vb
                dp = np.where(allowed, gr @ vb.T, 0.0)
                delta = np.sum(a * dp, axis=1)
                ds = a * (dp - delta[:, None])
                mag = a * (np.abs(dp) + np.abs(delta)[:, None])
                e = (LAM * u * (np.sqrt(np.sum(gr * gr * out * out, axis=1)) +
                                np.sqrt(np.sum(a * a * dp * dp, axis=1))) +
                     FP32_SLACK * np.sum(np.abs(gr) * np.abs(out), axis=1))
                dl_ref[b, h, rr] = delta
                dl_e[b, h, rr] = e
                dq[b, h, rr] = scale * (ds @ kb)
                dq_s2[b, h, rr] = scale ** 2 * ((ds * ds) @ (kb * kb))
                dq_D[b, h, rr] = scale * e[:, None] * (a @ np.abs(kb))
                dq_A[b, h, rr] = scale * (mag @ np.abs(kb))
                sl = keys
                dk[b, hk, sl] += scale * (ds.T @ qr)
                dk_s2[b, hk, sl] += scale ** 2 * ((ds * ds).T @ (qr * qr))
                dk_D[b, hk, sl] += scale * ((a * e[:, None]).T @ np.abs(qr))
                dk_A[b, hk, sl] += scale * (mag.T @ np.abs(qr))
                dv[b, hk, sl] += a.T @ gr
                dv_s2[b, hk, sl] += (a * a).T @ (gr * gr)
                dv_A[b, hk, sl] += a.T @ np.abs(gr)

    def bound(ref, s2, D, A):
        return u * np.abs(ref) + (1.0 + u) * (LAM * u * np.sqrt(s2) + D + FP32_SLACK * A)

    return {"dq": (dq, bound(dq, dq_s2, dq_D, dq_A)),
            "dk": (dk, bound(dk, dk_s2, dk_D, dk_A)),
            "dv": (dv, bound(dv, dv_s2, 0.0, dv_A)),
            "delta": (dl_ref, dl_e)}


def emulate_kernel_bwd(q, k, v, dout, W: int, scale: float, plant: str = "",
                       kind: str = "window", stride: int = 0):
    """The backward as the kernels round it (roundings 1-4 above, everything else in fp64):
    the forward's bf16 weights and bf16 output, bf16 a_ij in dV, bf16 ds_ij in dK and dQ,
    bf16 gradients.  `plant` injects a mistake for the tests of the bound's power:
    "window" (one key too many before each window), "delta" (delta dropped), "scale" (dq
    without the scale), "head" (dv from the neighbouring query head's dout)."""
    q, k, v, g = _widen(q), _widen(k), _widen(v), _widen(dout)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    grp = Hq // Hkv
    W = min(int(W), N)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            hk = h // grp
            kk, vv = k[b, hk], v[b, hk]
            for rr in _row_chunks(np.arange(N), 256):
                widen = 1 if plant == "window" else 0
                keys, allowed, s = _band(q[b, h, rr], rr, kk, W, scale, kind, stride, widen)
                kb, vb, gr, qr = kk[keys], vv[keys], g[b, h, rr], q[b, h, rr]
                # the forward sees the true mask: scores outside it are -inf
                s_true = np.where(_allowed(rr, keys, W, kind, stride), s, -np.inf)
                # forward: bf16 weights against the row maximum, fp32-exact normaliser
                m = s_true.max(axis=1, keepdims=True)
                p = np.exp(s_true - m)
                l = p.sum(axis=1, keepdims=True)
                out16 = bf16_round((bf16_round(p) @ vb) / l)
                lse = m + np.log(l)
                a = np.exp(s - lse)
                dp = np.where(np.isfinite(s), gr @ vb.T, 0.0)
                delta = 0.0 if plant == "delta" else np.sum(out16 * gr, axis=1)[:, None]
                ds16 = bf16_round(a * (dp - delta))
                sq = 1.0 if plant == "scale" else scale
                dq[b, h, rr] = sq * (ds16 @ kb)
                sl = keys
                dk[b, hk, sl] += scale * (ds16.T @ qr)
                gv = g[b, (h + 1) % Hq, rr] if plant == "head" else gr
                dv[b, hk, sl] += bf16_round(a).T @ gv
    return bf16_round(dq), bf16_round(dk), bf16_round(dv)


def worst_ratio(got, ref, bound) -> float:
    """max |got - ref| / bound over the elements (0 for empty arrays)."""
    if np.size(got) == 0:
        return 0.0
    return float(np.max(np.abs(np.asarray(got) - ref) / bound))

"""GPU parity of the backward pass (dq, dk, dv of causal SWA) against the fp64 oracle's
gradients, on seeded bf16 inputs.  The forward output and row log-sum-exp the backward needs
come from the GPU forward (swa_attn_fwd_lse), as in training.

Tolerance, per element: |gpu - oracle| <= the bound of tests/bwd_error_model.py, a
first-order model of the four bf16 roundings the kernels make (the forward's weights and
output, a_ij in dV, ds_ij in dK and dQ, the gradients) with a 6-sigma-style Hoeffding factor.
The bound of each element is scaled by that element's own terms, so a fault confined to a few
rows or keys (a window edge, a wrong delta on the first rows) is measured against those rows'
magnitudes, not the tensor's.  The CPU tests of that module show that an emulation of the
kernels' roundings stays within 0.41 of the bound and that planted mistakes exceed it.

At the full Mistral shape the oracle checks sub-problems that hold every term of the sampled
elements (causal windows make a prefix, or a slice of W - 1 positions before the rows, a
complete problem of its own)."""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import oracle
import swa_inputs
from swa_inputs import f32_to_bf16_bits
import sparse_causal_attention_swa_b300 as pkg
from bwd_error_model import bwd_bounds
from gpu_util import canary_intact, check_bound as _check, check_bound_one as _check_one, out_like, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _rand(rng, shape):
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def _bwd_gpu(q, k, v, g, W, scale):
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    tq, tk, tv, tg = to_dev(q), to_dev(k), to_dev(v), to_dev(g)
    out = torch.empty_like(tq)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    pkg.swa_attn_fwd_lse(tq, tk, tv, out, lse, B, Hq, Hkv, N, d, W, scale)
    nb = pkg.swa_attn_bwd_workspace_bytes(B, Hq, N)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    dq, bq = out_like(tq)
    dk, bk = out_like(tk)
    dv, bv = out_like(tv)
    pkg.swa_attn_bwd(tq, tk, tv, out, lse, tg, dq, dk, dv, B, Hq, Hkv, N, d, W, scale, ws, nb)
    torch.cuda.synchronize()
    assert pkg.swa_device_status() == 0
    for t, b in ((dq, bq), (dk, bk), (dv, bv)):
        assert canary_intact(b, t.numel()), "write past the end of a gradient"
    return to_f64(dq), to_f64(dk), to_f64(dv)


def _case(B, Hq, Hkv, N, d, W, seed, scale=None):
    rng = np.random.default_rng(seed)
    q = _rand(rng, (B, Hq, N, d))
    k = _rand(rng, (B, Hkv, N, d))
    v = _rand(rng, (B, Hkv, N, d))
    g = _rand(rng, (B, Hq, N, d))
    sc = 1.0 / np.sqrt(d) if scale is None else scale
    got = _bwd_gpu(q, k, v, g, W, sc)
    ref = oracle.attn_bwd(q, k, v, g, W, sc)
    model = bwd_bounds(q, k, v, g, W, sc)
    _check(got, ref, [model[n][1] for n in ("dq", "dk", "dv")],
           f"B={B} heads=({Hq},{Hkv}) N={N} d={d} W={W}")
    return got, ref


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("heads", [(1, 1), (4, 2), (3, 1)])
def test_bwd_sweep(d, heads):
    Hq, Hkv = heads
    for N, W in ((1, 1), (60, 7), (128, 128), (200, 63), (300, 129), (513, 200), (257, 1000)):
        _case(1, Hq, Hkv, N, d, W, seed=N + W + d)


def test_bwd_batch_and_scale():
    _case(2, 4, 1, 700, 64, 300, seed=5, scale=0.09)
    _case(3, 2, 2, 390, 128, 130, seed=6)


def test_bwd_w1_gives_dv_sum_and_no_q_k_gradient():
    got, _ = _case(2, 6, 2, 300, 128, 1, seed=8)
    dq, dk, _ = got
    assert np.max(np.abs(dq)) < 1e-3 and np.max(np.abs(dk)) < 1e-3


def test_bwd_deterministic():
    rng = np.random.default_rng(9)
    B, Hq, Hkv, N, d, W = 1, 4, 2, 1000, 128, 300
    a = [_rand(rng, (B, h, N, d)) for h in (Hq, Hkv, Hkv, Hq)]
    r1 = _bwd_gpu(*a, W, 0.1)
    r2 = _bwd_gpu(*a, W, 0.1)
    for x, y in zip(r1, r2):
        assert np.array_equal(x, y)


def _sub_problem(inp, hk, g, p0, p1):
    """Positions [p0, p1) of KV head hk and its g query heads, as a sequence of its own."""
    qs = slice(hk * g, (hk + 1) * g)
    return (np.ascontiguousarray(inp["q"][:1, qs, p0:p1]),
            np.ascontiguousarray(inp["k"][:1, hk:hk + 1, p0:p1]),
            np.ascontiguousarray(inp["v"][:1, hk:hk + 1, p0:p1]),
            np.ascontiguousarray(inp["dout"][:1, qs, p0:p1]))


def test_bwd_mistral_full_size_sampled():
    """The Mistral-shaped backward (B=1, Hq=32, Hkv=8, N=16384, d=128, W=4096), computed whole
    by the same C-ABI call the benchmark times, checked element by element on:
      - KV head 0: every dq row of positions 0..4607 and the dk, dv of keys 0..512 (every row
        that reads those keys lies in the prefix);
      - KV head 5: the dq rows of positions 8064..8319 (both sides of two tile boundaries);
      - KV head 7: the dq rows and the dk, dv keys of the last 256 positions;
      - every KV head: 16 seeded random dq rows."""
    w = swa_inputs.WORKLOADS["mistral_swa_bwd"]
    inp = swa_inputs.make_inputs(w)
    N, W, sc, g = w.N, w.W, w.scale, w.Hq // w.Hkv
    got = _bwd_gpu(inp["q"], inp["k"], inp["v"], inp["dout"], W, sc)

    jobs = []  # (label, sub-problem, oracle row subset, [(tensor, head slice, sub rows, full rows)])
    pre = 4608
    sub = _sub_problem(inp, 0, g, 0, pre)
    jobs.append(("prefix kv0", sub, np.arange(pre), [
        ("dq", slice(0, g), np.arange(pre), np.arange(pre)),
        ("dk", slice(0, 1), np.arange(pre - W + 1), np.arange(pre - W + 1)),
        ("dv", slice(0, 1), np.arange(pre - W + 1), np.arange(pre - W + 1))]))
    p0 = 8064 - (W - 1)
    sub = _sub_problem(inp, 5, g, p0, 8320)
    rows = np.arange(8064, 8320) - p0
    jobs.append(("rows 8064..8319 kv5", sub, rows, [
        ("dq", slice(5 * g, 6 * g), rows, rows + p0)]))
    p0 = N - 256 - (W - 1)
    sub = _sub_problem(inp, 7, g, p0, N)
    rows = np.arange(N - 256, N) - p0
    jobs.append(("last 256 kv7", sub, rows, [
        ("dq", slice(7 * g, 8 * g), rows, rows + p0),
        ("dk", slice(7, 8), rows, rows + p0),
        ("dv", slice(7, 8), rows, rows + p0)]))
    rng = np.random.default_rng(w.seed + 100)
    for hk in range(w.Hkv):
        pos = np.unique(rng.integers(0, N, size=16))
        p0 = max(0, int(pos[0]) - (W - 1))
        sub = _sub_problem(inp, hk, g, p0, int(pos[-1]) + 1)
        jobs.append((f"random rows kv{hk}", sub, pos - p0, [
            ("dq", slice(hk * g, (hk + 1) * g), pos - p0, pos)]))

    # the oracle's fp64 gradients of every sub-problem, up to eight host threads at once (the
    # prefix split into row ranges of about equal work; dk and dv of a split are partial sums)
    def oracle_job(sub, rows):
        return oracle.attn_bwd(*sub, W, sc, rows=rows, nthreads=1)

    with cf.ThreadPoolExecutor(max_workers=8) as ex:
        futs = []
        for label, sub, rows, _ in jobs:
            parts = np.split(rows, [2290, 3238, 3967]) if label.startswith("prefix") else [rows]
            futs.append([ex.submit(oracle_job, sub, part) for part in parts])
        refs = []
        for fl in futs:
            res = [f.result() for f in fl]
            refs.append(tuple(sum(r[t] for r in res) for t in range(3)))

    names = {"dq": 0, "dk": 1, "dv": 2}
    worst = {}
    for (label, sub, rows, checks), ref in zip(jobs, refs):
        model = bwd_bounds(*sub, W, sc, rows=rows)
        for name, heads, sub_rows, full_rows in checks:
            t = names[name]
            a = got[t][0, heads][:, full_rows]
            r = ref[t][0][:, sub_rows]
            bnd = model[name][1][0][:, sub_rows]
            worst[name] = max(worst.get(name, 0.0), _check_one(a, r, bnd, f"{label} {name}"))
    print(f"mistral_swa_bwd sampled: worst |gpu - oracle| / bound = {worst}")

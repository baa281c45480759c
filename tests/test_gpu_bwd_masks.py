"""GPU parity of the backward pass of the local + strided and window + global-prefix masks
(strided_attn_bwd, global_attn_bwd) against the fp64 oracle's gradients (oracle.attn_bwd with
kind "strided" / "global"), element by element, under the per-element bound of
tests/bwd_error_model.py for the same mask.  The forward output and row log-sum-exp come from
the GPU forward (strided_attn_fwd_lse, global_attn_fwd_lse), as in training.  The full strided
and global workloads are checked on every element."""
import numpy as np
import pytest
import torch

import oracle
import swa_inputs
from swa_inputs import f32_to_bf16_bits
import sparse_causal_attention_swa_b300 as pkg
from bwd_error_model import bwd_bounds
from gpu_util import canary_intact, check_bound as _check, out_like, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _rand(rng, shape):
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def _bwd_gpu(kind, q, k, v, g, W, x, scale):
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    tq, tk, tv, tg = to_dev(q), to_dev(k), to_dev(v), to_dev(g)
    out = torch.empty_like(tq)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    fwd = pkg.strided_attn_fwd_lse if kind == "strided" else pkg.global_attn_fwd_lse
    fwd(tq, tk, tv, out, lse, B, Hq, Hkv, N, d, W, x, scale)
    wsf = (pkg.strided_attn_bwd_workspace_bytes if kind == "strided"
           else pkg.global_attn_bwd_workspace_bytes)
    nb = wsf(B, Hq, Hkv, N, d, W, x)
    ws = torch.full((nb,), 0xFF, dtype=torch.uint8, device="cuda")  # no zero-init assumed
    dq, bq = out_like(tq)
    dk, bk = out_like(tk)
    dv, bv = out_like(tv)
    bwd = pkg.strided_attn_bwd if kind == "strided" else pkg.global_attn_bwd
    bwd(tq, tk, tv, out, lse, tg, dq, dk, dv, B, Hq, Hkv, N, d, W, x, scale, ws, nb)
    torch.cuda.synchronize()
    assert pkg.swa_device_status() == 0
    for t, b in ((dq, bq), (dk, bk), (dv, bv)):
        assert canary_intact(b, t.numel()), "write past the end of a gradient"
    return to_f64(dq), to_f64(dk), to_f64(dv)


def _case(kind, B, Hq, Hkv, N, d, W, x, seed, scale=None):
    rng = np.random.default_rng(seed)
    q = _rand(rng, (B, Hq, N, d))
    k = _rand(rng, (B, Hkv, N, d))
    v = _rand(rng, (B, Hkv, N, d))
    g = _rand(rng, (B, Hq, N, d))
    sc = 1.0 / np.sqrt(d) if scale is None else scale
    got = _bwd_gpu(kind, q, k, v, g, W, x, sc)
    ref = oracle.attn_bwd(q, k, v, g, W, sc, kind=kind, stride=x)
    model = bwd_bounds(q, k, v, g, W, sc, kind=kind, stride=x)
    return _check(got, ref, [model[n][1] for n in ("dq", "dk", "dv")],
                  f"{kind} B={B} heads=({Hq},{Hkv}) N={N} d={d} W={W} x={x}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("heads", [(1, 1), (4, 2), (3, 1)])
def test_strided_bwd_sweep(d, heads):
    Hq, Hkv = heads
    for N, W, s in ((1, 1, 1), (300, 64, 7), (513, 100, 128), (700, 256, 33), (400, 1, 5),
                    (300, 300, 3), (260, 20, 1), (200, 30, 500)):
        _case("strided", 1, Hq, Hkv, N, d, W, s, seed=N + W + s + d)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("heads", [(1, 1), (4, 2)])
def test_global_bwd_sweep(d, heads):
    Hq, Hkv = heads
    for N, W, ng in ((300, 64, 1), (513, 100, 64), (700, 128, 300), (300, 50, 0), (400, 40, 400),
                     (129, 1, 129)):
        _case("global", 1, Hq, Hkv, N, d, W, ng, seed=N + W + ng + d)


def test_strided_bwd_batch_and_scale():
    _case("strided", 2, 4, 1, 900, 64, 200, 64, seed=11, scale=0.09)
    _case("global", 3, 2, 2, 500, 128, 100, 16, seed=12)


def test_strided_bwd_deterministic():
    rng = np.random.default_rng(13)
    B, Hq, Hkv, N, d, W, s = 1, 4, 2, 1000, 64, 128, 32
    a = [_rand(rng, (B, h, N, d)) for h in (Hq, Hkv, Hkv, Hq)]
    r1 = _bwd_gpu("strided", *a, W, s, 0.1)
    r2 = _bwd_gpu("strided", *a, W, s, 0.1)
    for x, y in zip(r1, r2):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("name", ["strided", "global"])
def test_full_size_workload_every_element(name):
    """The strided (B=1, H=16, N=16384, d=64, W=256, s=128) and global-prefix (W=512, 64 global
    tokens) workloads, with an upstream gradient drawn after the inputs by the same recipe."""
    w = swa_inputs.WORKLOADS[name]
    inp = swa_inputs.make_inputs(w)
    rng = np.random.default_rng(w.seed + 200)
    g = _rand(rng, inp["q"].shape)
    got = _bwd_gpu(w.kind, inp["q"], inp["k"], inp["v"], g, w.W, w.stride, w.scale)
    ref = oracle.attn_bwd(inp["q"], inp["k"], inp["v"], g, w.W, w.scale, kind=w.kind,
                          stride=w.stride)
    model = bwd_bounds(inp["q"], inp["k"], inp["v"], g, w.W, w.scale, kind=w.kind,
                       stride=w.stride)
    ratios = _check(got, ref, [model[n][1] for n in ("dq", "dk", "dv")], name)
    print(f"{name} backward, every element: worst |gpu - oracle| / bound = {ratios}")

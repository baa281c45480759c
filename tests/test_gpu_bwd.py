"""GPU parity of the backward pass (dq, dk, dv of causal SWA) against the fp64 oracle's
gradients, on seeded bf16 inputs.  The forward output and row log-sum-exp the backward needs
come from the GPU forward (swa_attn_fwd_lse), as in training.

Tolerance, per gradient tensor: |gpu - oracle| <= 0.1 rms(oracle) + 2e-2 |oracle| + 1e-4.
The kernels round P and dS to bf16 for the tensor-core products (as the forward rounds P) and
the gradients to bf16; a numpy emulation of exactly those roundings against the oracle gives
errors up to 5.6 % of the tensor's rms on these shapes, so the bound keeps a 2x margin while a
wrong mask, scale or head mapping gives errors of the order of the rms itself."""
import numpy as np
import pytest
import torch

import oracle
from swa_inputs import f32_to_bf16_bits
import sparse_causal_attention_swa_b300 as pkg
from gpu_util import canary_intact, out_like, to_dev, to_f64

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


def _check(got, ref, label):
    for name, a, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.all(np.isfinite(a)), f"{label} {name}: non-finite"
        rms = float(np.sqrt(np.mean(r * r)))
        err = np.abs(a - r)
        bad = err > 0.1 * rms + 2e-2 * np.abs(r) + 1e-4
        assert not bad.any(), (f"{label} {name}: {int(bad.sum())} out of tolerance, max err "
                               f"{err.max():.3e}, rms {rms:.3e}")


def _case(B, Hq, Hkv, N, d, W, seed, scale=None):
    rng = np.random.default_rng(seed)
    q = _rand(rng, (B, Hq, N, d))
    k = _rand(rng, (B, Hkv, N, d))
    v = _rand(rng, (B, Hkv, N, d))
    g = _rand(rng, (B, Hq, N, d))
    sc = 1.0 / np.sqrt(d) if scale is None else scale
    got = _bwd_gpu(q, k, v, g, W, sc)
    ref = oracle.attn_bwd(q, k, v, g, W, sc)
    _check(got, ref, f"B={B} heads=({Hq},{Hkv}) N={N} d={d} W={W}")
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

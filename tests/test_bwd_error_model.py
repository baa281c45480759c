"""CPU checks of the backward tolerance model (tests/bwd_error_model.py).

1. The model's exact quantities are the oracle's: its fp64 gradients equal oracle.attn_bwd,
   in full and on row subsets.
2. The model accepts what the kernels compute: a numpy emulation of the kernels' bf16
   roundings stays inside the per-element bound on every element.
3. The bound has power: a planted mistake in that emulation (a window one key too wide, a
   dropped delta, a missing scale, the wrong query head) breaks it.
The same for the local + strided and global-prefix masks.
"""
import numpy as np
import pytest

import oracle
from bwd_error_model import bwd_bounds, emulate_kernel_bwd, worst_ratio
from swa_inputs import f32_to_bf16_bits


def _inputs(seed, B, Hq, Hkv, N, d):
    rng = np.random.default_rng(seed)
    mk = lambda h: f32_to_bf16_bits(rng.standard_normal((B, h, N, d), dtype=np.float32))
    return mk(Hq), mk(Hkv), mk(Hkv), mk(Hq)


@pytest.mark.parametrize("B,Hq,Hkv,N,d,W", [(1, 2, 1, 70, 16, 9), (2, 3, 3, 41, 8, 41),
                                            (1, 4, 2, 300, 32, 1), (1, 2, 2, 600, 16, 257)])
def test_model_gradients_are_the_oracles(oracle_mod, B, Hq, Hkv, N, d, W):
    q, k, v, g = _inputs(N + W, B, Hq, Hkv, N, d)
    sc = 1.0 / np.sqrt(d)
    ref = oracle_mod.attn_bwd(q, k, v, g, W, sc)
    got = bwd_bounds(q, k, v, g, W, sc)
    for name, r in zip(("dq", "dk", "dv"), ref):
        m, bnd = got[name]
        np.testing.assert_allclose(m, r, rtol=0, atol=1e-12 * max(1.0, np.abs(r).max()))
        assert np.all(bnd > 0)
    rows = np.r_[0:37, 100:130, 290:300]
    rows = rows[rows < N]
    ref_r = oracle_mod.attn_bwd(q, k, v, g, W, sc, rows=rows)
    got_r = bwd_bounds(q, k, v, g, W, sc, rows=rows)
    for name, r in zip(("dq", "dk", "dv"), ref_r):
        np.testing.assert_allclose(got_r[name][0], r, rtol=0,
                                   atol=1e-12 * max(1.0, np.abs(r).max()))


CASES = [  # (B, Hq, Hkv, N, d, W, scale or None)
    (1, 1, 1, 513, 64, 200, None),
    (1, 4, 2, 300, 128, 129, None),
    (2, 3, 1, 257, 64, 1000, None),
    (1, 2, 2, 200, 64, 63, None),
    (1, 6, 2, 300, 128, 1, None),
    (2, 4, 1, 700, 64, 300, 0.09),
    (1, 4, 1, 1500, 128, 1024, None),
]


@pytest.mark.parametrize("case", CASES)
def test_rounding_emulation_within_bound(oracle_mod, case):
    B, Hq, Hkv, N, d, W, sc = case
    sc = 1.0 / np.sqrt(d) if sc is None else sc
    q, k, v, g = _inputs(7 * N + W, B, Hq, Hkv, N, d)
    ref = oracle_mod.attn_bwd(q, k, v, g, W, sc)
    model = bwd_bounds(q, k, v, g, W, sc)
    emu = emulate_kernel_bwd(q, k, v, g, W, sc)
    for name, r, e in zip(("dq", "dk", "dv"), ref, emu):
        ratio = worst_ratio(e, r, model[name][1])
        print(f"{case} {name}: worst |emulation - oracle| / bound = {ratio:.3f}")
        assert ratio <= 1.0, f"{case} {name}: {ratio:.3f}"


@pytest.mark.parametrize("plant", ["window", "delta", "scale", "head"])
def test_planted_mistakes_break_the_bound(oracle_mod, plant):
    B, Hq, Hkv, N, d, W = 1, 4, 2, 400, 64, 63
    sc = 1.0 / np.sqrt(d)
    q, k, v, g = _inputs(11, B, Hq, Hkv, N, d)
    ref = oracle_mod.attn_bwd(q, k, v, g, W, sc)
    model = bwd_bounds(q, k, v, g, W, sc)
    emu = emulate_kernel_bwd(q, k, v, g, W, sc, plant=plant)
    worst = max(worst_ratio(e, r, model[n][1]) for n, r, e in zip(("dq", "dk", "dv"), ref, emu))
    print(f"planted {plant}: worst ratio {worst:.2f}")
    assert worst > 1.0


@pytest.mark.parametrize("kind,B,Hq,Hkv,N,d,W,x", [("strided", 1, 2, 1, 300, 16, 40, 7),
                                                  ("strided", 2, 3, 3, 200, 32, 1, 64),
                                                  ("strided", 1, 4, 2, 129, 16, 129, 5),
                                                  ("global", 1, 2, 2, 300, 16, 33, 10),
                                                  ("global", 1, 4, 1, 250, 32, 1, 250)])
def test_masks_gradients_are_the_oracles_and_emulation_within_bound(oracle_mod, kind, B, Hq, Hkv,
                                                                     N, d, W, x):
    q, k, v, g = _inputs(3 * N + W + x, B, Hq, Hkv, N, d)
    sc = 1.0 / np.sqrt(d)
    ref = oracle_mod.attn_bwd(q, k, v, g, W, sc, kind=kind, stride=x)
    model = bwd_bounds(q, k, v, g, W, sc, kind=kind, stride=x)
    emu = emulate_kernel_bwd(q, k, v, g, W, sc, kind=kind, stride=x)
    for name, r, e in zip(("dq", "dk", "dv"), ref, emu):
        m, bnd = model[name]
        np.testing.assert_allclose(m, r, rtol=0, atol=1e-12 * max(1.0, np.abs(r).max()))
        ratio = worst_ratio(e, r, bnd)
        print(f"{kind} N={N} W={W} x={x} {name}: worst |emulation - oracle| / bound = {ratio:.3f}")
        assert ratio <= 1.0
    planted = emulate_kernel_bwd(q, k, v, g, W, sc, plant="delta", kind=kind, stride=x)
    assert max(worst_ratio(e, r, model[n][1])
               for n, r, e in zip(("dq", "dk", "dv"), ref, planted)) > 1.0

"""GPU parity of the differential-attention backward (diff_attn_bwd) against the fp64 oracle's
gradients (oracle.diff_bwd), element by element.  The forward quantities the backward needs,
out1 / lse1 and out2 / lse2, come from swa_attn_fwd_lse on (q1, k1, v) and (q2, k2, v), as in
training.

Tolerance per element: map 1 is the SWA backward of (q1, k1, v, dout) and map 2 that of
(q2, k2, v, -lambda_h dout), so dq1 / dk1 and dq2 / dk2 take the bounds of
tests/bwd_error_model.py for those problems (with the exact -lambda_h dout in the model); dv,
the sum of both maps' dv rounded once, takes the sum of the two bounds; dlambda_h =
-sum_i dout_i . out2_i takes the sum of the rows' delta bounds e_i plus an fp32 reduction
slack of 2^-16 sum |delta_i|."""
import numpy as np
import pytest
import torch

import oracle
import swa_inputs
from swa_inputs import f32_to_bf16_bits
import sparse_causal_attention_swa_b300 as pkg
from bwd_error_model import bwd_bounds
from gpu_util import canary_intact, check_bound_one, out_like, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _rand(rng, shape):
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def _diff_bwd_gpu(q1, k1, q2, k2, v, g, lams, per_head, W, scale):
    B, Hq, N, d = q1.shape
    Hkv = k1.shape[1]
    t = [to_dev(a) for a in (q1, k1, q2, k2, v, g)]
    tq1, tk1, tq2, tk2, tv, tg = t
    outs, lses = [], []
    for tq, tk in ((tq1, tk1), (tq2, tk2)):
        o = torch.empty_like(tq)
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
        pkg.swa_attn_fwd_lse(tq, tk, tv, o, lse, B, Hq, Hkv, N, d, W, scale)
        outs.append(o)
        lses.append(lse)
    lam_t = torch.as_tensor(np.asarray(lams, dtype=np.float32), device="cuda") if per_head else None
    lam = 0.0 if per_head else float(lams)
    nb = pkg.diff_attn_bwd_workspace_bytes(B, Hq, Hkv, N, d)
    ws = torch.full((nb,), 0xFF, dtype=torch.uint8, device="cuda")
    grads = [out_like(x) for x in (tq1, tk1, tq2, tk2, tv)]
    dlam = torch.full((Hq,), float("nan"), dtype=torch.float32, device="cuda")
    pkg.diff_attn_bwd(tq1, tk1, tq2, tk2, tv, lam, lam_t, outs[0], lses[0], outs[1], lses[1], tg,
                      *[gr for gr, _ in grads], dlam, B, Hq, Hkv, N, d, W, scale, ws, nb)
    torch.cuda.synchronize()
    assert pkg.swa_device_status() == 0
    for gr, buf in grads:
        assert canary_intact(buf, gr.numel()), "write past the end of a gradient"
    return [to_f64(gr) for gr, _ in grads] + [dlam.cpu().numpy().astype(np.float64)]


def _bounds(q1, k1, q2, k2, v, g, lam_h, W, sc, rows=None):
    """Per-element bounds of (dq1, dk1, dq2, dk2, dv) and the rows' delta-error bounds of map 2."""
    g64 = swa_inputs.bf16_bits_to_f64(g)
    mu = -np.asarray(lam_h, dtype=np.float64)[None, :, None, None]
    m1 = bwd_bounds(q1, k1, v, g, W, sc, rows=rows)
    m2 = bwd_bounds(q2, k2, v, mu * g64, W, sc, rows=rows)
    m2u = bwd_bounds(q2, k2, v, g, W, sc, rows=rows)
    return ([m1["dq"][1], m1["dk"][1], m2["dq"][1], m2["dk"][1], m1["dv"][1] + m2["dv"][1]],
            m2u["delta"])


def _case(B, Hq, Hkv, N, d, W, lams, per_head, seed, scale=None):
    rng = np.random.default_rng(seed)
    q1, k1, q2, k2, v = (_rand(rng, (B, h, N, d)) for h in (Hq, Hkv, Hq, Hkv, Hkv))
    g = _rand(rng, (B, Hq, N, d))
    sc = 1.0 / np.sqrt(d) if scale is None else scale
    lam_h = np.broadcast_to(np.asarray(lams, dtype=np.float32).astype(np.float64), (Hq,))
    got = _diff_bwd_gpu(q1, k1, q2, k2, v, g, lams, per_head, W, sc)
    ref = oracle.diff_bwd(q1, k1, q2, k2, v, lam_h, g, W, sc)
    bnds, (delta2, e2) = _bounds(q1, k1, q2, k2, v, g, lam_h, W, sc)
    label = f"B={B} heads=({Hq},{Hkv}) N={N} d={d} W={W} lam={lams}"
    worst = {}
    for name, a, r, bnd in zip(("dq1", "dk1", "dq2", "dk2", "dv"), got[:5], ref[:5], bnds):
        worst[name] = check_bound_one(a, r, bnd, f"{label} {name}")
    dl_bound = e2.sum(axis=(0, 2)) + 2.0 ** -16 * np.abs(delta2).sum(axis=(0, 2)) + 1e-30
    worst["dlam"] = check_bound_one(got[5], ref[5], dl_bound, f"{label} dlam")
    return worst


@pytest.mark.parametrize("d", [64, 128])
def test_diff_bwd_sweep(d):
    for (Hq, Hkv), N, W, lams, per_head in (((1, 1), 1, 1, 0.8, False),
                                            ((2, 2), 130, 130, 0.8, False),
                                            ((4, 2), 300, 64, [0.8, 0.5, -0.3, 0.0], True),
                                            ((3, 1), 513, 513, 0.5, False),
                                            ((4, 4), 257, 100, [1.2, 0.1, 0.7, 0.9], True),
                                            ((2, 1), 400, 1, 0.6, False)):
        _case(1, Hq, Hkv, N, d, W, lams, per_head, seed=N + W + d)


def test_diff_bwd_batch_scale_and_lambda_zero():
    _case(2, 4, 2, 350, 64, 120, 0.8, False, seed=21, scale=0.09)
    got = _case(1, 2, 1, 200, 128, 200, 0.0, False, seed=22)  # map 2 gets no gradient
    assert got["dq2"] == 0.0 and got["dk2"] == 0.0


def test_diff_bwd_deterministic():
    rng = np.random.default_rng(23)
    B, Hq, Hkv, N, d, W = 1, 4, 2, 700, 64, 300
    a = [_rand(rng, (B, h, N, d)) for h in (Hq, Hkv, Hq, Hkv, Hkv, Hq)]
    r1 = _diff_bwd_gpu(*a, [0.8, 0.2, 0.5, 0.9], True, W, 0.1)
    r2 = _diff_bwd_gpu(*a, [0.8, 0.2, 0.5, 0.9], True, W, 0.1)
    for x, y in zip(r1, r2):
        assert np.array_equal(x, y)


def test_diff_swa_full_size_sampled():
    """The windowed differential workload (B=1, H=16, N=16384, d=64, W=1024, lambda=0.8, K1 key 0
    shifted by +3), computed whole; checked on heads 0, 7 and 15: every dq1, dq2 row of positions
    0..2047 and the dk1, dk2, dv of keys 0..1024 (a prefix holds every reader of those keys), and
    the dq rows and dk, dv keys of the last 256 positions (the W - 1 positions before them hold
    every key their rows read)."""
    w = swa_inputs.WORKLOADS["diff_swa"]
    inp = swa_inputs.make_inputs(w)
    rng = np.random.default_rng(w.seed + 300)
    g = _rand(rng, inp["q1"].shape)
    N, W, sc = w.N, w.W, w.scale
    got = _diff_bwd_gpu(inp["q1"], inp["k1"], inp["q2"], inp["k2"], inp["v"], g, w.lam, False, W,
                        sc)
    names = ("dq1", "dk1", "dq2", "dk2", "dv")
    worst = {}
    for h in (0, 7, 15):
        for p0, p1, rows_q, keys in ((0, 2048, np.arange(2048), np.arange(2048 - W + 1)),
                                     (N - 256 - (W - 1), N, np.arange(N - 256, N),
                                      np.arange(N - 256, N))):
            sub = [np.ascontiguousarray(inp[n][:, h:h + 1, p0:p1]) for n in ("q1", "k1", "q2", "k2",
                                                                             "v")]
            gs = np.ascontiguousarray(g[:, h:h + 1, p0:p1])
            rows = np.arange(rows_q[0], p1) - p0  # every row that reads a checked key
            lam = np.array([np.float32(w.lam)], dtype=np.float64)  # the fp32 lambda the GPU uses
            ref = oracle.diff_bwd(*sub, lam, gs, W, sc)
            bnds, _ = _bounds(*sub, gs, lam, W, sc, rows=rows)
            for t, name in enumerate(names):
                sel = rows_q if name.startswith("dq") else keys
                a = got[t][0, h][sel]
                r = ref[t][0, 0][sel - p0]
                bnd = bnds[t][0, 0][sel - p0]
                worst[name] = max(worst.get(name, 0.0),
                                  check_bound_one(a, r, bnd, f"diff_swa head {h} [{p0},{p1}) {name}"))
    print(f"diff_swa backward sampled: worst |gpu - oracle| / bound = {worst}")


def test_trainable_wrappers_match_the_calls():
    """diff_attention_trainable (a learnable lambda per head) and strided_attention_trainable
    give, through torch autograd, the gradients of the direct C-ABI calls, bit for bit."""
    rng = np.random.default_rng(31)
    B, Hq, Hkv, N, d, W = 1, 4, 2, 300, 64, 100
    arrs = [_rand(rng, (B, h, N, d)) for h in (Hq, Hkv, Hq, Hkv, Hkv, Hq)]
    lams = np.array([0.8, 0.3, -0.2, 0.5], dtype=np.float32)
    sc = 1.0 / np.sqrt(d)
    t = [to_dev(a).requires_grad_() for a in arrs[:5]]
    lam = torch.tensor(lams, device="cuda", requires_grad=True)
    out = pkg.diff_attention_trainable(*t, lam, window=W)
    out.backward(to_dev(arrs[5]))
    want = _diff_bwd_gpu(*arrs, lams, True, W, sc)
    for x, y in zip([a.grad for a in t] + [lam.grad], want):
        assert np.array_equal(x.detach().float().cpu().numpy().astype(np.float64), y)
    # local + strided through its wrapper against strided_attn_bwd
    q, k, v = (to_dev(a).requires_grad_() for a in (arrs[0], arrs[1], arrs[4]))
    o = pkg.strided_attention_trainable(q, k, v, 64, 16)
    o.backward(to_dev(arrs[5]))
    B_, Hq_, N_, d_ = q.shape
    tq, tk, tv, tg = (to_dev(a) for a in (arrs[0], arrs[1], arrs[4], arrs[5]))
    of = torch.empty_like(tq)
    lse = torch.empty((B_, Hq_, N_), dtype=torch.float32, device="cuda")
    pkg.strided_attn_fwd_lse(tq, tk, tv, of, lse, B_, Hq_, Hkv, N_, d_, 64, 16, sc)
    nb = pkg.strided_attn_bwd_workspace_bytes(B_, Hq_, Hkv, N_, d_, 64, 16)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(tq), torch.empty_like(tk), torch.empty_like(tv)
    pkg.strided_attn_bwd(tq, tk, tv, of, lse, tg, dq, dk, dv, B_, Hq_, Hkv, N_, d_, 64, 16, sc,
                         ws, nb)
    torch.cuda.synchronize()
    for x, y in ((q.grad, dq), (k.grad, dk), (v.grad, dv)):
        assert torch.equal(x, y)

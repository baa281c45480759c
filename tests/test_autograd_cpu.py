"""The autograd wrapper's marshalling, on CPU: the library calls are replaced by fakes built on
the fp64 oracle, and the gradients that reach q, k and v through the wrapper are compared with
autograd of a dense masked softmax written in torch.  A wrong argument order, a lost saved
tensor or a dropped window or scale changes the result."""
import numpy as np
import torch

import oracle
import sparse_causal_attention_swa_b300 as pkg


def _f64(t):
    return t.detach().to(torch.float64).numpy()


def _fake_fwd_lse(q, k, v, out, lse, B, Hq, Hkv, N, d, W, scale, stream=None):
    assert q.shape == (B, Hq, N, d) and k.shape == (B, Hkv, N, d) and out.shape == q.shape
    out.copy_(torch.from_numpy(oracle.attn(_f64(q), _f64(k), _f64(v), W, scale)))
    lse.copy_(torch.from_numpy(oracle.lse(_f64(q), _f64(k), W, scale)))


def _fake_bwd(q, k, v, out, lse, g, dq, dk, dv, B, Hq, Hkv, N, d, W, scale, ws, nb, stream=None):
    assert g.dtype == torch.bfloat16 and g.is_contiguous() and ws.numel() == nb
    assert lse.shape == (B, Hq, N) and out.shape == q.shape
    a, b, c = oracle.attn_bwd(_f64(q), _f64(k), _f64(v), _f64(g), W, scale)
    for dst, src in ((dq, a), (dk, b), (dv, c)):
        dst.copy_(torch.from_numpy(src))


def _reference(q, k, v, W, scale):
    q, k, v = (t.detach().to(torch.float64).requires_grad_() for t in (q, k, v))
    g = q.shape[1] // k.shape[1]
    kk, vv = k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1)
    N = q.shape[2]
    i = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    allowed = (j <= i) & (j > i - W)
    s = (q @ kk.transpose(-1, -2)) * scale
    s = s.masked_fill(~allowed, float("-inf"))
    return torch.softmax(s, dim=-1) @ vv, (q, k, v)


def test_autograd_wrapper_marshalling(monkeypatch):
    monkeypatch.setattr(pkg, "swa_attn_fwd_lse", _fake_fwd_lse)
    monkeypatch.setattr(pkg, "swa_attn_bwd", _fake_bwd)
    monkeypatch.setattr(pkg, "swa_attn_bwd_workspace_bytes", lambda B, Hq, N: 64)
    torch.manual_seed(0)
    B, Hq, Hkv, N, d, W, scale = 2, 4, 2, 23, 8, 5, 0.3
    q, k, v = (torch.randn(B, h, N, d).to(torch.bfloat16).requires_grad_()
               for h in (Hq, Hkv, Hkv))
    out = pkg._swa_autograd_fn().apply(q, k, v, W, scale)
    dout = torch.randn(B, Hq, N, d).to(torch.bfloat16)
    out.backward(dout)
    ref_out, (rq, rk, rv) = _reference(q, k, v, W, scale)
    ref_out.backward(dout.to(torch.float64))
    tol = dict(rtol=2e-2, atol=2e-2)
    torch.testing.assert_close(out.to(torch.float64), ref_out.detach(), **tol)
    for got, ref in ((q.grad, rq.grad), (k.grad, rk.grad), (v.grad, rv.grad)):
        assert got.dtype == torch.bfloat16 and got.shape == ref.shape
        torch.testing.assert_close(got.to(torch.float64), ref, **tol)


def test_trainable_wrapper_wants_cuda_bf16():
    x = torch.zeros(1, 1, 4, 8, dtype=torch.bfloat16)
    try:
        pkg.swa_attention_trainable(x, x, x, 2)
    except ValueError:
        return
    raise AssertionError("CPU tensors must be rejected")


# ------------------------------------------------------------------ local + strided, global prefix
def _dense_mask(N, W, kind, x):
    i = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    m = (j <= i) & (j > i - W)
    if kind == "strided":
        m |= (j <= i) & (j % x == 0)
    else:
        m |= (j <= i) & (j < x)
    return m


def _reference_mask(q, k, v, W, kind, x, scale):
    q, k, v = (t.detach().to(torch.float64).requires_grad_() for t in (q, k, v))
    g = q.shape[1] // k.shape[1]
    kk, vv = k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1)
    s = (q @ kk.transpose(-1, -2)) * scale
    s = s.masked_fill(~_dense_mask(q.shape[2], W, kind, x), float("-inf"))
    return torch.softmax(s, dim=-1) @ vv, (q, k, v)


def test_mask_autograd_wrapper_marshalling(monkeypatch):
    for kind, x in (("strided", 4), ("global", 3)):
        def fwd(q, k, v, out, lse, B, Hq, Hkv, N, d, W, xx, scale, stream=None, kind=kind):
            assert xx == x
            out.copy_(torch.from_numpy(oracle.attn(_f64(q), _f64(k), _f64(v), W, scale, kind=kind,
                                                   stride=xx)))
            lse.copy_(torch.from_numpy(oracle.lse(_f64(q), _f64(k), W, scale, kind=kind,
                                                  stride=xx)))

        def bwd(q, k, v, out, lse, g, dq, dk, dv, B, Hq, Hkv, N, d, W, xx, scale, ws, nb,
                stream=None, kind=kind):
            assert g.dtype == torch.bfloat16 and ws.numel() == nb and xx == x
            a, b, c = oracle.attn_bwd(_f64(q), _f64(k), _f64(v), _f64(g), W, scale, kind=kind,
                                      stride=xx)
            for dst, src in ((dq, a), (dk, b), (dv, c)):
                dst.copy_(torch.from_numpy(src))

        monkeypatch.setattr(pkg, f"{kind}_attn_fwd_lse", fwd)
        monkeypatch.setattr(pkg, f"{kind}_attn_bwd", bwd)
        monkeypatch.setattr(pkg, f"{kind}_attn_bwd_workspace_bytes", lambda *a: 64)
        torch.manual_seed(1)
        B, Hq, Hkv, N, d, W, scale = 2, 4, 2, 29, 8, 5, 0.3
        q, k, v = (torch.randn(B, h, N, d).to(torch.bfloat16).requires_grad_()
                   for h in (Hq, Hkv, Hkv))
        out = pkg._mask_autograd_fn().apply(q, k, v, kind, W, x, scale)
        dout = torch.randn(B, Hq, N, d).to(torch.bfloat16)
        out.backward(dout)
        ref_out, (rq, rk, rv) = _reference_mask(q, k, v, W, kind, x, scale)
        ref_out.backward(dout.to(torch.float64))
        tol = dict(rtol=2e-2, atol=2e-2)
        torch.testing.assert_close(out.to(torch.float64), ref_out.detach(), **tol)
        for got, ref in ((q.grad, rq.grad), (k.grad, rk.grad), (v.grad, rv.grad)):
            torch.testing.assert_close(got.to(torch.float64), ref, **tol)


# ------------------------------------------------------------------ differential, learnable lambda
def test_diff_autograd_wrapper_marshalling(monkeypatch):
    def fwd_lse(q, k, v, out, lse, B, Hq, Hkv, N, d, W, scale, stream=None):
        out.copy_(torch.from_numpy(oracle.attn(_f64(q), _f64(k), _f64(v), W, scale)))
        lse.copy_(torch.from_numpy(oracle.lse(_f64(q), _f64(k), W, scale)))

    def diff_fwd(q1, k1, q2, k2, v, lam, lam_heads, out, B, Hq, Hkv, N, d, W, scale, stream=None):
        assert lam_heads is not None and lam_heads.dtype == torch.float32
        out.copy_(torch.from_numpy(oracle.diff_heads(_f64(q1), _f64(k1), _f64(q2), _f64(k2),
                                                     _f64(v), lam_heads.numpy(), scale, W=W)))

    def diff_bwd(q1, k1, q2, k2, v, lam, lam_heads, o1, l1, o2, l2, g, dq1, dk1, dq2, dk2, dv,
                 dlam, B, Hq, Hkv, N, d, W, scale, ws, nb, stream=None):
        assert ws.numel() == nb and g.dtype == torch.bfloat16
        res = oracle.diff_bwd(_f64(q1), _f64(k1), _f64(q2), _f64(k2), _f64(v),
                              lam_heads.numpy().astype(np.float64), _f64(g), W, scale)
        for dst, src in zip((dq1, dk1, dq2, dk2, dv, dlam), res):
            dst.copy_(torch.from_numpy(src))

    monkeypatch.setattr(pkg, "swa_attn_fwd_lse", fwd_lse)
    monkeypatch.setattr(pkg, "diff_swa_attn_fwd", diff_fwd)
    monkeypatch.setattr(pkg, "diff_attn_bwd", diff_bwd)
    monkeypatch.setattr(pkg, "diff_attn_bwd_workspace_bytes", lambda *a: 64)
    torch.manual_seed(2)
    B, Hq, Hkv, N, d, W, scale = 1, 4, 2, 19, 8, 6, 0.35
    q1, k1, q2, k2, v = (torch.randn(B, h, N, d).to(torch.bfloat16).requires_grad_()
                         for h in (Hq, Hkv, Hq, Hkv, Hkv))
    lam = torch.tensor([0.8, 0.3, 0.5, 0.1], requires_grad=True)
    out = pkg._diff_autograd_fn().apply(q1, k1, q2, k2, v, lam, W, scale)
    dout = torch.randn(B, Hq, N, d).to(torch.bfloat16)
    out.backward(dout)
    # reference: autograd of the dense masked softmaxes
    r = [t.detach().to(torch.float64).requires_grad_() for t in (q1, k1, q2, k2, v)]
    rl = lam.detach().to(torch.float64).requires_grad_()
    mask = _dense_mask(N, W, "global", 0)  # the window alone
    g = Hq // Hkv

    def amap(q, k):
        s = (q @ k.repeat_interleave(g, dim=1).transpose(-1, -2)) * scale
        return torch.softmax(s.masked_fill(~mask, float("-inf")), dim=-1)

    vv = r[4].repeat_interleave(g, dim=1)
    ref = (amap(r[0], r[1]) - rl.view(1, Hq, 1, 1) * amap(r[2], r[3])) @ vv
    ref.backward(dout.to(torch.float64))
    tol = dict(rtol=2e-2, atol=2e-2)
    torch.testing.assert_close(out.to(torch.float64), ref.detach(), **tol)
    for got, want in zip((q1.grad, k1.grad, q2.grad, k2.grad, v.grad), r):
        torch.testing.assert_close(got.to(torch.float64), want.grad, **tol)
    torch.testing.assert_close(lam.grad.to(torch.float64), rl.grad, rtol=2e-2, atol=5e-2)

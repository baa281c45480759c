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

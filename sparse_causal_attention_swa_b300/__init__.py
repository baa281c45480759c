"""B300 (sm_103a) causal sliding-window, local+strided and differential attention forward.

The compute lives in ``libswa_b300.so`` (hand-written CUDA for sm_103a: TMA-fed shared
memory rings, tcgen05 MMAs accumulating in tensor memory, an exp2 online softmax).  This
module is a thin ctypes binding with the same names as the C ABI declared in
``include/swa_b300.h``; it only marshals arguments.  PyTorch is used for device memory
and streams.  There is no CPU fallback: if the library is missing, every call raises.

Low-level calls (pointers or tensors, explicit sizes, asynchronous on ``stream``):
    swa_attn_fwd, strided_attn_fwd, diff_attn_fwd, diff_attn_fwd_heads, diff_swa_attn_fwd,
    strided_attn_fwd_noalloc, swa_attn_fwd_lse, strided_attn_fwd_lse, global_attn_fwd,
    global_attn_fwd_lse, swa_attn_bwd_workspace_bytes, swa_attn_bwd,
    strided_attn_bwd_workspace_bytes, strided_attn_bwd, global_attn_bwd_workspace_bytes,
    global_attn_bwd, diff_attn_bwd_workspace_bytes, diff_attn_bwd,
    swa_decode_workspace_bytes, swa_decode_fwd, swa_cache_append, swa_chunk_fwd,
    swa_cache_gather,
    swa_status_string, swa_device_status, swa_watchdog_selftest
Convenience wrappers on [B, H, N, d] bf16 tensors (allocate ``out``; CPU inputs are
copied to the current CUDA device and the result copied back):
    swa_attention, strided_attention, diff_attention, swa_decode
For training, swa_attention_trainable, strided_attention_trainable,
global_attention_trainable and diff_attention_trainable (CUDA tensors) record the forward for
autograd and run swa_attn_bwd / strided_attn_bwd / global_attn_bwd / diff_attn_bwd in the
backward.
"""
from __future__ import annotations

import ctypes
import math
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_PKG, "libswa_b300.so")

SWA_OK = 0
_lib = None


class SwaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        detail = ""
        if code == 5:  # SWA_ERR_CUDA: which CUDA call failed, and how
            detail = load().swa_last_error_detail().decode()
        super().__init__(f"{where}: {swa_status_string(code)} (status {code})"
                         + (f" [{detail}]" if detail else ""))


def load():
    """Load the compiled library; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIBRARY_PATH):
            raise RuntimeError(
                f"{LIBRARY_PATH} is missing: the CUDA extension is not built "
                "(run `python -m sparse_causal_attention_swa_b300._build`)")
        lib = ctypes.CDLL(LIBRARY_PATH)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.swa_attn_fwd.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P]
        lib.swa_attn_fwd.restype = I
        lib.strided_attn_fwd.argtypes = [P, P, P, P, I, I, I, I, I, I, I, F, P]
        lib.strided_attn_fwd.restype = I
        lib.global_attn_fwd.argtypes = [P, P, P, P, I, I, I, I, I, I, I, F, P]
        lib.global_attn_fwd.restype = I
        lib.swa_attn_fwd_lse.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, P]
        lib.swa_attn_fwd_lse.restype = I
        lib.strided_attn_fwd_lse.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, P]
        lib.strided_attn_fwd_lse.restype = I
        lib.strided_attn_fwd_noalloc.argtypes = [P, P, P, P, I, I, I, I, I, I, I, F, P]
        lib.strided_attn_fwd_noalloc.restype = I
        lib.diff_attn_fwd.argtypes = [P, P, P, P, P, F, P, I, I, I, I, I, F, P]
        lib.diff_attn_fwd.restype = I
        lib.diff_attn_fwd_heads.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, F, P]
        lib.diff_attn_fwd_heads.restype = I
        lib.diff_swa_attn_fwd.argtypes = [P, P, P, P, P, F, P, P, I, I, I, I, I, I, F, P]
        lib.diff_swa_attn_fwd.restype = I
        lib.swa_attn_bwd_workspace_bytes.argtypes = [I, I, I]
        lib.swa_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.swa_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P,
                                     ctypes.c_size_t, P]
        lib.swa_attn_bwd.restype = I
        lib.strided_attn_bwd_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
        lib.strided_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.strided_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P,
                                         ctypes.c_size_t, P]
        lib.strided_attn_bwd.restype = I
        lib.global_attn_bwd_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
        lib.global_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.global_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P,
                                        ctypes.c_size_t, P]
        lib.global_attn_bwd.restype = I
        lib.global_attn_fwd_lse.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, P]
        lib.global_attn_fwd_lse.restype = I
        lib.diff_attn_bwd_workspace_bytes.argtypes = [I, I, I, I, I]
        lib.diff_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.diff_attn_bwd.argtypes = [P, P, P, P, P, F, P, P, P, P, P, P, P, P, P, P, P, P, I, I,
                                      I, I, I, I, F, P, ctypes.c_size_t, P]
        lib.diff_attn_bwd.restype = I
        SZ = ctypes.c_size_t
        lib.swa_decode_workspace_bytes.argtypes = [I, I, I, I]
        lib.swa_decode_workspace_bytes.restype = SZ
        lib.swa_decode_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, F, P, SZ, P]
        lib.swa_decode_fwd.restype = I
        lib.swa_cache_append.argtypes = [P, P, P, P, P, I, I, I, I, I, P]
        lib.swa_cache_append.restype = I
        lib.swa_chunk_fwd.argtypes = [P, P, P, P, I, I, I, I, I, I, I, F, P]
        lib.swa_chunk_fwd.restype = I
        lib.swa_cache_gather.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P]
        lib.swa_cache_gather.restype = I
        lib.swa_status_string.argtypes = [I]
        lib.swa_status_string.restype = ctypes.c_char_p
        lib.swa_last_error_detail.argtypes = []
        lib.swa_last_error_detail.restype = ctypes.c_char_p
        lib.swa_device_status.argtypes = [P]
        lib.swa_device_status.restype = I
        lib.swa_watchdog_selftest.argtypes = [I, P]
        lib.swa_watchdog_selftest.restype = I
        _lib = lib
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, where: str):
    if code != SWA_OK:
        raise SwaError(code, where)


def swa_status_string(status: int) -> str:
    return load().swa_status_string(int(status)).decode()


# ---------------------------------------------------------------- C-ABI mirrors
def swa_attn_fwd(q, k, v, out, B, Hq, Hkv, N, d, W, scale, stream=None):
    _check(load().swa_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, N, d, W,
                               float(scale), _stream(stream)), "swa_attn_fwd")


def strided_attn_fwd(q, k, v, out, B, Hq, Hkv, N, d, W, stride, scale, stream=None):
    _check(load().strided_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, N, d, W,
                                   stride, float(scale), _stream(stream)), "strided_attn_fwd")


def global_attn_fwd(q, k, v, out, B, Hq, Hkv, N, d, W, n_global, scale, stream=None):
    """Window plus a global prefix of n_global tokens (causal)."""
    _check(load().global_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, N, d, W,
                                  n_global, float(scale), _stream(stream)), "global_attn_fwd")


def swa_attn_fwd_lse(q, k, v, out, lse, B, Hq, Hkv, N, d, W, scale, stream=None):
    """swa_attn_fwd that also writes each row's log-sum-exp (float32 [B, Hq, N])."""
    _check(load().swa_attn_fwd_lse(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, N,
                                   d, W, float(scale), _stream(stream)), "swa_attn_fwd_lse")


def strided_attn_fwd_lse(q, k, v, out, lse, B, Hq, Hkv, N, d, W, stride, scale, stream=None):
    _check(load().strided_attn_fwd_lse(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq,
                                       Hkv, N, d, W, stride, float(scale), _stream(stream)),
           "strided_attn_fwd_lse")


def strided_attn_fwd_noalloc(q, k, v, out, B, Hq, Hkv, N, d, W, stride, scale, stream=None):
    """strided_attn_fwd for callers that cannot allocate device memory: the tile list is
    rebuilt on the stream inside a fixed device array owned by the library."""
    _check(load().strided_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, N,
                                           d, W, stride, float(scale), _stream(stream)),
           "strided_attn_fwd_noalloc")


def diff_attn_fwd(q1, k1, q2, k2, v, lam, out, B, Hq, Hkv, N, d, scale, stream=None):
    _check(load().diff_attn_fwd(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v), float(lam),
                                _ptr(out), B, Hq, Hkv, N, d, float(scale), _stream(stream)),
           "diff_attn_fwd")


def swa_decode_workspace_bytes(B, Hq, W, d) -> int:
    return int(load().swa_decode_workspace_bytes(B, Hq, W, d))


def swa_decode_fwd(q, k_cache, v_cache, pos, out, B, Hq, Hkv, W, d, scale, workspace,
                   workspace_bytes, stream=None):
    _check(load().swa_decode_fwd(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(pos), _ptr(out), B,
                                 Hq, Hkv, W, d, float(scale), _ptr(workspace),
                                 int(workspace_bytes), _stream(stream)), "swa_decode_fwd")


def swa_cache_append(k_new, v_new, k_cache, v_cache, pos, B, Hkv, W, d, n=1, stream=None):
    _check(load().swa_cache_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(pos), B, Hkv, W, d, n, _stream(stream)),
           "swa_cache_append")


def swa_chunk_fwd(q, k, v, out, B, Hq, Hkv, C, L, d, W, scale, stream=None):
    """Queries are the last C of L context positions (chunked prefill)."""
    _check(load().swa_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, C, L, d, W,
                                float(scale), _stream(stream)), "swa_chunk_fwd")


def swa_cache_gather(k_cache, v_cache, k_ctx, v_ctx, B, Hkv, W, d, pos0, nctx, ctx_rows,
                     stream=None):
    _check(load().swa_cache_gather(_ptr(k_cache), _ptr(v_cache), _ptr(k_ctx), _ptr(v_ctx), B, Hkv,
                                   W, d, pos0, nctx, ctx_rows, _stream(stream)),
           "swa_cache_gather")


def diff_attn_fwd_heads(q1, k1, q2, k2, v, lam, out, B, Hq, Hkv, N, d, scale, stream=None):
    """diff_attn_fwd with one lambda per query head; ``lam`` is a float32 [Hq] device tensor."""
    _check(load().diff_attn_fwd_heads(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v), _ptr(lam),
                                      _ptr(out), B, Hq, Hkv, N, d, float(scale), _stream(stream)),
           "diff_attn_fwd_heads")


def diff_swa_attn_fwd(q1, k1, q2, k2, v, lam, lam_heads, out, B, Hq, Hkv, N, d, W, scale,
                      stream=None):
    """Differential attention with both maps under the window W; ``lam_heads`` is a float32
    [Hq] device tensor or None (then the scalar ``lam`` serves every head)."""
    _check(load().diff_swa_attn_fwd(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v), float(lam),
                                    None if lam_heads is None else _ptr(lam_heads), _ptr(out), B,
                                    Hq, Hkv, N, d, int(W), float(scale), _stream(stream)),
           "diff_swa_attn_fwd")


def swa_attn_bwd_workspace_bytes(B, Hq, N) -> int:
    return int(load().swa_attn_bwd_workspace_bytes(B, Hq, N))


def swa_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, W, scale, workspace,
                 workspace_bytes, stream=None):
    """Gradients dq, dk, dv of causal SWA for the upstream gradient ``dout``; ``out`` and
    ``lse`` come from swa_attn_fwd_lse with the same arguments."""
    _check(load().swa_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                               _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, int(W),
                               float(scale), _ptr(workspace), int(workspace_bytes),
                               _stream(stream)), "swa_attn_bwd")


def strided_attn_bwd_workspace_bytes(B, Hq, Hkv, N, d, W, stride) -> int:
    return int(load().strided_attn_bwd_workspace_bytes(B, Hq, Hkv, N, d, W, stride))


def strided_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, W, stride, scale,
                     workspace, workspace_bytes, stream=None):
    """Gradients of local + strided attention; ``out`` and ``lse`` come from
    strided_attn_fwd_lse with the same arguments."""
    _check(load().strided_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                   _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, int(W),
                                   int(stride), float(scale), _ptr(workspace),
                                   int(workspace_bytes), _stream(stream)), "strided_attn_bwd")


def global_attn_fwd_lse(q, k, v, out, lse, B, Hq, Hkv, N, d, W, n_global, scale, stream=None):
    _check(load().global_attn_fwd_lse(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq,
                                      Hkv, N, d, int(W), int(n_global), float(scale),
                                      _stream(stream)), "global_attn_fwd_lse")


def global_attn_bwd_workspace_bytes(B, Hq, Hkv, N, d, W, n_global) -> int:
    return int(load().global_attn_bwd_workspace_bytes(B, Hq, Hkv, N, d, W, n_global))


def global_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, W, n_global, scale,
                    workspace, workspace_bytes, stream=None):
    """Gradients of the window plus a global prefix; ``out`` and ``lse`` come from
    global_attn_fwd_lse with the same arguments."""
    _check(load().global_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                  _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, int(W),
                                  int(n_global), float(scale), _ptr(workspace),
                                  int(workspace_bytes), _stream(stream)), "global_attn_bwd")


def diff_attn_bwd_workspace_bytes(B, Hq, Hkv, N, d) -> int:
    return int(load().diff_attn_bwd_workspace_bytes(B, Hq, Hkv, N, d))


def diff_attn_bwd(q1, k1, q2, k2, v, lam, lam_heads, out1, lse1, out2, lse2, dout, dq1, dk1,
                  dq2, dk2, dv, dlam, B, Hq, Hkv, N, d, W, scale, workspace, workspace_bytes,
                  stream=None):
    """Gradients of differential attention; out1 / lse1 and out2 / lse2 come from
    swa_attn_fwd_lse on (q1, k1, v) and (q2, k2, v); ``dlam`` (float32 [Hq] or None) receives
    each head's lambda gradient."""
    _check(load().diff_attn_bwd(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v), float(lam),
                                _ptr(lam_heads), _ptr(out1), _ptr(lse1), _ptr(out2), _ptr(lse2),
                                _ptr(dout), _ptr(dq1), _ptr(dk1), _ptr(dq2), _ptr(dk2), _ptr(dv),
                                _ptr(dlam), B, Hq, Hkv, N, d, int(W), float(scale),
                                _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "diff_attn_bwd")


def swa_device_status(stream=None) -> int:
    return int(load().swa_device_status(_stream(stream)))


def swa_watchdog_selftest(limit_us: int, stream=None):
    _check(load().swa_watchdog_selftest(int(limit_us), _stream(stream)), "swa_watchdog_selftest")


# ---------------------------------------------------------------- tensor wrappers
def _prepare(*ts):
    import torch

    dev = None
    for t in ts:
        if t.is_cuda:
            dev = t.device
    if dev is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    out = []
    for t in ts:
        if t.dtype != torch.bfloat16 or t.dim() != 4:
            raise ValueError("expected bf16 tensors of shape [B, H, N, d]")
        out.append(t.to(dev, non_blocking=True).contiguous())
    return out, dev


def _finish(out, like):
    return out if like.is_cuda else out.to("cpu", non_blocking=False)


def swa_attention(q, k, v, window: int, scale: float | None = None, out=None):
    """Causal sliding-window attention, window counting the current position."""
    import torch

    (qd, kd, vd), dev = _prepare(q, k, v)
    B, Hq, N, d = qd.shape
    o = out if out is not None else torch.empty_like(qd)
    swa_attn_fwd(qd, kd, vd, o, B, Hq, kd.shape[1], N, d, int(window),
                 scale if scale is not None else 1.0 / math.sqrt(d))
    return _finish(o, q)


def strided_attention(q, k, v, window: int, stride: int, scale: float | None = None, out=None):
    """Local window plus every stride-th key (absolute multiples of stride), causal."""
    import torch

    (qd, kd, vd), dev = _prepare(q, k, v)
    B, Hq, N, d = qd.shape
    o = out if out is not None else torch.empty_like(qd)
    strided_attn_fwd(qd, kd, vd, o, B, Hq, kd.shape[1], N, d, int(window), int(stride),
                     scale if scale is not None else 1.0 / math.sqrt(d))
    return _finish(o, q)


def diff_attention(q1, k1, q2, k2, v, lam: float, scale: float | None = None, out=None,
                   window: int | None = None):
    """(softmax(Q1 K1^T s + M) - lam softmax(Q2 K2^T s + M)) V, M causal, or the sliding
    window of width ``window`` when one is given."""
    import torch

    (a, b_, c, e, f), dev = _prepare(q1, k1, q2, k2, v)
    B, Hq, N, d = a.shape
    o = out if out is not None else torch.empty_like(a)
    sc = scale if scale is not None else 1.0 / math.sqrt(d)
    if window is None:
        diff_attn_fwd(a, b_, c, e, f, lam, o, B, Hq, b_.shape[1], N, d, sc)
    else:
        diff_swa_attn_fwd(a, b_, c, e, f, lam, None, o, B, Hq, b_.shape[1], N, d, int(window), sc)
    return _finish(o, q1)


_SWA_AUTOGRAD = None


def _swa_autograd_fn():
    """torch.autograd.Function whose forward is swa_attn_fwd_lse and whose backward is
    swa_attn_bwd (built on first use, so importing this module does not import torch)."""
    global _SWA_AUTOGRAD
    if _SWA_AUTOGRAD is None:
        import torch

        class SwaAttention(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q, k, v, window, scale):
                B, Hq, N, d = q.shape
                out = torch.empty_like(q)
                lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
                swa_attn_fwd_lse(q, k, v, out, lse, B, Hq, k.shape[1], N, d, window, scale)
                ctx.save_for_backward(q, k, v, out, lse)
                ctx.window, ctx.scale = window, scale
                return out

            @staticmethod
            def backward(ctx, dout):
                q, k, v, out, lse = ctx.saved_tensors
                B, Hq, N, d = q.shape
                g = dout.to(torch.bfloat16).contiguous()
                dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
                nb = swa_attn_bwd_workspace_bytes(B, Hq, N)
                ws = torch.empty(nb, dtype=torch.uint8, device=q.device)
                swa_attn_bwd(q, k, v, out, lse, g, dq, dk, dv, B, Hq, k.shape[1], N, d,
                             ctx.window, ctx.scale, ws, nb)
                return dq, dk, dv, None, None

        _SWA_AUTOGRAD = SwaAttention
    return _SWA_AUTOGRAD


def swa_attention_trainable(q, k, v, window: int, scale: float | None = None):
    """Causal sliding-window attention that records itself for autograd: the forward is
    swa_attn_fwd_lse, the backward swa_attn_bwd (dq, dk, dv, all bf16).  q, k, v: bf16 CUDA
    tensors [B, H, N, d]."""
    import torch

    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_cuda:
            raise ValueError("expected bf16 CUDA tensors of shape [B, H, N, d]")
    sc = scale if scale is not None else 1.0 / math.sqrt(q.shape[-1])
    return _swa_autograd_fn().apply(q.contiguous(), k.contiguous(), v.contiguous(), int(window),
                                    float(sc))


_MASK_AUTOGRAD = None


def _mask_autograd_fn():
    """torch.autograd.Function for the local + strided and global-prefix masks: the forward is
    strided_attn_fwd_lse / global_attn_fwd_lse, the backward strided_attn_bwd /
    global_attn_bwd (``x`` is the stride or the number of global tokens)."""
    global _MASK_AUTOGRAD
    if _MASK_AUTOGRAD is None:
        import torch

        class MaskedAttention(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q, k, v, kind, window, x, scale):
                B, Hq, N, d = q.shape
                out = torch.empty_like(q)
                lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
                fwd = strided_attn_fwd_lse if kind == "strided" else global_attn_fwd_lse
                fwd(q, k, v, out, lse, B, Hq, k.shape[1], N, d, window, x, scale)
                ctx.save_for_backward(q, k, v, out, lse)
                ctx.kind, ctx.window, ctx.x, ctx.scale = kind, window, x, scale
                return out

            @staticmethod
            def backward(ctx, dout):
                q, k, v, out, lse = ctx.saved_tensors
                B, Hq, N, d = q.shape
                Hkv = k.shape[1]
                g = dout.to(torch.bfloat16).contiguous()
                dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
                if ctx.kind == "strided":
                    wsf, bwd = strided_attn_bwd_workspace_bytes, strided_attn_bwd
                else:
                    wsf, bwd = global_attn_bwd_workspace_bytes, global_attn_bwd
                nb = wsf(B, Hq, Hkv, N, d, ctx.window, ctx.x)
                ws = torch.empty(nb, dtype=torch.uint8, device=q.device)
                bwd(q, k, v, out, lse, g, dq, dk, dv, B, Hq, Hkv, N, d, ctx.window, ctx.x,
                    ctx.scale, ws, nb)
                return dq, dk, dv, None, None, None, None

        _MASK_AUTOGRAD = MaskedAttention
    return _MASK_AUTOGRAD


_DIFF_AUTOGRAD = None


def _diff_autograd_fn():
    """torch.autograd.Function for differential attention with one lambda per head: the forward
    is diff_swa_attn_fwd (per-head lambda) for the output, plus swa_attn_fwd_lse on both maps
    for the outputs and log-sum-exps the backward needs; the backward is diff_attn_bwd, which
    also returns the gradient of every head's lambda."""
    global _DIFF_AUTOGRAD
    if _DIFF_AUTOGRAD is None:
        import torch

        class DiffAttention(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q1, k1, q2, k2, v, lam, window, scale):
                B, Hq, N, d = q1.shape
                Hkv = k1.shape[1]
                outs = []
                for qq, kk in ((q1, k1), (q2, k2)):
                    o = torch.empty_like(qq)
                    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=qq.device)
                    swa_attn_fwd_lse(qq, kk, v, o, lse, B, Hq, Hkv, N, d, window, scale)
                    outs += [o, lse]
                lam32 = lam.detach().to(torch.float32).contiguous()
                out = torch.empty_like(q1)
                diff_swa_attn_fwd(q1, k1, q2, k2, v, 0.0, lam32, out, B, Hq, Hkv, N, d, window,
                                  scale)
                ctx.save_for_backward(q1, k1, q2, k2, v, lam32, *outs)
                ctx.window, ctx.scale = window, scale
                return out

            @staticmethod
            def backward(ctx, dout):
                q1, k1, q2, k2, v, lam32, o1, l1, o2, l2 = ctx.saved_tensors
                B, Hq, N, d = q1.shape
                Hkv = k1.shape[1]
                g = dout.to(torch.bfloat16).contiguous()
                grads = [torch.empty_like(x) for x in (q1, k1, q2, k2, v)]
                dlam = torch.empty(Hq, dtype=torch.float32, device=q1.device)
                nb = diff_attn_bwd_workspace_bytes(B, Hq, Hkv, N, d)
                ws = torch.empty(nb, dtype=torch.uint8, device=q1.device)
                diff_attn_bwd(q1, k1, q2, k2, v, 0.0, lam32, o1, l1, o2, l2, g, *grads, dlam, B,
                              Hq, Hkv, N, d, ctx.window, ctx.scale, ws, nb)
                return (*grads, dlam, None, None)

        _DIFF_AUTOGRAD = DiffAttention
    return _DIFF_AUTOGRAD


def _want_cuda_bf16(*ts):
    import torch

    for t in ts:
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_cuda:
            raise ValueError("expected bf16 CUDA tensors of shape [B, H, N, d]")


def strided_attention_trainable(q, k, v, window: int, stride: int, scale: float | None = None):
    """Local + strided attention that records itself for autograd (forward
    strided_attn_fwd_lse, backward strided_attn_bwd)."""
    _want_cuda_bf16(q, k, v)
    sc = scale if scale is not None else 1.0 / math.sqrt(q.shape[-1])
    return _mask_autograd_fn().apply(q.contiguous(), k.contiguous(), v.contiguous(), "strided",
                                     int(window), int(stride), float(sc))


def global_attention_trainable(q, k, v, window: int, n_global: int, scale: float | None = None):
    """Window plus a global prefix that records itself for autograd (forward
    global_attn_fwd_lse, backward global_attn_bwd)."""
    _want_cuda_bf16(q, k, v)
    sc = scale if scale is not None else 1.0 / math.sqrt(q.shape[-1])
    return _mask_autograd_fn().apply(q.contiguous(), k.contiguous(), v.contiguous(), "global",
                                     int(window), int(n_global), float(sc))


def diff_attention_trainable(q1, k1, q2, k2, v, lam, window: int | None = None,
                             scale: float | None = None):
    """Differential attention with a learnable lambda per head (``lam``: a float tensor [Hq] on
    the device, e.g. an nn.Parameter) that records itself for autograd; gradients reach q1, k1,
    q2, k2, v and lam.  window None is the causal form."""
    _want_cuda_bf16(q1, k1, q2, k2, v)
    N = q1.shape[2]
    sc = scale if scale is not None else 1.0 / math.sqrt(q1.shape[-1])
    return _diff_autograd_fn().apply(q1.contiguous(), k1.contiguous(), q2.contiguous(),
                                     k2.contiguous(), v.contiguous(), lam,
                                     N if window is None else int(window), float(sc))


def swa_decode(q, k_cache, v_cache, pos, scale: float | None = None, out=None, workspace=None):
    """One decode step against W-slot rolling caches: q [B, Hq, d], k_cache / v_cache
    [B, Hkv, W, d] (bf16), pos [B] int32 absolute query positions.  Allocates the output and,
    unless one is passed, the split workspace (a uint8 tensor)."""
    import torch

    (qd, kd, vd), dev = _prepare(q.unsqueeze(2), k_cache, v_cache)
    qd = qd.squeeze(2)
    pd = pos.to(dev, dtype=torch.int32).contiguous()
    B, Hq, d = qd.shape
    Hkv, W = kd.shape[1], kd.shape[2]
    nbytes = swa_decode_workspace_bytes(B, Hq, W, d)
    ws = workspace if workspace is not None else torch.empty(nbytes, dtype=torch.uint8,
                                                             device=dev)
    o = out if out is not None else torch.empty_like(qd)
    swa_decode_fwd(qd, kd, vd, pd, o, B, Hq, Hkv, W, d,
                   scale if scale is not None else 1.0 / math.sqrt(d), ws, ws.numel())
    return _finish(o, q)

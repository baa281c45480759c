"""GPU parity of chunked prefill (the SWA note's §4.3: a chunk's queries need different
windows across the history and the chunk itself): swa_chunk_fwd, and the rolling-cache
flow swa_cache_gather -> swa_chunk_fwd -> swa_cache_append, against the fp64 oracle's rows
of windowed attention over the whole sequence."""
import numpy as np
import pytest
import torch

import oracle
from swa_inputs import f32_to_bf16_bits
import sparse_causal_attention_swa_b300 as pkg
from gpu_util import ATOL, RTOL, to_dev

pytestmark = pytest.mark.gpu


def _rand(rng, shape):
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def _check(got, ref, label):
    assert np.all(np.isfinite(got)), f"{label}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{label}: {int(bad.sum())} out of tolerance, max err {err.max():.3e}"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("heads", [(4, 2), (3, 1), (2, 2)])
def test_chunk_is_the_last_rows_of_window_attention(d, heads):
    Hq, Hkv = heads
    B = 2
    for L, C, W in ((300, 77, 64), (700, 256, 300), (513, 513, 100), (1000, 129, 1000),
                    (260, 1, 17), (900, 400, 128)):
        rng = np.random.default_rng(L + C + W + d)
        q = _rand(rng, (B, Hq, L, d))
        k = _rand(rng, (B, Hkv, L, d))
        v = _rand(rng, (B, Hkv, L, d))
        scale = 1.0 / np.sqrt(d)
        qc = np.ascontiguousarray(q[:, :, L - C:])
        tq, tk, tv = to_dev(qc), to_dev(k), to_dev(v)
        out = torch.full_like(tq, float("nan"))
        pkg.swa_chunk_fwd(tq, tk, tv, out, B, Hq, Hkv, C, L, d, W, scale)
        torch.cuda.synchronize()
        assert pkg.swa_device_status() == 0
        got = out.float().cpu().numpy().astype(np.float64)
        ref = oracle.attn(q, k, v, W, scale, kind="window", rows=np.arange(L - C, L))
        _check(got, ref, f"L={L} C={C} W={W} d={d} heads={heads}")


def test_rolling_cache_chunked_prefill():
    """A whole sequence prefilled chunk by chunk through a W-slot rolling cache: the context
    of a chunk is the W-1 positions before it (gathered from the cache in time order) plus
    the chunk itself; the chunk is then appended to the cache.  Every output row must equal
    that row of windowed attention over the whole sequence."""
    B, Hq, Hkv, T, d, W = 2, 4, 2, 1000, 128, 300
    rng = np.random.default_rng(11)
    q = _rand(rng, (B, Hq, T, d))
    k = _rand(rng, (B, Hkv, T, d))
    v = _rand(rng, (B, Hkv, T, d))
    scale = 0.09
    ref = oracle.attn(q, k, v, W, scale, kind="window")
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    kc = torch.full((B, Hkv, W, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    got = torch.empty((B, Hq, T, d), dtype=torch.bfloat16, device="cuda")
    pos0 = 0
    for C in (100, 250, 1, 130, 300, 219):  # ragged chunk sizes, summing to T
        nctx = min(pos0, W - 1)
        L = nctx + C
        kx = torch.empty((B, Hkv, L, d), dtype=torch.bfloat16, device="cuda")
        vx = torch.empty_like(kx)
        pkg.swa_cache_gather(kc, vc, kx, vx, B, Hkv, W, d, pos0, nctx, L)
        kx[:, :, nctx:] = tk[:, :, pos0:pos0 + C]
        vx[:, :, nctx:] = tv[:, :, pos0:pos0 + C]
        qc = tq[:, :, pos0:pos0 + C].contiguous()
        out = torch.empty_like(qc)
        pkg.swa_chunk_fwd(qc, kx, vx, out, B, Hq, Hkv, C, L, d, W, scale)
        got[:, :, pos0:pos0 + C] = out
        pos = torch.full((B,), pos0, dtype=torch.int32, device="cuda")
        pkg.swa_cache_append(tk[:, :, pos0:pos0 + C].contiguous(),
                             tv[:, :, pos0:pos0 + C].contiguous(), kc, vc, pos, B, Hkv, W, d, C)
        pos0 += C
    assert pos0 == T
    torch.cuda.synchronize()
    assert pkg.swa_device_status() == 0
    _check(got.float().cpu().numpy().astype(np.float64), ref, "rolling chunked prefill")


def test_chunk_equal_to_whole_is_swa_bitwise():
    B, Hq, Hkv, N, d, W = 1, 4, 2, 640, 128, 200
    rng = np.random.default_rng(12)
    t = [to_dev(_rand(rng, (B, h, N, d))) for h in (Hq, Hkv, Hkv)]
    a = torch.empty_like(t[0])
    b = torch.empty_like(t[0])
    pkg.swa_chunk_fwd(t[0], t[1], t[2], a, B, Hq, Hkv, N, N, d, W, 0.1)
    pkg.swa_attn_fwd(t[0], t[1], t[2], b, B, Hq, Hkv, N, d, W, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))

"""GPU parity of the decode step against a rolling W-slot KV cache (the SWA note's cache
section): the sm_103a kernels, called through the C ABI, against the fp64 oracle on the
same seeded bf16 inputs, |gpu - oracle| <= 1.5e-2 + 1e-2 |oracle|."""
import numpy as np
import pytest
import torch

import oracle
import swa_inputs
from swa_inputs import Workload, f32_to_bf16_bits, bf16_bits_to_f64
import sparse_causal_attention_swa_b300 as pkg
from gpu_util import ATOL, RTOL, to_dev

pytestmark = pytest.mark.gpu

NAN_BF16 = 0x7FC0


def _decode_gpu(q, kc, vc, pos, W, scale):
    """q, kc, vc: bf16 bit arrays; pos: int array.  Returns fp64 [B, Hq, d]."""
    B, Hq, d = q.shape
    Hkv = kc.shape[1]
    tq, tk, tv = to_dev(q), to_dev(kc), to_dev(vc)
    tp = torch.as_tensor(np.asarray(pos, dtype=np.int32), device="cuda")
    out = torch.full_like(tq, float("nan"))
    nbytes = pkg.swa_decode_workspace_bytes(B, Hq, W, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    pkg.swa_decode_fwd(tq, tk, tv, tp, out, B, Hq, Hkv, W, d, scale, ws, nbytes)
    torch.cuda.synchronize()
    assert pkg.swa_device_status() == 0
    return out.float().cpu().numpy().astype(np.float64)


def _check(got, ref, label):
    assert np.all(np.isfinite(got)), f"{label}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{label}: {int(bad.sum())} out of tolerance, max err {err.max():.3e}"
    return float(err.max())


def _random_case(B, Hq, Hkv, W, d, pos, seed):
    rng = np.random.default_rng(seed)
    q = f32_to_bf16_bits(rng.standard_normal((B, Hq, d), dtype=np.float32))
    kc = f32_to_bf16_bits(rng.standard_normal((B, Hkv, W, d), dtype=np.float32))
    vc = f32_to_bf16_bits(rng.standard_normal((B, Hkv, W, d), dtype=np.float32))
    # slots outside a sequence's window were never written: fill them with NaN, which a
    # read of them would carry into the output
    for b, t in enumerate(pos):
        if t + 1 < W:
            kc[b, :, t + 1:] = NAN_BF16
            vc[b, :, t + 1:] = NAN_BF16
    return q, kc, vc


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("heads", [(1, 1), (2, 1), (4, 1), (8, 2), (6, 2), (7, 1), (8, 1), (16, 1),
                                   (32, 8), (3, 3)])
def test_decode_sweep(d, heads):
    """Every query-head group size the kernels are built for (1, 2, 4, 8, 16, padded from 3,
    6, 7); W from one slot to nine splits of 128 (the combine takes the splits eight at a
    time), ragged last splits included."""
    Hq, Hkv = heads
    for W in (1, 7, 128, 129, 300, 1100):
        pos = [0, max(0, W - 2), W - 1, W, 5 * W + 3]
        q, kc, vc = _random_case(len(pos), Hq, Hkv, W, d, pos, seed=W * 31 + Hq + d)
        scale = 1.0 / np.sqrt(d)
        got = _decode_gpu(q, kc, vc, pos, W, scale)
        ref = oracle.decode(q, kc, vc, pos, W, scale)
        _check(got, ref, f"W={W} d={d} heads={heads}")


def test_rolling_append_then_decode_matches_window_rows():
    """A whole generated sequence: every step appends its K, V to the rolling caches and
    decodes its query; each output must equal that row of windowed attention over the
    whole sequence."""
    B, Hq, Hkv, T, d, W = 2, 4, 2, 300, 64, 64
    rng = np.random.default_rng(7)
    q = f32_to_bf16_bits(rng.standard_normal((B, Hq, T, d), dtype=np.float32))
    k = f32_to_bf16_bits(rng.standard_normal((B, Hkv, T, d), dtype=np.float32))
    v = f32_to_bf16_bits(rng.standard_normal((B, Hkv, T, d), dtype=np.float32))
    scale = 0.125
    ref = oracle.attn(q, k, v, W, scale, kind="window")
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    kc = torch.full((B, Hkv, W, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    nbytes = pkg.swa_decode_workspace_bytes(B, Hq, W, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((T, B, Hq, d), dtype=torch.bfloat16, device="cuda")
    for t in range(T):
        pos = torch.full((B,), t, dtype=torch.int32, device="cuda")
        kn = tk[:, :, t].contiguous()
        vn = tv[:, :, t].contiguous()
        pkg.swa_cache_append(kn, vn, kc, vc, pos, B, Hkv, W, d)
        qt = tq[:, :, t].contiguous()
        pkg.swa_decode_fwd(qt, kc, vc, pos, out[t], B, Hq, Hkv, W, d, scale, ws, nbytes)
    torch.cuda.synchronize()
    assert pkg.swa_device_status() == 0
    got = out.float().cpu().numpy().astype(np.float64).transpose(1, 2, 0, 3)
    _check(got, ref, "rolling")


def test_full_size_workload():
    w = swa_inputs.WORKLOADS["mistral_decode"]
    inp = swa_inputs.make_inputs(w)
    got = _decode_gpu(inp["q"], inp["kc"], inp["vc"], inp["pos"], w.W, w.scale)
    ref = oracle.decode(inp["q"], inp["kc"], inp["vc"], inp["pos"], w.W, w.scale)
    err = _check(got, ref, "mistral_decode")
    print(f"mistral_decode: all {w.B * w.Hq} rows checked, max err {err:.3e}")


def test_negative_position_gives_zero_and_w1_gives_v():
    B, Hq, Hkv, W, d = 2, 4, 2, 1, 128
    q, kc, vc = _random_case(B, Hq, Hkv, W, d, [10, 3], seed=3)
    got = _decode_gpu(q, kc, vc, [10, 3], W, 0.1)
    v = bf16_bits_to_f64(vc)[:, :, 0]
    assert np.array_equal(got, np.repeat(v, Hq // Hkv, axis=1))
    got = _decode_gpu(q, kc, vc, [-1, 3], W, 0.1)
    assert np.all(got[0] == 0)


def test_workspace_too_small_is_rejected_and_deterministic():
    B, Hq, Hkv, W, d = 2, 8, 2, 1000, 128
    q, kc, vc = _random_case(B, Hq, Hkv, W, d, [999, 5000], seed=4)
    tq, tk, tv = to_dev(q), to_dev(kc), to_dev(vc)
    tp = torch.tensor([999, 5000], dtype=torch.int32, device="cuda")
    out = torch.empty_like(tq)
    nbytes = pkg.swa_decode_workspace_bytes(B, Hq, W, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkg.SwaError):
        pkg.swa_decode_fwd(tq, tk, tv, tp, out, B, Hq, Hkv, W, d, 0.1, ws, nbytes - 1)
    outs = []
    for _ in range(2):
        pkg.swa_decode_fwd(tq, tk, tv, tp, out, B, Hq, Hkv, W, d, 0.1, ws, nbytes)
        torch.cuda.synchronize()
        outs.append(out.clone())
    assert torch.equal(outs[0], outs[1])


def test_cache_append_slot_near_int_max_and_long_blocks():
    """Slots come from 64-bit arithmetic: rows at positions past 2^31 - 1 land in the slot
    the oracle's slot map gives.  Blocks and contexts longer than 65535 rows (more rows than a
    grid's y extent) are copied whole."""
    B, Hkv, d = 2, 3, 64
    W, n = 7, 4
    rng = np.random.default_rng(11)
    kn = f32_to_bf16_bits(rng.standard_normal((B, Hkv, n, d), dtype=np.float32))
    vn = f32_to_bf16_bits(rng.standard_normal((B, Hkv, n, d), dtype=np.float32))
    pos = np.array([2**31 - 2, 5], dtype=np.int32)
    kc = torch.zeros((B, Hkv, W, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    tp = torch.as_tensor(pos, device="cuda")
    pkg.swa_cache_append(to_dev(kn), to_dev(vn), kc, vc, tp, B, Hkv, W, d, n)
    torch.cuda.synchronize()
    kcb = kc.view(torch.int16).cpu().numpy().view(np.uint16)
    vcb = vc.view(torch.int16).cpu().numpy().view(np.uint16)
    for b in range(B):
        for r in range(n):
            slot = oracle.cache_slot(int(pos[b]) + r, W)
            assert np.array_equal(kcb[b, :, slot], kn[b, :, r])
            assert np.array_equal(vcb[b, :, slot], vn[b, :, r])

    # a block of 70000 rows into a cache of the same length, then gathered back
    B, Hkv, W = 1, 2, 70000
    n = W
    kn = f32_to_bf16_bits(rng.standard_normal((B, Hkv, n, d), dtype=np.float32))
    vn = f32_to_bf16_bits(rng.standard_normal((B, Hkv, n, d), dtype=np.float32))
    kc = torch.zeros((B, Hkv, W, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    p0 = 123
    tp = torch.tensor([p0], dtype=torch.int32, device="cuda")
    pkg.swa_cache_append(to_dev(kn), to_dev(vn), kc, vc, tp, B, Hkv, W, d, n)
    kx = torch.zeros((B, Hkv, n, d), dtype=torch.bfloat16, device="cuda")
    vx = torch.zeros_like(kx)
    pkg.swa_cache_gather(kc, vc, kx, vx, B, Hkv, W, d, p0 + n, n, n)
    torch.cuda.synchronize()
    assert pkg.swa_device_status() == 0
    assert np.array_equal(kx.view(torch.int16).cpu().numpy().view(np.uint16), kn)
    assert np.array_equal(vx.view(torch.int16).cpu().numpy().view(np.uint16), vn)

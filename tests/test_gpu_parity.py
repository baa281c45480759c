"""GPU parity: the sm_103a kernels, called through the C ABI, against the fp64 oracle on
the same seeded bf16 inputs.  Tolerances: |gpu - oracle| <= 1.5e-2 + 1e-2 |oracle| for
causal SWA and local+strided, |gpu - oracle| <= 3e-2 for differential attention."""
import numpy as np
import pytest
import torch

import swa_inputs
from swa_inputs import Workload
import sparse_causal_attention_swa_b300 as pkg
from gpu_util import assert_close, canary_intact, run_gpu, run_oracle, to_dev, to_f64, out_like

pytestmark = pytest.mark.gpu

HEADS = [(1, 1), (2, 1), (3, 3), (4, 2), (6, 2), (8, 2)]


def _w(kind, B, Hq, Hkv, N, d, W, stride=0, lam=0.0, seed=0):
    return Workload(f"t_{kind}", kind, B, Hq, Hkv, N, d, W, stride=stride, lam=lam,
                    seed_index=1000 + seed)


def check(w, rows=None, label=""):
    inp = swa_inputs.make_inputs(w)
    got = run_gpu(w, inp)
    ref = run_oracle(w, inp, rows=rows)
    if rows is not None:
        got = got[:, :, rows]
    return assert_close(w, got, ref, label or f"{w}")


# ------------------------------------------------------------------------- causal SWA
def test_small_config_full():
    w = swa_inputs.WORKLOADS["swa_small"]
    err = check(w, label="swa_small")
    print(f"swa_small max err {err:.3e}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("heads", HEADS)
def test_window_sweep(d, heads):
    Hq, Hkv = heads
    for N in (1, 17, 128, 129, 255, 300, 513):
        for W in sorted({1, 2, 63, 64, 65, 127, 128, 129, max(1, N - 1), N, 2 * N}):
            check(_w("swa", 1, Hq, Hkv, N, d, W, seed=N * 7 + W), label=f"N={N} W={W} d={d} {heads}")


def test_batch_and_many_heads():
    check(_w("swa", 3, 8, 4, 700, 128, 200, seed=5))
    check(_w("swa", 2, 9, 3, 640, 64, 77, seed=6))


def test_w1_returns_v_bit_exact():
    for Hq, Hkv, d in ((2, 2, 64), (8, 2, 128), (3, 1, 128)):
        w = _w("swa", 2, Hq, Hkv, 389, d, 1, seed=11)
        inp = swa_inputs.make_inputs(w)
        got = run_gpu(w, inp)
        v = swa_inputs.bf16_bits_to_f64(inp["v"])
        expect = np.repeat(v, Hq // Hkv, axis=1)
        assert np.array_equal(got, expect)


def test_w_ge_n_bitwise_identical():
    w = _w("swa", 1, 4, 2, 777, 128, 777, seed=12)
    inp = swa_inputs.make_inputs(w)
    a = run_gpu(w, inp)
    for W in (778, 2 * 777, 1 << 30):
        assert np.array_equal(run_gpu(w.replace(W=W), inp), a)


def test_deterministic_and_stream():
    w = _w("swa", 1, 4, 2, 1000, 128, 300, seed=13)
    inp = swa_inputs.make_inputs(w)
    d = {n: to_dev(a) for n, a in inp.items()}
    outs = []
    s = torch.cuda.Stream()
    for _ in range(2):
        out, _ = out_like(d["q"])
        with torch.cuda.stream(s):
            pkg.swa_attn_fwd(d["q"], d["k"], d["v"], out, 1, 4, 2, 1000, 128, 300, w.scale,
                             stream=s)
        s.synchronize()
        outs.append(to_f64(out))
    assert np.array_equal(outs[0], outs[1])


def test_tensor_wrapper_host_roundtrip():
    w = _w("swa", 1, 2, 1, 300, 64, 50, seed=14)
    inp = swa_inputs.make_inputs(w)
    q = torch.from_numpy(inp["q"].view(np.int16)).view(torch.bfloat16)
    k = torch.from_numpy(inp["k"].view(np.int16)).view(torch.bfloat16)
    v = torch.from_numpy(inp["v"].view(np.int16)).view(torch.bfloat16)
    out = pkg.swa_attention(q, k, v, 50)
    assert out.device.type == "cpu"
    assert_close(w, out.float().numpy().astype(np.float64), run_oracle(w, inp), "wrapper")


def _full_size_all_rows(name):
    """Every output element of the workload against the oracle (all rows of all heads)."""
    w = swa_inputs.WORKLOADS[name]
    err = check(w, label=name)
    print(f"{name}: all {w.N} rows x {w.B * w.Hq} heads checked, max err {err:.3e}")


def _full_size(name, n_random=200, boundary_step=1):
    w = swa_inputs.WORKLOADS[name]
    rows = swa_inputs.sample_rows(w.N, n_random, seed=w.seed, tile=128)
    if boundary_step > 1:
        keep = set(range(256)) | set(range(w.N - 128, w.N))
        keep |= {r for r in rows if (r // 128) % boundary_step == 0 or r % 128 not in (0, 127)}
        rows = np.array(sorted(keep), dtype=np.int64)
    err = check(w, rows=rows, label=name)
    print(f"{name}: {rows.size} rows x {w.B * w.Hq} heads checked, max err {err:.3e}")


def test_mistral_full_size_sampled():
    _full_size_all_rows("mistral_swa")


def test_gemma_swa_full_size_sampled():
    _full_size("gemma_swa", n_random=100)


def test_gemma_global_full_size_sampled():
    _full_size("gemma_global", n_random=40, boundary_step=16)


LSE_ATOL, LSE_RTOL = 1e-3, 1e-4  # fp32 log-sum-exp: fp32 scores and sums, approximate exp2


@pytest.mark.parametrize("kind", ["swa", "strided"])
def test_lse_output(kind):
    import oracle

    for (Hq, Hkv, N, d, W, s) in ((4, 2, 300, 128, 77, 16), (3, 1, 513, 64, 200, 7),
                                  (2, 2, 129, 128, 1, 3), (8, 2, 1000, 128, 1000, 128)):
        w = _w(kind, 2, Hq, Hkv, N, d, W, stride=s, seed=N + W)
        inp = swa_inputs.make_inputs(w)
        t = {n: to_dev(a) for n, a in inp.items()}
        out, _ = out_like(t["q"])
        lse = torch.full((w.B, Hq, N), float("nan"), dtype=torch.float32, device="cuda")
        if kind == "swa":
            pkg.swa_attn_fwd_lse(t["q"], t["k"], t["v"], out, lse, w.B, Hq, Hkv, N, d, W, w.scale)
        else:
            pkg.strided_attn_fwd_lse(t["q"], t["k"], t["v"], out, lse, w.B, Hq, Hkv, N, d, W, s,
                                     w.scale)
        torch.cuda.synchronize()
        assert pkg.swa_device_status() == 0
        mk = "window" if kind == "swa" else "strided"
        ref = oracle.lse(inp["q"], inp["k"], W, w.scale, kind=mk, stride=s)
        got = lse.double().cpu().numpy()
        assert np.all(np.isfinite(got))
        err = np.abs(got - ref)
        assert np.all(err <= LSE_ATOL + LSE_RTOL * np.abs(ref)), f"{kind} {N} {W}: {err.max():.3e}"
        # the output matches the call without the log-sum-exp bitwise
        out2, _ = out_like(t["q"])
        if kind == "swa":
            pkg.swa_attn_fwd(t["q"], t["k"], t["v"], out2, w.B, Hq, Hkv, N, d, W, w.scale)
        else:
            pkg.strided_attn_fwd(t["q"], t["k"], t["v"], out2, w.B, Hq, Hkv, N, d, W, s, w.scale)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


# ------------------------------------------------------------------------- local + strided
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("heads", [(1, 1), (4, 2), (3, 1)])
def test_strided_sweep(d, heads):
    Hq, Hkv = heads
    for N in (1, 100, 129, 300, 700):
        for W, s in ((1, 1), (2, 3), (16, 4), (64, 7), (128, 128), (129, 64), (200, 1000),
                     (N, 5), (3, 128), (300, 13)):
            check(_w("strided", 1, Hq, Hkv, N, d, W, stride=s, seed=N + 3 * W + s),
                  label=f"strided N={N} W={W} s={s} d={d} {heads}")


def test_strided_full_size_sampled():
    _full_size_all_rows("strided")


# ------------------------------------------------------------------------- global prefix
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("heads", [(4, 2), (3, 1)])
def test_global_prefix_sweep(d, heads):
    import oracle

    Hq, Hkv = heads
    for N in (100, 300, 700):
        for W, ng in ((16, 0), (16, 1), (128, 16), (200, 129), (64, N), (1, 5), (N, 3)):
            w = _w("swa", 2, Hq, Hkv, N, d, W, seed=N + 7 * W + ng)
            inp = swa_inputs.make_inputs(w)
            t = {n: to_dev(a) for n, a in inp.items()}
            out, buf = out_like(t["q"])
            pkg.global_attn_fwd(t["q"], t["k"], t["v"], out, w.B, Hq, Hkv, N, d, W, ng, w.scale)
            torch.cuda.synchronize()
            assert pkg.swa_device_status() == 0
            assert canary_intact(buf, out.numel())
            ref = oracle.attn(inp["q"], inp["k"], inp["v"], W, w.scale, kind="global", stride=ng)
            assert_close(w, to_f64(out), ref, f"global N={N} W={W} n_g={ng} d={d} {heads}")


# ------------------------------------------------------------------------- differential
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("heads", [(1, 1), (2, 2), (4, 2)])
def test_diff_sweep(d, heads):
    Hq, Hkv = heads
    for N in (1, 60, 128, 200, 513):
        for lam in (0.0, 0.8, 1.0):
            check(_w("diff", 1, Hq, Hkv, N, d, N, lam=lam, seed=N + int(10 * lam)),
                  label=f"diff N={N} lam={lam} d={d} {heads}")


def test_diff_full_size_sampled():
    _full_size_all_rows("diff")


@pytest.mark.parametrize("heads", [(4, 2), (3, 3)])
def test_diff_per_head_lambda(heads):
    import oracle

    Hq, Hkv = heads
    for d, N in ((64, 300), (128, 129)):
        w = _w("diff", 2, Hq, Hkv, N, d, N, lam=0.0, seed=N + d)
        inp = swa_inputs.make_inputs(w)
        lams = np.linspace(-0.5, 1.2, Hq).astype(np.float32)
        t = {n: to_dev(a) for n, a in inp.items()}
        out, buf = out_like(t["q1"])
        lam_dev = torch.from_numpy(lams).cuda()
        pkg.diff_attn_fwd_heads(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], lam_dev, out, w.B,
                                Hq, Hkv, N, d, w.scale)
        torch.cuda.synchronize()
        assert pkg.swa_device_status() == 0
        got = to_f64(out)
        ref = oracle.diff_heads(inp["q1"], inp["k1"], inp["q2"], inp["k2"], inp["v"], lams,
                                w.scale)
        assert_close(w, got, ref, f"per-head lambda {heads} d={d}")
        # a scalar call with every head's lambda equal matches the per-head call bitwise
        lam_dev.fill_(0.8)
        pkg.diff_attn_fwd_heads(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], lam_dev, out, w.B,
                                Hq, Hkv, N, d, w.scale)
        out2, _ = out_like(t["q1"])
        pkg.diff_attn_fwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], 0.8, out2, w.B, Hq, Hkv,
                          N, d, w.scale)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


# ------------------------------------------------------ differential head in an SWA layer
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("heads", [(1, 1), (4, 2), (3, 3)])
def test_diff_window_sweep(d, heads):
    Hq, Hkv = heads
    for N in (1, 60, 200, 513):
        for W in sorted({1, 2, 63, 128, 129, 300, max(1, N - 1)}):
            if W >= N:
                continue
            lam = (0.0, 0.8, 1.0)[(N + W) % 3]
            check(_w("diff", 1, Hq, Hkv, N, d, W, lam=lam, seed=N * 3 + W),
                  label=f"diff N={N} W={W} lam={lam} d={d} {heads}")


def test_diff_window_full_size_sampled():
    _full_size_all_rows("diff_swa")


def test_diff_window_per_head_lambda_and_limits():
    import oracle

    Hq, Hkv, N, d, W = 4, 2, 700, 64, 130
    w = _w("diff", 2, Hq, Hkv, N, d, W, lam=0.0, seed=77)
    inp = swa_inputs.make_inputs(w)
    t = {n: to_dev(a) for n, a in inp.items()}
    lams = np.array([-0.3, 0.0, 0.6, 1.1], dtype=np.float32)
    lam_dev = torch.from_numpy(lams).cuda()
    out, buf = out_like(t["q1"])
    pkg.diff_swa_attn_fwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], 0.0, lam_dev, out, 2, Hq,
                          Hkv, N, d, W, w.scale)
    torch.cuda.synchronize()
    assert pkg.swa_device_status() == 0
    assert canary_intact(buf, out.numel())
    ref = oracle.diff_heads(inp["q1"], inp["k1"], inp["q2"], inp["k2"], inp["v"], lams, w.scale,
                            W=W)
    assert_close(w, to_f64(out), ref, "windowed diff, per-head lambda")
    # W >= N is the causal call, bit for bit (per-head and scalar lambda)
    a, _ = out_like(t["q1"])
    b, _ = out_like(t["q1"])
    pkg.diff_swa_attn_fwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], 0.0, lam_dev, a, 2, Hq, Hkv,
                          N, d, N + 5, w.scale)
    pkg.diff_attn_fwd_heads(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], lam_dev, b, 2, Hq, Hkv, N,
                            d, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    pkg.diff_swa_attn_fwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], 0.8, None, a, 2, Hq, Hkv, N,
                          d, N, w.scale)
    pkg.diff_attn_fwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], 0.8, b, 2, Hq, Hkv, N, d,
                      w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # W = 1: both maps keep only the row's own key, out_i = (1 - lambda) v_i
    pkg.diff_swa_attn_fwd(t["q1"], t["k1"], t["q2"], t["k2"], t["v"], 0.5, None, a, 2, Hq, Hkv, N,
                          d, 1, w.scale)
    torch.cuda.synchronize()
    v = np.repeat(swa_inputs.bf16_bits_to_f64(inp["v"]), Hq // Hkv, axis=1)
    assert np.max(np.abs(to_f64(a) - 0.5 * v)) <= 2.0 ** -8 * np.max(np.abs(v))


# ------------------------------------------------------------------------- watchdog
def test_watchdog_reports_timeout_and_clears():
    assert pkg.swa_device_status() == 0
    pkg.swa_watchdog_selftest(20_000)  # 20 ms bounded wait on a barrier nobody arrives at
    assert pkg.swa_device_status() == 6
    assert pkg.swa_device_status() == 0
    # the context is still usable afterwards
    check(_w("swa", 1, 2, 2, 200, 64, 30, seed=99))

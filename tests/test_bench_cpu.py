"""bench.py's host-side legs that need no GPU: the FLOP and byte accounting and the oracle
legs (CPU baseline and the reference arm) of the backward workload, on a reduced shape."""
import argparse
import io
import json
from contextlib import redirect_stdout

import numpy as np

import bench
import swa_inputs
from sparse_causal_attention_swa_b300 import flops


def _small_bwd():
    return swa_inputs.WORKLOADS["mistral_swa_bwd"].replace(N=300, Hq=4, Hkv=2, d=64, W=64)


def test_bwd_units():
    w = swa_inputs.WORKLOADS["mistral_swa_bwd"]
    fl, by = bench.workload_units(w)
    assert fl == 2.5 * flops.useful_flops("swa", w.B, w.Hq, w.N, w.d, w.W)
    q = w.B * w.Hq * w.N * w.d * 2
    kv = w.B * w.Hkv * w.N * w.d * 2
    assert by == 4 * q + 4 * kv + w.B * w.Hq * w.N * 4
    assert bench.kernel_family(w) == "attn_bwd"
    assert bench.kernel_family(swa_inputs.WORKLOADS["mistral_swa"]) == "attn_fwd"
    assert bench.kernel_family(swa_inputs.WORKLOADS["mistral_decode"]) == "decode"


def test_bwd_inputs():
    w = _small_bwd()
    inp = swa_inputs.make_inputs(w)
    assert set(inp) == {"q", "k", "v", "dout"}
    assert inp["dout"].shape == (1, 4, 300, 64) and inp["k"].shape == (1, 2, 300, 64)


def test_bwd_prefix_is_a_complete_problem():
    import oracle

    w = _small_bwd()
    inp = bench.oracle_inputs_f64(swa_inputs.make_inputs(w))
    sub = bench.bwd_prefix(w, inp, 200)
    assert sub["q"].shape == (1, 4, 200, 64) and sub["k"].shape == (1, 2, 200, 64)
    # the prefix problem's dq equals the full problem's dq on those rows: a query row only
    # sees keys before it
    dq, _, _ = oracle.attn_bwd(sub["q"], sub["k"], sub["v"], sub["dout"], w.W, w.scale)
    dq_full, _, _ = oracle.attn_bwd(inp["q"], inp["k"], inp["v"], inp["dout"], w.W, w.scale)
    np.testing.assert_allclose(dq, dq_full[:, :, :200], rtol=0, atol=1e-12)


def test_bwd_cpu_baseline_and_reference_arm():
    w = _small_bwd()
    cb = bench.cpu_baseline(w, swa_inputs.make_inputs(w), budget_s=0.5)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
    args = argparse.Namespace(steps=2, warmup=3)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.reference_arm(args, w, 1, 0)
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["dtype"] == "f64"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["config"]["kind"] == "bwd"


def test_small_workload_cpu_baseline_has_one_core_time():
    import oracle

    w = swa_inputs.WORKLOADS["swa_small"]
    nt = oracle.max_threads()
    cb = bench.cpu_baseline(w, swa_inputs.make_inputs(w), budget_s=0.5)
    assert cb["value"] > 0 and cb["one_core"]["value"] > 0
    assert oracle.max_threads() == nt  # the thread count is restored


def test_strided_and_diff_bwd_units_inputs_and_oracle_legs():
    ws = swa_inputs.WORKLOADS["strided_bwd"]
    fl, by = bench.workload_units(ws)
    assert fl == 2.5 * flops.useful_flops("strided", ws.B, ws.Hq, ws.N, ws.d, ws.W, ws.stride)
    wd = swa_inputs.WORKLOADS["diff_swa_bwd"]
    fl, by = bench.workload_units(wd)
    assert fl == 2.5 * flops.useful_flops("diff", wd.B, wd.Hq, wd.N, wd.d, wd.W)
    q = wd.B * wd.Hq * wd.N * wd.d * 2
    assert by == 7 * q + 6 * q + 2 * wd.B * wd.Hq * wd.N * 4  # Hq == Hkv here
    assert bench.kernel_family(ws) == bench.kernel_family(wd) == "attn_bwd"
    for w in (ws.replace(N=300, Hq=2, Hkv=2), wd.replace(N=300, Hq=2, Hkv=2)):
        inp = swa_inputs.make_inputs(w)
        assert "dout" in inp and inp["dout"].shape == (1, 2, 300, 64)
        cb = bench.cpu_baseline(w, inp, budget_s=0.3)
        assert cb["kind"] == "oracle" and cb["value"] > 0
        args = argparse.Namespace(steps=2, warmup=3)
        buf = io.StringIO()
        with redirect_stdout(buf):
            bench.reference_arm(args, w, 1, 0)
        line = json.loads(buf.getvalue().strip().splitlines()[-1])
        assert line["impl"] == "reference" and line["value"] > 0 and line["config"]["kind"] == w.kind

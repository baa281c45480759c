"""Helpers for the GPU parity tests: move seeded bf16 inputs to the device, run the C ABI
through the binding, compare with the oracle element by element."""
import numpy as np
import torch

import oracle
import swa_inputs
import sparse_causal_attention_swa_b300 as pkg

ATOL, RTOL = 1.5e-2, 1e-2      # causal SWA and local+strided
DIFF_ATOL = 3e-2               # differential attention


def to_dev(a: np.ndarray, pad: int = 0) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return t.to("cuda")


def out_like(q: torch.Tensor, canary: int = 4096):
    """An output tensor followed by a canary region (bf16 NaN pattern) to catch stray writes."""
    n = q.numel()
    buf = torch.full((n + canary,), float("nan"), dtype=torch.bfloat16, device=q.device)
    buf.view(torch.int16)[n:] = 0x7FC1
    return buf[:n].view(q.shape), buf


def canary_intact(buf: torch.Tensor, n: int) -> bool:
    return bool((buf.view(torch.int16)[n:] == 0x7FC1).all().item())


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def run_gpu(w: swa_inputs.Workload, inp: dict, check_canary: bool = True) -> np.ndarray:
    d = {n: to_dev(a) for n, a in inp.items()}
    first = d["q1"] if w.kind == "diff" else d["q"]
    out, buf = out_like(first)
    if w.kind == "swa":
        pkg.swa_attn_fwd(d["q"], d["k"], d["v"], out, w.B, w.Hq, w.Hkv, w.N, w.d, w.W, w.scale)
    elif w.kind == "strided":
        pkg.strided_attn_fwd(d["q"], d["k"], d["v"], out, w.B, w.Hq, w.Hkv, w.N, w.d, w.W,
                             w.stride, w.scale)
    elif w.W < w.N:
        pkg.diff_swa_attn_fwd(d["q1"], d["k1"], d["q2"], d["k2"], d["v"], w.lam, None, out, w.B,
                              w.Hq, w.Hkv, w.N, w.d, w.W, w.scale)
    else:
        pkg.diff_attn_fwd(d["q1"], d["k1"], d["q2"], d["k2"], d["v"], w.lam, out, w.B, w.Hq,
                          w.Hkv, w.N, w.d, w.scale)
    torch.cuda.synchronize()
    assert pkg.swa_device_status() == 0
    if check_canary:
        assert canary_intact(buf, out.numel()), "write past the end of out"
    return to_f64(out)


def run_oracle(w: swa_inputs.Workload, inp: dict, rows=None) -> np.ndarray:
    if w.kind == "swa":
        return oracle.attn(inp["q"], inp["k"], inp["v"], w.W, w.scale, kind="window", rows=rows)
    if w.kind == "strided":
        return oracle.attn(inp["q"], inp["k"], inp["v"], w.W, w.scale, kind="strided",
                           stride=w.stride, rows=rows)
    return oracle.diff(inp["q1"], inp["k1"], inp["q2"], inp["k2"], inp["v"], w.lam, w.scale,
                       rows=rows, W=w.W if w.W < w.N else 0)


def assert_close(w: swa_inputs.Workload, got: np.ndarray, ref: np.ndarray, label: str = ""):
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{label}: non-finite output"
    err = np.abs(got - ref)
    if w.kind == "diff":
        bad = err > DIFF_ATOL
    else:
        bad = err > ATOL + RTOL * np.abs(ref)
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{label}: {int(bad.sum())} elements out of tolerance; first at "
                             f"{tuple(idx)} gpu={got[tuple(idx)]} ref={ref[tuple(idx)]}; "
                             f"max err {err.max():.3e}")
    return float(err.max())


def check_bound_one(a: np.ndarray, r: np.ndarray, bnd: np.ndarray, label: str) -> float:
    """Element by element: |a - r| <= bnd; returns the worst ratio |a - r| / bnd."""
    assert np.all(np.isfinite(a)), f"{label}: non-finite"
    bad = np.abs(a - r) > bnd
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{label}: {int(bad.sum())} of {a.size} out of tolerance; first "
                             f"at {idx}: gpu={a[idx]} oracle={r[idx]} bound={bnd[idx]:.3e}")
    pos = bnd > 0
    return float(np.max(np.abs(a - r)[pos] / bnd[pos])) if pos.any() else 0.0


def check_bound(got, ref, bounds, label: str) -> dict:
    """dq, dk, dv element by element against per-element bounds; worst ratio per tensor."""
    return {name: check_bound_one(a, r, bnd, f"{label} {name}")
            for name, a, r, bnd in zip(("dq", "dk", "dv"), got, ref, bounds)}

"""The allocation-free strided call.

Some callers cannot call cudaMalloc: code running under an external memory manager or a
pool allocator that forbids foreign device allocations, or a service that must not grow
its device footprint once it is serving.  For them the library offers
strided_attn_fwd_noalloc, which keeps its tile list in one fixed device array instead of
allocating one.  This test calls it through the C ABI twice in a row, on two different
shapes (so the shared array is rewritten between the calls), and checks each result
against the regular strided_attn_fwd: both calls run the same kernel on a tile list with
the same entries, so the outputs must be bit-identical.  The smaller shape is also checked
against the fp64 oracle within the parity tolerance used everywhere else, and a call on a
shape the process has not seen before must leave the device's free memory unchanged.
It lives in its own file, named to be collected last.
"""
import numpy as np
import pytest
import torch

import swa_inputs
from swa_inputs import Workload
import sparse_causal_attention_swa_b300 as pkg
from gpu_util import assert_close, run_oracle, to_dev

pytestmark = pytest.mark.gpu


def _run(fn, w, d):
    out = torch.empty_like(d["q"])
    fn(d["q"], d["k"], d["v"], out, w.B, w.Hq, w.Hkv, w.N, w.d, w.W, w.stride, w.scale)
    torch.cuda.synchronize()
    assert pkg.swa_device_status() == 0
    return out.view(torch.int16).cpu().numpy()


def _f64(bits):
    return swa_inputs.bf16_bits_to_f64(bits.view(np.uint16))


def test_noalloc_matches_regular_call_twice():
    cases = [
        Workload("na1", "strided", 1, 16, 16, 16384, 64, 256, stride=128, seed_index=4),
        Workload("na2", "strided", 2, 4, 2, 3000, 128, 300, stride=7, seed_index=77),
    ]
    for w in cases:
        inp = swa_inputs.make_inputs(w)
        d = {n: to_dev(a) for n, a in inp.items()}
        ref = _run(pkg.strided_attn_fwd, w, d)
        got = _run(pkg.strided_attn_fwd_noalloc, w, d)
        assert np.array_equal(got, ref), f"{w.name}: differs from strided_attn_fwd"
        if w.N <= 4096:
            assert_close(w, _f64(got), run_oracle(w, inp), w.name)


def test_noalloc_fresh_shape_allocates_nothing():
    # same kernel instantiation (d = 64, odd group size) as a first call, so no module code
    # is loaded during the measured call; inputs and output exist before it
    warm = Workload("na3", "strided", 1, 3, 3, 700, 64, 100, stride=9, seed_index=78)
    fresh = Workload("na4", "strided", 1, 3, 3, 1234, 64, 77, stride=13, seed_index=79)
    dw = {n: to_dev(a) for n, a in swa_inputs.make_inputs(warm).items()}
    _run(pkg.strided_attn_fwd_noalloc, warm, dw)
    df = {n: to_dev(a) for n, a in swa_inputs.make_inputs(fresh).items()}
    out = torch.empty_like(df["q"])
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    pkg.strided_attn_fwd_noalloc(df["q"], df["k"], df["v"], out, fresh.B, fresh.Hq, fresh.Hkv,
                                 fresh.N, fresh.d, fresh.W, fresh.stride, fresh.scale)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
    assert pkg.swa_device_status() == 0

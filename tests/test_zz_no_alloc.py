"""The allocation-free strided call.

Some callers cannot call cudaMalloc: code running under an external memory manager or a
pool allocator that forbids foreign device allocations, or a service that must not grow
its device footprint once it is serving.  For them the library offers
strided_attn_fwd_noalloc, which keeps its tile list in one fixed device array instead of
allocating one.  This test calls it through the C ABI twice in a row, on two different
shapes (so the shared array is rewritten between the calls), and checks each result
against the regular strided_attn_fwd within the parity tolerance used everywhere else.
It lives in its own file, named to be collected last.
"""
import numpy as np
import pytest
import torch

import swa_inputs
from swa_inputs import Workload
import sparse_causal_attention_swa_b300 as pkg
from gpu_util import ATOL, RTOL, to_dev

pytestmark = pytest.mark.gpu


def _run(fn, w, d):
    out = torch.empty_like(d["q"])
    fn(d["q"], d["k"], d["v"], out, w.B, w.Hq, w.Hkv, w.N, w.d, w.W, w.stride, w.scale)
    torch.cuda.synchronize()
    assert pkg.swa_device_status() == 0
    return out.float().cpu().numpy().astype(np.float64)


def test_noalloc_matches_regular_call_twice():
    cases = [
        Workload("na1", "strided", 1, 16, 16, 16384, 64, 256, stride=128, seed_index=4),
        Workload("na2", "strided", 2, 4, 2, 3000, 128, 300, stride=7, seed_index=77),
    ]
    for w in cases:
        d = {n: to_dev(a) for n, a in swa_inputs.make_inputs(w).items()}
        ref = _run(pkg.strided_attn_fwd, w, d)
        got = _run(pkg.strided_attn_fwd_noalloc, w, d)
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref)), w.name

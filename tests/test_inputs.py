"""The seeded input module: bf16 rounding and the workload recipe."""
import numpy as np
import torch

import swa_inputs


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(100_000).astype(np.float32),
        # ties and near-ties around the bf16 grid, both signs
        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 1.0 + 2.0 ** -8 + 2.0 ** -20,
                  3.0e38, -0.0, 1e-40], dtype=np.float32),
    ])
    ours = swa_inputs.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = swa_inputs.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_inputs_are_seeded_and_shaped():
    w = swa_inputs.WORKLOADS["swa_small"]
    a = swa_inputs.make_inputs(w)
    b = swa_inputs.make_inputs(w)
    assert set(a) == {"q", "k", "v"}
    for name in a:
        assert a[name].dtype == np.uint16 and np.array_equal(a[name], b[name])
    assert a["q"].shape == (1, 2, 512, 64) and a["k"].shape == (1, 2, 512, 64)
    x = swa_inputs.bf16_bits_to_f32(a["q"])
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 1.0) < 0.02


def test_diff_sink_shift():
    w = swa_inputs.WORKLOADS["diff"].replace(N=64, Hq=2, Hkv=2)
    inp = swa_inputs.make_inputs(w)
    k1 = swa_inputs.bf16_bits_to_f32(inp["k1"])
    assert float(k1[:, :, 0, :].mean()) > 2.0  # key 0 of K1 carries the +3 sink shift
    assert abs(float(k1[:, :, 1:, :].mean())) < 0.2


def test_sample_rows_cover_tiles():
    rows = swa_inputs.sample_rows(1000, 10, seed=1)
    assert rows[0] == 0 and rows[-1] == 999
    for b in (127, 128, 255, 256, 895, 896):
        assert b in rows
    assert np.all(np.diff(rows) > 0)

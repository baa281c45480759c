"""Pins for the fp64 oracle: each test checks it against something other than itself.

Sources: the SWA note ("SWA：滑动窗口注意力与跨层信息传递", §3.1 mask, §3.2 worked
example, §4.1 pair counts), the attention-variants lesson ("注意力变体——滑动窗口、
稀疏、差分", concept figure and "Build it" steps 1-4, FlexAttention predicate in
"Use it") and its Portuguese translation ("Variantes de Atenção", "Atenção
Diferencial" formulas).
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from conftest import golden_path, read_kv_fixture
from sparse_causal_attention_swa_b300 import flops

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------------------------------------
# An independent dense brute force: the mask is built as a full N x N matrix the way the lesson
# describes it (start from -inf, open the allowed keys), and softmax(Q K^T * scale + M) V is
# evaluated with numpy in fp64.  No code is shared with the C oracle.
# ---------------------------------------------------------------------------------------------
def dense_mask(n, kind, window=0, stride=0):
    M = np.full((n, n), -np.inf)
    for i in range(n):
        if kind == "causal":
            M[i, : i + 1] = 0.0
            continue
        M[i, max(0, i - window + 1): i + 1] = 0.0
        if kind == "strided":
            M[i, np.arange(0, i + 1, stride)] = 0.0
    return M


def dense_softmax(Q, K, scale, M):
    S = Q @ K.T * scale + M
    S = S - S.max(axis=1, keepdims=True)
    P = np.exp(S)
    return P / P.sum(axis=1, keepdims=True)


def dense_attn(q, k, v, scale, kind, window=0, stride=0):
    B, Hq, N, d = q.shape
    g = Hq // k.shape[1]
    M = dense_mask(N, kind, window, stride)
    out = np.empty_like(q)
    for b in range(B):
        for h in range(Hq):
            A = dense_softmax(q[b, h], k[b, h // g], scale, M)
            out[b, h] = A @ v[b, h // g]
    return out


def rand(rng, *shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------------------------------------
# Worked example (SWA note §3.2) and pair counts (§4.1)
# ---------------------------------------------------------------------------------------------
def _frac(s):
    return float(Fraction(s))


def _worked_inputs(v_key):
    fx = read_kv_fixture("swa_note_worked_example.txt")
    kv = {"0": 0.0, "ln2": math.log(2.0), "ln3": math.log(3.0)}
    k = np.array([kv[t] for t in fx["k"].split()], dtype=np.float64)
    v = np.array([float(t) for t in fx[v_key].split()], dtype=np.float64)
    q = np.zeros(5)
    q[4] = float(fx["q5"])
    return fx, q.reshape(1, 1, 5, 1), k.reshape(1, 1, 5, 1), v.reshape(1, 1, 5, 1)


@pytest.mark.parametrize("v_key", ["v_split_a", "v_split_b"])
def test_worked_example_window_and_full(oracle_mod, v_key):
    fx, q, k, v = _worked_inputs(v_key)
    W = int(fx["W"])
    out_w = oracle_mod.attn(q, k, v, W, 1.0, kind="window")[0, 0, 4, 0]
    assert abs(out_w - _frac(fx["out_window"])) < 1e-14
    for W_full in (5, 6, 100):
        out_f = oracle_mod.attn(q, k, v, W_full, 1.0, kind="window")[0, 0, 4, 0]
        assert abs(out_f - _frac(fx["out_full"])) < 1e-14
    out_c = oracle_mod.attn(q, k, v, 0, 1.0, kind="causal")[0, 0, 4, 0]
    assert abs(out_c - _frac(fx["out_full"])) < 1e-14


def test_worked_example_weights(oracle_mod):
    fx, q, k, _ = _worked_inputs("v_split_a")
    w = oracle_mod.weights_row(q, k, int(fx["W"]), 1.0, 0, 0, 4, kind="window")
    expect = [0.0, 0.0] + [_frac(t) for t in fx["weights_window"].split()]
    np.testing.assert_allclose(w, expect, rtol=0, atol=1e-15)


def test_pair_counts_worked_example(oracle_mod):
    fx = read_kv_fixture("swa_note_worked_example.txt")
    assert oracle_mod.pair_count(5, 3, "window") == int(fx["pairs_window"])
    assert oracle_mod.pair_count(5, 0, "causal") == int(fx["pairs_full"])
    assert flops.pairs_window(5, 3) == int(fx["pairs_window"])
    assert flops.pairs_causal(5) == int(fx["pairs_full"])


@pytest.mark.parametrize("N,W", [(1, 1), (7, 1), (64, 63), (64, 64), (64, 65), (100, 7),
                                 (8192, 1024), (1000, 999), (513, 64)])
def test_pair_count_closed_form(oracle_mod, N, W):
    # SWA note §4.1: sum_i min(i, W) = T W - W (W - 1) / 2 for T >= W
    assert oracle_mod.pair_count(N, W, "window") == flops.pairs_window(N, W)


def test_pages_8192_1024_figure(oracle_mod):
    # The lesson's "about 1024 x 8192 entries" is the rounded form of the exact count.
    n = oracle_mod.pair_count(8192, 1024, "window")
    assert n == 8192 * 1024 - 1024 * 1023 // 2 == 7_864_832
    assert abs(n / (1024 * 8192) - 1) < 0.07


# ---------------------------------------------------------------------------------------------
# Mask convention: the window figure, the FlexAttention predicate, W >= N, W = 1
# ---------------------------------------------------------------------------------------------
def _read_figure():
    sections, cur = {}, None
    with open(golden_path("av_window_figure.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                cur = line.strip("[]").split()[0]
                sections[cur] = {}
                continue
            row, keys = line.split(":")
            sections[cur][int(row)] = [int(t) for t in keys.split()]
    return sections


def test_window_figure(oracle_mod):
    fig = _read_figure()
    for i, keys in fig["sliding_window"].items():
        assert np.flatnonzero(oracle_mod.mask_row(8, 4, i, "window")).tolist() == keys
    for i, keys in fig["full_causal"].items():
        assert np.flatnonzero(oracle_mod.mask_row(8, 0, i, "causal")).tolist() == keys


@pytest.mark.parametrize("N,W", [(8, 4), (50, 1), (50, 7), (50, 50), (50, 80)])
def test_flex_predicate(oracle_mod, N, W):
    # FlexAttention mask function of the lesson's "Use it": (q - kv < W) & (q >= kv)
    for i in range(N):
        pred = np.array([(i - j < W) and (i >= j) for j in range(N)])
        assert (oracle_mod.mask_row(N, W, i, "window") == pred).all()


def test_window_does_not_wrap(oracle_mod):
    # SWA note §1: at the start of the sequence the window uses the positions that exist
    for i in range(5):
        assert np.flatnonzero(oracle_mod.mask_row(10, 5, i, "window")).tolist() == list(range(i + 1))


def test_w_ge_n_is_full_causal_bitwise(oracle_mod):
    rng = np.random.default_rng(1)
    q, k, v = rand(rng, 1, 2, 37, 8), rand(rng, 1, 2, 37, 8), rand(rng, 1, 2, 37, 8)
    ref = oracle_mod.attn(q, k, v, 0, 0.3, kind="causal")
    for W in (37, 38, 74, 1 << 30):
        out = oracle_mod.attn(q, k, v, W, 0.3, kind="window")
        assert np.array_equal(out, ref)


def test_w1_returns_v(oracle_mod):
    rng = np.random.default_rng(2)
    q, k, v = rand(rng, 2, 3, 19, 5), rand(rng, 2, 3, 19, 5), rand(rng, 2, 3, 19, 5)
    out = oracle_mod.attn(q, k, v, 1, 0.7, kind="window")
    assert np.array_equal(out, v)


def test_rows_sum_to_one(oracle_mod):
    rng = np.random.default_rng(3)
    q, k = rand(rng, 1, 1, 64, 16), rand(rng, 1, 1, 64, 16)
    for kind, W, s in (("window", 9, 0), ("strided", 5, 4), ("causal", 0, 0)):
        for i in range(64):
            w = oracle_mod.weights_row(q, k, W, 0.25, 0, 0, i, kind=kind, stride=s)
            assert abs(w.sum() - 1.0) < 1e-12
            assert (w[i + 1:] == 0).all() and (w >= 0).all()


def test_uniform_keys_give_window_mean(oracle_mod):
    # Equal scores make the softmax uniform over the allowed keys: out_i = mean of v over the window.
    rng = np.random.default_rng(4)
    N, W = 40, 6
    q, v = rand(rng, 1, 1, N, 4), rand(rng, 1, 1, N, 4)
    k = np.zeros((1, 1, N, 4))
    out = oracle_mod.attn(q, k, v, W, 1.0, kind="window")[0, 0]
    for i in range(N):
        lo = max(0, i - W + 1)
        np.testing.assert_allclose(out[i], v[0, 0, lo: i + 1].mean(axis=0), rtol=0, atol=1e-14)


def test_large_scores_pick_argmax(oracle_mod):
    # Scores far apart make the softmax one-hot at the row maximum; an exp without the max
    # subtraction would overflow to inf/nan here.
    N, d = 12, 1
    q = np.ones((1, 1, N, d))
    k = np.arange(N, dtype=np.float64).reshape(1, 1, N, d) * 1000.0
    v = np.arange(N, dtype=np.float64).reshape(1, 1, N, d) + 0.5
    out = oracle_mod.attn(q, k, v, 4, 1.0, kind="window")[0, 0, :, 0]
    np.testing.assert_array_equal(out, np.arange(N) + 0.5)  # the newest key always wins


# ---------------------------------------------------------------------------------------------
# Brute force against the dense masked softmax on tiny inputs
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("seed", [10, 11])
@pytest.mark.parametrize("N", [1, 5, 33, 64])
def test_window_brute_force(oracle_mod, seed, N):
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, d = 2, 4, 2, 8
    q, k, v = rand(rng, B, Hq, N, d), rand(rng, B, Hkv, N, d), rand(rng, B, Hkv, N, d)
    for W in range(1, N + 3):
        ref = dense_attn(q, k, v, 0.4, "window", W)
        out = oracle_mod.attn(q, k, v, W, 0.4, kind="window")
        assert np.max(np.abs(out - ref)) < 1e-12, W


@pytest.mark.parametrize("N", [1, 17, 48, 64])
def test_strided_brute_force(oracle_mod, N):
    rng = np.random.default_rng(N)
    q, k, v = rand(rng, 1, 2, N, 8), rand(rng, 1, 2, N, 8), rand(rng, 1, 2, N, 8)
    for W in (1, 2, 5, 16, N, N + 2):
        for s in (1, 2, 3, 7, 16, N, N + 1):
            ref = dense_attn(q, k, v, 0.5, "strided", W, s)
            out = oracle_mod.attn(q, k, v, W, 0.5, kind="strided", stride=s)
            assert np.max(np.abs(out - ref)) < 1e-12, (W, s)


def test_causal_brute_force(oracle_mod):
    rng = np.random.default_rng(5)
    q, k, v = rand(rng, 1, 3, 45, 16), rand(rng, 1, 3, 45, 16), rand(rng, 1, 3, 45, 16)
    assert np.max(np.abs(oracle_mod.attn(q, k, v, 0, 0.25, kind="causal")
                         - dense_attn(q, k, v, 0.25, "causal"))) < 1e-12


def test_strided_special_cases(oracle_mod):
    N = 40
    rng = np.random.default_rng(6)
    q, k, v = rand(rng, 1, 1, N, 4), rand(rng, 1, 1, N, 4), rand(rng, 1, 1, N, 4)
    causal = oracle_mod.attn(q, k, v, 0, 0.5, kind="causal")
    # stride 1 opens every earlier key; a window covering everything does the same
    assert np.array_equal(oracle_mod.attn(q, k, v, 3, 0.5, kind="strided", stride=1), causal)
    assert np.array_equal(oracle_mod.attn(q, k, v, N, 0.5, kind="strided", stride=7), causal)
    # a stride past the end adds only key 0 to the window
    for i in range(N):
        m = oracle_mod.mask_row(N, 3, i, "strided", N)
        expect = oracle_mod.mask_row(N, 3, i, "window")
        expect[0] = True
        assert (m == expect).all()


@pytest.mark.parametrize("N,W,s", [(64, 8, 4), (100, 10, 7), (16384, 256, 128), (300, 300, 5),
                                   (50, 1, 1)])
def test_strided_pair_count_closed_form(oracle_mod, N, W, s):
    assert oracle_mod.pair_count(N, W, "strided", s) == flops.pairs_strided(N, W, s)


def test_strided_headline_pair_count():
    assert flops.pairs_strided(16384, 256, 128) == 5_185_792


# ---------------------------------------------------------------------------------------------
# Differential attention (A1 - lambda A2) V
# ---------------------------------------------------------------------------------------------
def _diff_inputs(seed, B=1, Hq=2, Hkv=2, N=30, d=8):
    rng = np.random.default_rng(seed)
    return (rand(rng, B, Hq, N, d), rand(rng, B, Hkv, N, d), rand(rng, B, Hq, N, d),
            rand(rng, B, Hkv, N, d), rand(rng, B, Hkv, N, d))


def test_diff_lambda_zero_is_causal(oracle_mod):
    q1, k1, q2, k2, v = _diff_inputs(7)
    ref = oracle_mod.attn(q1, k1, v, 0, 0.35, kind="causal")
    np.testing.assert_allclose(oracle_mod.diff(q1, k1, q2, k2, v, 0.0, 0.35), ref, rtol=0, atol=1e-14)


def test_diff_same_maps(oracle_mod):
    q1, k1, _, _, v = _diff_inputs(8)
    ref = oracle_mod.attn(q1, k1, v, 0, 0.35, kind="causal")
    out = oracle_mod.diff(q1, k1, q1, k1, v, 0.8, 0.35)
    np.testing.assert_allclose(out, 0.2 * ref, rtol=0, atol=1e-13)


def test_diff_affine_in_lambda(oracle_mod):
    args = _diff_inputs(9)
    o0 = oracle_mod.diff(*args, 0.0, 0.35)
    o1 = oracle_mod.diff(*args, 1.0, 0.35)
    o8 = oracle_mod.diff(*args, 0.8, 0.35)
    np.testing.assert_allclose(o8, o0 + 0.8 * (o1 - o0), rtol=0, atol=1e-13)


def test_diff_brute_force(oracle_mod):
    q1, k1, q2, k2, v = _diff_inputs(10, B=2, Hq=4, Hkv=2, N=41, d=8)
    N = q1.shape[2]
    M = dense_mask(N, "causal")
    ref = np.empty_like(q1)
    for b in range(2):
        for h in range(4):
            A1 = dense_softmax(q1[b, h], k1[b, h // 2], 0.3, M)
            A2 = dense_softmax(q2[b, h], k2[b, h // 2], 0.3, M)
            ref[b, h] = (A1 - 0.8 * A2) @ v[b, h // 2]
    out = oracle_mod.diff(q1, k1, q2, k2, v, 0.8, 0.3)
    assert np.max(np.abs(out - ref)) < 1e-12


# A differential head inside an SWA layer: both maps under the same window mask.
def test_diff_window_brute_force(oracle_mod):
    q1, k1, q2, k2, v = _diff_inputs(12, B=2, Hq=4, Hkv=2, N=41, d=8)
    N = q1.shape[2]
    for W in (1, 5, 17, 40, 41, 60):
        M = dense_mask(N, "window", window=W)
        ref = np.empty_like(q1)
        for b in range(2):
            for h in range(4):
                A1 = dense_softmax(q1[b, h], k1[b, h // 2], 0.3, M)
                A2 = dense_softmax(q2[b, h], k2[b, h // 2], 0.3, M)
                ref[b, h] = (A1 - 0.8 * A2) @ v[b, h // 2]
        out = oracle_mod.diff(q1, k1, q2, k2, v, 0.8, 0.3, W=W)
        assert np.max(np.abs(out - ref)) < 1e-12, W


def test_diff_window_reductions(oracle_mod):
    q1, k1, q2, k2, v = _diff_inputs(13, N=37)
    N = q1.shape[2]
    for W in (3, 16):
        # lambda = 0: the window attention of the first map alone
        ref = oracle_mod.attn(q1, k1, v, W, 0.35, kind="window")
        out = oracle_mod.diff(q1, k1, q2, k2, v, 0.0, 0.35, W=W)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-14)
        # equal maps: (1 - lambda) times the window attention
        out = oracle_mod.diff(q1, k1, q1, k1, v, 0.8, 0.35, W=W)
        np.testing.assert_allclose(out, 0.2 * ref, rtol=0, atol=1e-13)
    # W = 1: each row keeps only its own key in both maps, out_i = (1 - lambda) v_i
    out = oracle_mod.diff(q1, k1, q2, k2, v, 0.8, 0.35, W=1)
    np.testing.assert_allclose(out, 0.2 * v, rtol=0, atol=1e-15)
    # W >= N is the causal form, bit for bit
    assert np.array_equal(oracle_mod.diff(q1, k1, q2, k2, v, 0.8, 0.35, W=N),
                          oracle_mod.diff(q1, k1, q2, k2, v, 0.8, 0.35))
    assert np.array_equal(oracle_mod.diff(q1, k1, q2, k2, v, 0.8, 0.35, W=5 * N),
                          oracle_mod.diff(q1, k1, q2, k2, v, 0.8, 0.35))
    with pytest.raises(ValueError):
        oracle_mod.diff(q1, k1, q2, k2, v, 0.8, 0.35, W=-1)


# ---------------------------------------------------------------------------------------------
# GQA mapping, row subsets, bf16 inputs
# ---------------------------------------------------------------------------------------------
def test_gqa_equals_repeated_kv(oracle_mod):
    rng = np.random.default_rng(12)
    B, Hq, Hkv, N, d = 2, 6, 2, 23, 4
    q, k, v = rand(rng, B, Hq, N, d), rand(rng, B, Hkv, N, d), rand(rng, B, Hkv, N, d)
    g = Hq // Hkv
    k_rep, v_rep = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)  # head h -> kv head h // g
    for kind, W, s in (("window", 5, 0), ("strided", 4, 3), ("causal", 0, 0)):
        a = oracle_mod.attn(q, k, v, W, 0.5, kind=kind, stride=s)
        b = oracle_mod.attn(q, k_rep, v_rep, W, 0.5, kind=kind, stride=s)
        assert np.array_equal(a, b)


def test_row_subset_matches_full(oracle_mod):
    rng = np.random.default_rng(13)
    q, k, v = rand(rng, 1, 2, 50, 4), rand(rng, 1, 2, 50, 4), rand(rng, 1, 2, 50, 4)
    full = oracle_mod.attn(q, k, v, 7, 0.5)
    rows = np.array([0, 3, 49, 17])
    assert np.array_equal(oracle_mod.attn(q, k, v, 7, 0.5, rows=rows), full[:, :, rows])
    d_full = oracle_mod.diff(q, k, k, q, v, 0.5, 0.5)
    assert np.array_equal(oracle_mod.diff(q, k, k, q, v, 0.5, 0.5, rows=rows), d_full[:, :, rows])


def test_bad_arguments_rejected(oracle_mod):
    q = np.zeros((1, 3, 4, 2))
    k = np.zeros((1, 2, 4, 2))
    with pytest.raises(ValueError):
        oracle_mod.attn(q, k, k, 2, 1.0)  # Hq not a multiple of Hkv
    q = np.zeros((1, 2, 4, 2))
    with pytest.raises(ValueError):
        oracle_mod.attn(q, k, k, 0, 1.0)  # W < 1
    with pytest.raises(ValueError):
        oracle_mod.attn(q, k, k, 2, 1.0, rows=[4])


def test_bf16_inputs_widen_exactly(oracle_mod):
    import swa_inputs

    rng = np.random.default_rng(14)
    x = rng.standard_normal((1, 1, 16, 8)).astype(np.float32)
    h = swa_inputs.f32_to_bf16_bits(x)
    ref = oracle_mod.attn(swa_inputs.bf16_bits_to_f64(h), swa_inputs.bf16_bits_to_f64(h),
                          swa_inputs.bf16_bits_to_f64(h), 3, 0.5)
    assert np.array_equal(oracle_mod.attn(h, h, h, 3, 0.5), ref)


# ------------------------------------------------------------------ decode, rolling cache
def _rolling_fill(kseq, vseq, t, W):
    """Write positions 0..t of a [B, H, T, d] sequence into W-slot caches, in order, the way
    the SWA note's rolling cache does (§4.2): position j goes to slot cache_slot(j, W)."""
    import oracle

    B, H, _, d = kseq.shape
    kc = np.full((B, H, W, d), np.nan)
    vc = np.full((B, H, W, d), np.nan)
    for j in range(t + 1):
        sl = oracle.cache_slot(j, W)
        kc[:, :, sl] = kseq[:, :, j]
        vc[:, :, sl] = vseq[:, :, j]
    return kc, vc


def test_rolling_cache_walkthrough(oracle_mod):
    fx = read_kv_fixture("swa_note_rolling_cache.txt")
    W = int(fx["W"])
    pos1 = [int(x) for x in fx["positions_1indexed"].split()]
    assert [oracle_mod.cache_slot(p - 1, W) for p in pos1] == [int(x) for x in fx["slots"].split()]
    held = {}
    for p in range(1, 5):
        held[oracle_mod.cache_slot(p - 1, W)] = p
    assert [held[s] for s in range(W)] == [int(x) for x in fx["held_after_4"].split()]
    # the window of position 4 is exactly what the cache holds after position 1 was overwritten
    assert sorted(held.values()) == [int(x) for x in fx["window_of_4"].split()]
    assert [int(x) for x in fx["window_of_4"].split()] == [
        j + 1 for j in np.flatnonzero(oracle_mod.mask_row(6, W, 3))]


@pytest.mark.parametrize("W", [1, 3, 7, 16])
def test_decode_equals_window_row(oracle_mod, W):
    rng = np.random.default_rng(40 + W)
    B, Hq, Hkv, T, d = 2, 4, 2, 37, 8
    q = rng.standard_normal((B, Hq, T, d))
    k = rng.standard_normal((B, Hkv, T, d))
    v = rng.standard_normal((B, Hkv, T, d))
    full = oracle_mod.attn(q, k, v, W, 0.35, kind="window")
    for t in (0, 1, W - 1, W, 20, T - 1):
        if t < 0 or t >= T:
            continue
        kc, vc = _rolling_fill(k, v, t, W)
        # slots never written (t < W - 1) hold NaN: the decode must not read them
        kc = np.nan_to_num(kc, nan=1e300) if t >= W - 1 else kc
        got = oracle_mod.decode(q[:, :, t], kc, vc, np.full(B, t), W, 0.35)
        assert np.all(np.isfinite(got))
        np.testing.assert_allclose(got, full[:, :, t], rtol=0, atol=1e-12)


def test_decode_per_sequence_positions(oracle_mod):
    rng = np.random.default_rng(50)
    B, H, W, d = 3, 2, 5, 4
    T = 12
    k = rng.standard_normal((B, H, T, d))
    v = rng.standard_normal((B, H, T, d))
    q = rng.standard_normal((B, H, T, d))
    pos = np.array([2, 11, 6])
    kc = np.empty((B, H, W, d))
    vc = np.empty((B, H, W, d))
    for b in range(B):
        kb, vb = _rolling_fill(k[b:b + 1], v[b:b + 1], int(pos[b]), W)
        kc[b], vc[b] = np.nan_to_num(kb[0]), np.nan_to_num(vb[0])
    got = oracle_mod.decode(q[np.arange(B), :, pos], kc, vc, pos, W, 0.5)
    for b in range(B):
        ref = oracle_mod.attn(q[b:b + 1], k[b:b + 1], v[b:b + 1], W, 0.5, kind="window",
                              rows=[int(pos[b])])
        np.testing.assert_allclose(got[b], ref[0, :, 0], rtol=0, atol=1e-12)


def test_decode_w_beyond_position_is_causal_and_w1_is_v(oracle_mod):
    rng = np.random.default_rng(51)
    B, H, T, d = 1, 2, 9, 6
    q = rng.standard_normal((B, H, T, d))
    k = rng.standard_normal((B, H, T, d))
    v = rng.standard_normal((B, H, T, d))
    t = 5
    W = 16  # larger than the history: every earlier position is in the window
    kc, vc = _rolling_fill(k, v, t, W)
    got = oracle_mod.decode(q[:, :, t], np.nan_to_num(kc), np.nan_to_num(vc), [t], W, 0.4)
    ref = oracle_mod.attn(q, k, v, T, 0.4, kind="causal", rows=[t])
    np.testing.assert_allclose(got, ref[:, :, 0], rtol=0, atol=1e-12)
    kc1, vc1 = _rolling_fill(k, v, t, 1)
    got1 = oracle_mod.decode(q[:, :, t], kc1, vc1, [t], 1, 0.4)
    np.testing.assert_array_equal(got1, v[:, :, t])


def test_decode_gqa_equals_repeated_kv(oracle_mod):
    rng = np.random.default_rng(52)
    B, Hq, Hkv, W, d = 2, 6, 2, 9, 4
    q = rng.standard_normal((B, Hq, d))
    kc = rng.standard_normal((B, Hkv, W, d))
    vc = rng.standard_normal((B, Hkv, W, d))
    pos = np.array([4, 30])
    a = oracle_mod.decode(q, kc, vc, pos, W, 0.3)
    b = oracle_mod.decode(q, np.repeat(kc, 3, axis=1), np.repeat(vc, 3, axis=1), pos, W, 0.3)
    np.testing.assert_array_equal(a, b)


# ------------------------------------------------------------------ per-head lambda
def test_diff_heads_equal_lambdas_is_diff(oracle_mod):
    rng = np.random.default_rng(60)
    B, Hq, Hkv, N, d = 2, 4, 2, 19, 8
    a = [rng.standard_normal((B, Hq if i in (0, 2) else Hkv, N, d)) for i in range(5)]
    ref = oracle_mod.diff(*a, 0.7, 0.3)
    got = oracle_mod.diff_heads(*a, np.full(Hq, 0.7), 0.3)
    np.testing.assert_array_equal(got, ref)


def test_diff_heads_lambda_zero_head_is_causal(oracle_mod):
    rng = np.random.default_rng(61)
    B, Hq, Hkv, N, d = 1, 3, 3, 15, 4
    a = [rng.standard_normal((B, Hq, N, d)) for _ in range(5)]
    got = oracle_mod.diff_heads(*a, np.array([0.0, 0.5, 1.0]), 0.4)
    causal = oracle_mod.attn(a[0], a[1], a[4], N, 0.4, kind="causal")
    np.testing.assert_allclose(got[:, 0], causal[:, 0], rtol=0, atol=1e-12)
    half = oracle_mod.diff(*a, 0.5, 0.4)
    np.testing.assert_array_equal(got[:, 1], half[:, 1])


# ------------------------------------------------------------------ row log-sum-exp
def test_lse_worked_example(oracle_mod):
    # the worked example's window scores exponentiate to 1, 2, 3 (denominator 6); under full
    # causal attention positions 1..3 add 1 each (denominator 8)
    fx, q, k, _ = _worked_inputs("v_split_a")
    assert abs(oracle_mod.lse(q, k, int(fx["W"]), 1.0)[0, 0, 4] - math.log(6.0)) < 1e-14
    assert abs(oracle_mod.lse(q, k, 5, 1.0)[0, 0, 4] - math.log(8.0)) < 1e-14
    assert abs(oracle_mod.lse(q, k, 0, 1.0, kind="causal")[0, 0, 4] - math.log(8.0)) < 1e-14


def test_lse_w1_is_own_score_and_matches_weights(oracle_mod):
    rng = np.random.default_rng(70)
    B, Hq, Hkv, N, d = 1, 4, 2, 23, 8
    q = rng.standard_normal((B, Hq, N, d))
    k = rng.standard_normal((B, Hkv, N, d))
    own = 0.3 * np.einsum("bhnd,bhnd->bhn", q, np.repeat(k, 2, axis=1))
    np.testing.assert_allclose(oracle_mod.lse(q, k, 1, 0.3), own, rtol=0, atol=1e-12)
    # exp(scale q.k_j - lse) are the softmax weights of the row
    for kind, W, s in (("window", 5, 0), ("strided", 3, 4), ("causal", 0, 0)):
        L = oracle_mod.lse(q, k, W, 0.3, kind=kind, stride=s)
        for i in (0, 7, 22):
            w = oracle_mod.weights_row(q, k, W, 0.3, 0, 3, i, kind=kind, stride=s)
            allowed = oracle_mod.mask_row(N, W, i, kind=kind, stride=s)
            z = 0.3 * (np.repeat(k, 2, axis=1)[0, 3] @ q[0, 3, i])
            np.testing.assert_allclose(np.where(allowed, np.exp(z - L[0, 3, i]), 0.0), w,
                                       rtol=0, atol=1e-12)


def test_lse_brute_force(oracle_mod):
    rng = np.random.default_rng(71)
    N, d = 17, 4
    q = rng.standard_normal((1, 1, N, d))
    k = rng.standard_normal((1, 1, N, d))
    for W in (1, 3, 17, 20):
        L = oracle_mod.lse(q, k, W, 0.5)
        for i in range(N):
            lo = max(0, i - W + 1)
            z = 0.5 * (k[0, 0, lo:i + 1] @ q[0, 0, i])
            assert abs(L[0, 0, i] - math.log(np.exp(z).sum())) < 1e-12


# ------------------------------------------------------------------ global prefix tokens
def _dense_global_mask(N, W, ng):
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    return (j <= i) & ((j >= i - W + 1) | (j < ng))


def test_global_special_cases(oracle_mod):
    rng = np.random.default_rng(80)
    B, Hq, Hkv, N, d = 1, 2, 1, 40, 8
    q = rng.standard_normal((B, Hq, N, d))
    k = rng.standard_normal((B, Hkv, N, d))
    v = rng.standard_normal((B, Hkv, N, d))
    win = oracle_mod.attn(q, k, v, 7, 0.3, kind="window")
    np.testing.assert_array_equal(oracle_mod.attn(q, k, v, 7, 0.3, kind="global", stride=0), win)
    causal = oracle_mod.attn(q, k, v, N, 0.3, kind="causal")
    np.testing.assert_array_equal(oracle_mod.attn(q, k, v, 7, 0.3, kind="global", stride=N), causal)
    np.testing.assert_array_equal(oracle_mod.attn(q, k, v, N, 0.3, kind="global", stride=5), causal)
    # one global token = the window plus key 0 = strided with a stride past the sequence
    np.testing.assert_array_equal(oracle_mod.attn(q, k, v, 7, 0.3, kind="global", stride=1),
                                  oracle_mod.attn(q, k, v, 7, 0.3, kind="strided", stride=N))


@pytest.mark.parametrize("N", [1, 9, 33])
def test_global_brute_force_and_pair_count(oracle_mod, N):
    rng = np.random.default_rng(81 + N)
    d = 4
    q = rng.standard_normal((1, 1, N, d))
    k = rng.standard_normal((1, 1, N, d))
    v = rng.standard_normal((1, 1, N, d))
    for W in (1, 3, N, N + 2):
        for ng in (0, 1, 4, N + 1):
            allowed = _dense_global_mask(N, W, ng)
            for i in range(N):
                assert np.array_equal(oracle_mod.mask_row(N, W, i, kind="global", stride=ng),
                                      allowed[i])
            z = 0.5 * q[0, 0] @ k[0, 0].T
            z = np.where(allowed, z, -np.inf)
            a = np.exp(z - z.max(axis=1, keepdims=True))
            a /= a.sum(axis=1, keepdims=True)
            np.testing.assert_allclose(oracle_mod.attn(q, k, v, W, 0.5, kind="global",
                                                       stride=ng)[0, 0], a @ v[0, 0],
                                       rtol=0, atol=1e-12)
            assert oracle_mod.pair_count(N, W, "global", ng) == int(allowed.sum())
            assert flops.pairs_global(N, W, ng) == int(allowed.sum())


# ------------------------------------------------------------------ backward (gradients)
def _bwd_inputs(seed, B=1, Hq=4, Hkv=2, N=13, d=5):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, Hq, N, d)), rng.standard_normal((B, Hkv, N, d)),
            rng.standard_normal((B, Hkv, N, d)), rng.standard_normal((B, Hq, N, d)))


@pytest.mark.parametrize("kind,W,stride", [("window", 4, 0), ("window", 1, 0), ("causal", 0, 0),
                                           ("strided", 3, 4), ("global", 3, 2)])
def test_bwd_matches_central_differences(oracle_mod, kind, W, stride):
    """Every entry of dq, dk, dv against a central difference of L = sum(dout * out) through
    the (separately pinned) forward oracle: the definition of a gradient, not its formula."""
    q, k, v, g = _bwd_inputs(90 + W + stride)
    scale, h = 0.45, 1e-5
    dq, dk, dv = oracle_mod.attn_bwd(q, k, v, g, W, scale, kind=kind, stride=stride)

    def loss(q_, k_, v_):
        return float(np.sum(g * oracle_mod.attn(q_, k_, v_, W, scale, kind=kind, stride=stride)))

    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd[idx] = (loss(**{n + "_": a for n, a in args_p.items()}) -
                       loss(**{n + "_": a for n, a in args_m.items()})) / (2 * h)
        assert np.max(np.abs(fd - grad)) < 1e-7 * max(1.0, np.max(np.abs(grad))), name


def test_bwd_w1_closed_form(oracle_mod):
    # a row that keeps only its own key has a constant softmax: no gradient to q or k, and
    # dv_j is the sum of dout_j over the query heads that read KV head j
    q, k, v, g = _bwd_inputs(95, B=2, Hq=6, Hkv=2, N=9, d=4)
    dq, dk, dv = oracle_mod.attn_bwd(q, k, v, g, 1, 0.7)
    assert np.all(dq == 0.0) and np.all(dk == 0.0)
    expect = g.reshape(2, 2, 3, 9, 4).sum(axis=2)
    np.testing.assert_allclose(dv, expect, rtol=0, atol=1e-14)


def test_bwd_gqa_equals_repeated_kv_and_w_ge_n_is_causal(oracle_mod):
    q, k, v, g = _bwd_inputs(96, Hq=4, Hkv=1, N=11, d=3)
    dq, dk, dv = oracle_mod.attn_bwd(q, k, v, g, 5, 0.6)
    dq_r, dk_r, dv_r = oracle_mod.attn_bwd(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1),
                                           g, 5, 0.6)
    np.testing.assert_allclose(dq, dq_r, rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk, dk_r.sum(axis=1, keepdims=True), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, dv_r.sum(axis=1, keepdims=True), rtol=0, atol=1e-13)
    causal = oracle_mod.attn_bwd(q, k, v, g, 0, 0.6, kind="causal")
    for W in (11, 30):
        for a, b in zip(oracle_mod.attn_bwd(q, k, v, g, W, 0.6), causal):
            assert np.array_equal(a, b)


def test_bwd_row_subsets_partition_the_gradients(oracle_mod):
    """The row-subset form: every row listed is the full form bit for bit; dq of a subset is
    the full dq on its rows and zero elsewhere; the dk, dv of a partition of the rows add up to
    the full dk, dv; a key read only by rows of a subset gets its full gradient from it."""
    q, k, v, g = _bwd_inputs(97, B=2, Hq=4, Hkv=2, N=23, d=6)
    W, sc = 5, 0.4
    full = oracle_mod.attn_bwd(q, k, v, g, W, sc)
    every = oracle_mod.attn_bwd(q, k, v, g, W, sc, rows=np.arange(23))
    for a, b in zip(full, every):
        assert np.array_equal(a, b)
    part_a = np.array([0, 3, 4, 5, 9, 10, 11, 12, 13, 21])
    part_b = np.setdiff1d(np.arange(23), part_a)
    ra = oracle_mod.attn_bwd(q, k, v, g, W, sc, rows=part_a)
    rb = oracle_mod.attn_bwd(q, k, v, g, W, sc, rows=part_b)
    np.testing.assert_array_equal(ra[0][:, :, part_a], full[0][:, :, part_a])
    assert np.all(ra[0][:, :, part_b] == 0.0)
    for x, y, f in zip(ra[1:], rb[1:], full[1:]):
        np.testing.assert_allclose(x + y, f, rtol=0, atol=1e-13)
    # keys 9..13 are read by rows 9..17 only (W = 5): the contiguous subset 9..17 covers them
    sub = oracle_mod.attn_bwd(q, k, v, g, W, sc, rows=np.arange(9, 18))
    for x, f in zip(sub[1:], full[1:]):
        np.testing.assert_allclose(x[:, :, 9:14], f[:, :, 9:14], rtol=0, atol=1e-13)
    with pytest.raises(ValueError):
        oracle_mod.attn_bwd(q, k, v, g, W, sc, rows=np.array([0, 23]))


# ------------------------------------------------------------------ differential gradients
def _diff_bwd_inputs(seed, B=1, Hq=4, Hkv=2, N=11, d=4):
    rng = np.random.default_rng(seed)
    return ([rng.standard_normal((B, h, N, d)) for h in (Hq, Hkv, Hq, Hkv, Hkv)],
            rng.standard_normal((B, Hq, N, d)))


@pytest.mark.parametrize("W", [4, 0])
def test_diff_bwd_matches_central_differences(oracle_mod, W):
    """Every entry of dq1, dk1, dq2, dk2, dv and each head's lambda against a central difference
    of L = sum(dout * out) through the (separately pinned) differential forward."""
    (q1, k1, q2, k2, v), g = _diff_bwd_inputs(120 + W, B=2)
    lams = np.array([0.8, 0.3, -0.2, 1.1])
    scale, h = 0.5, 1e-5
    grads = oracle_mod.diff_bwd(q1, k1, q2, k2, v, lams, g, W, scale)
    args = {"q1": q1, "k1": k1, "q2": q2, "k2": k2, "v": v}

    def loss(a, lm):
        return float(np.sum(g * oracle_mod.diff_heads(a["q1"], a["k1"], a["q2"], a["k2"], a["v"],
                                                      lm, scale, W=W)))

    for name, grad in zip(("q1", "k1", "q2", "k2", "v"), grads[:5]):
        x = args[name]
        fd = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            ap, am = dict(args), dict(args)
            ap[name], am[name] = x.copy(), x.copy()
            ap[name][idx] += h
            am[name][idx] -= h
            fd[idx] = (loss(ap, lams) - loss(am, lams)) / (2 * h)
        assert np.max(np.abs(fd - grad)) < 1e-7 * max(1.0, np.max(np.abs(grad))), name
    fd = np.empty(4)
    for i in range(4):
        lp, lm = lams.copy(), lams.copy()
        lp[i] += h
        lm[i] -= h
        fd[i] = (loss(args, lp) - loss(args, lm)) / (2 * h)
    np.testing.assert_allclose(grads[5], fd, rtol=0, atol=1e-7 * max(1.0, np.abs(fd).max()))


def test_diff_bwd_reductions(oracle_mod):
    (q1, k1, q2, k2, v), g = _diff_bwd_inputs(130, B=2, Hq=6, Hkv=3, N=17, d=5)
    W, sc = 6, 0.4
    # lambda = 0: map 1 is window attention, map 2 gets no gradient
    dq1, dk1, dq2, dk2, dv, dlam = oracle_mod.diff_bwd(q1, k1, q2, k2, v, 0.0, g, W, sc)
    ref = oracle_mod.attn_bwd(q1, k1, v, g, W, sc)
    for a, b in zip((dq1, dk1, dv), ref):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)
    assert np.all(dq2 == 0.0) and np.all(dk2 == 0.0)
    # dlam = -sum_i dout_i . (A2 V)_i
    out2 = oracle_mod.attn(q2, k2, v, W, sc, kind="window")
    np.testing.assert_allclose(dlam, -np.sum(g * out2, axis=(0, 2, 3)), rtol=0, atol=1e-12)
    # equal maps: dq2 = -lambda dq1, dk2 = -lambda dk1, dv = (1 - lambda) x the attention's
    lam = 0.7
    dq1, dk1, dq2, dk2, dv, _ = oracle_mod.diff_bwd(q1, k1, q1, k1, v, lam, g, W, sc)
    np.testing.assert_allclose(dq2, -lam * dq1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk2, -lam * dk1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, (1 - lam) * ref[2], rtol=0, atol=1e-13)

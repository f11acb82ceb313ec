"""Pins for the oracle's attention (CPU only): closed forms, hand-computed values,
invariants.  None of them re-evaluates the oracle's own formula."""

import math
import os

import numpy as np
import pytest

from oracle import attention as oatt
from oracle import quant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_cache(rng, L, Hkv, D, gs=None):
    gs = gs or D
    k = rng.standard_normal((L, Hkv, D)).astype(np.float16)
    v = rng.standard_normal((L, Hkv, D)).astype(np.float16)
    kc, ks = quant.quantize(k, gs)
    vc, vs = quant.quantize(v, gs)
    return quant.dequantize(kc, ks, gs), quant.dequantize(vc, vs, gs)


def test_golden_two_keys_hand_computed():
    rec = {}
    with open(os.path.join(GOLDEN, "attention_two_keys.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *vals = line.split()
                rec[key] = [float(x) for x in vals]
    kh = np.stack([quant.dequantize(np.array(rec[f"kcodes{j}"], np.int8)[None],
                                    np.array(rec[f"kscale{j}"], np.float16)[None], 4)[0]
                   for j in (0, 1)])[:, None, :]
    vh = np.stack([quant.dequantize(np.array(rec[f"vcodes{j}"], np.int8)[None],
                                    np.array(rec[f"vscale{j}"], np.float16)[None], 4)[0]
                   for j in (0, 1)])[:, None, :]
    q = np.array(rec["q"], np.float16)[None]
    o = oatt.decode(q, kh, vh, 2, scale=math.log(rec["scale_ln"][0]))
    assert np.allclose(o[0], rec["o"], rtol=0, atol=1e-14)


def test_context_one_returns_dequantized_v_row_and_gqa_mapping():
    """L = 1: o[h] = V^[0, h // G] exactly, for every head (pins the head mapping)."""
    rng = np.random.default_rng(0)
    H, Hkv, D = 8, 2, 16
    kh, vh = _rand_cache(rng, 1, Hkv, D)
    q = rng.standard_normal((H, D)).astype(np.float16)
    o = oatt.decode(q, kh, vh, 1)
    for h in range(H):
        assert np.array_equal(o[h], vh[0, h // (H // Hkv)])
    assert not np.array_equal(vh[0, 0], vh[0, 1])


def test_identical_keys_return_mean_of_v():
    rng = np.random.default_rng(1)
    L, Hkv, D = 37, 2, 32
    kh, vh = _rand_cache(rng, L, Hkv, D)
    kh[:] = kh[:1]
    q = rng.standard_normal((4, D)).astype(np.float16)
    o = oatt.decode(q, kh, vh, L)
    for h in range(4):
        assert np.allclose(o[h], vh[:, h // 2].mean(axis=0), rtol=0, atol=1e-13)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(2)
    L, D = 50, 8
    kh = np.zeros((L, 1, D))
    vh = rng.standard_normal((L, 1, D))
    q = np.zeros((1, D), np.float16)
    q[0, 0] = 1
    kh[17, 0, 0] = 400.0                          # score 400/sqrt(8) ~ 141 above the others
    o = oatt.decode(q, kh, vh, L)
    assert np.allclose(o[0], vh[17, 0], rtol=0, atol=1e-40 + 1e-15)


def test_permutation_of_key_value_pairs():
    rng = np.random.default_rng(3)
    L, Hkv, D = 90, 2, 16
    kh, vh = _rand_cache(rng, L, Hkv, D)
    q = rng.standard_normal((4, D)).astype(np.float16)
    perm = rng.permutation(L)
    a = oatt.decode(q, kh, vh, L)
    b = oatt.decode(q, kh[perm], vh[perm], L)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("n_splits", [1, 2, 3, 4, 7, 16, 40])
@pytest.mark.parametrize("L,window", [(512, 0), (300, 0), (300, 100), (65, 0), (1, 0)])
def test_split_equals_single_pass(n_splits, L, window):
    """genie-ai-runtime v1.3.0: split-K is exact against the single-block kernel."""
    rng = np.random.default_rng(L + n_splits)
    kh, vh = _rand_cache(rng, L, 2, 32)
    q = rng.standard_normal((8, 32)).astype(np.float16)
    a = oatt.decode(q, kh, vh, L, window=window)
    b = oatt.decode_split(q, kh, vh, L, n_splits, page_size=16, window=window)
    assert np.allclose(a, b, rtol=0, atol=1e-12)


def test_split_bounds_cover_the_range_once():
    for lo, hi, n, ps in [(0, 512, 4, 64), (0, 300, 7, 64), (200, 300, 3, 16), (0, 1, 5, 64),
                          (10, 10, 3, 64), (0, 8192, 128, 64)]:
        b = oatt.split_bounds(lo, hi, n, ps)
        assert len(b) == n
        covered = [j for (a, e) in b for j in range(a, e)]
        assert covered == list(range(lo, hi))
        for (a, e) in b:
            assert a == e or a == lo or a % ps == 0     # splits start on page boundaries


def test_window_keeps_exactly_the_last_w_positions():
    """Window 2 at L = 5: keys 3, 4 only.  Keys 0..2 carry a score 60 above the rest,
    so admitting any of them would move the output far away from mean(V^3, V^4)."""
    D = 4
    kh = np.zeros((5, 1, D))
    kh[:3, 0, 0] = 120.0
    vh = np.zeros((5, 1, D))
    vh[:3, 0] = 100.0
    vh[3, 0] = [1, 2, 3, 4]
    vh[4, 0] = [3, 2, 1, 0]
    q = np.array([[1, 0, 0, 0]], np.float16)
    o = oatt.decode(q, kh, vh, 5, window=2)
    assert np.array_equal(o[0], np.array([2.0, 2.0, 2.0, 2.0]))
    o3 = oatt.decode(q, kh, vh, 5, window=3)       # now key 2 is in: it dominates
    assert np.allclose(o3[0], 100.0)


def test_empty_context_gives_zeros():
    kh = np.zeros((0, 1, 4))
    q = np.ones((2, 4), np.float16)
    assert np.array_equal(oatt.decode(q, kh, kh, 0), np.zeros((2, 4)))


def test_prefill_row_equals_decode_at_its_length_and_is_causal():
    rng = np.random.default_rng(5)
    start, n_new, Hkv, D = 40, 6, 2, 16
    kh, vh = _rand_cache(rng, start + n_new, Hkv, D)
    q = rng.standard_normal((n_new, 4, D)).astype(np.float16)
    o = oatt.prefill_chunk(q, kh, vh, start)
    for i in range(n_new):
        assert np.allclose(o[i], oatt.decode(q[i], kh, vh, start + i + 1), rtol=0, atol=1e-14)
    # a future key with an overwhelming score must not change earlier rows
    kh2, vh2 = kh.copy(), vh.copy()
    kh2[start + n_new - 1] = 1e4
    vh2[start + n_new - 1] = 1e4
    o2 = oatt.prefill_chunk(q, kh2, vh2, start)
    assert np.array_equal(o[:-1], o2[:-1])


def test_combine_skips_empty_splits_and_matches_two_key_closed_form():
    # two splits, one key each: z = 0 and ln 3 -> weights 1/4, 3/4
    v0, v1 = np.array([4.0, 0.0]), np.array([0.0, 8.0])
    parts = [(0.0, 1.0, v0), (-math.inf, 0.0, np.zeros(2)), (math.log(3), 1.0, v1)]
    assert np.allclose(oatt.combine(parts), [1.0, 6.0], rtol=0, atol=1e-15)


def test_default_scale_is_inverse_sqrt_head_dim():
    """head_dim 4, two keys: q.k = 0 and 2, so with the default scale 1/sqrt(4) the
    scores are 0 and 1 and the weights are 1 - sigmoid(1) and sigmoid(1), where
    sigmoid(1) = 0.7310585786300049 (the logistic function at 1)."""
    kh = np.zeros((2, 1, 4))
    kh[1, 0, 0] = 2.0
    vh = np.zeros((2, 1, 4))
    vh[0, 0, 0] = 1.0
    vh[1, 0, 1] = 1.0
    q = np.array([[1, 0, 0, 0]], np.float16)
    o = oatt.decode(q, kh, vh, 2)
    sig1 = 0.7310585786300049
    assert np.allclose(o[0], [1.0 - sig1, sig1, 0.0, 0.0], rtol=0, atol=1e-15)

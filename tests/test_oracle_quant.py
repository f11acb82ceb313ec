"""Pins for the oracle's quantization (CPU only).

The oracle takes its decisions in fp32 (division) and fp16 (scale rounding);
these tests check them against exact arithmetic that shares none of that code:
integer comparisons for the scale, exact fp64 brute force over all 255 codes for
the codes, and hand-computed groups in tests/golden/quant_groups.txt.
"""

import os

import numpy as np
import pytest

from int8_kv_cache_02_gb300 import inputs
from oracle import quant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _all_nonneg_finite_fp16():
    bits = np.arange(0, 0x7C00, dtype=np.uint16)          # +0 .. 65504, monotone in value
    return bits.view(np.float16)


def _all_finite_fp16():
    pos = _all_nonneg_finite_fp16()
    neg = (np.arange(0, 0x7C00, dtype=np.uint16) | np.uint16(0x8000)).view(np.float16)
    return np.concatenate([pos, neg])


def _nearest_fp16_of_ratio(num_units: np.ndarray, den: int) -> np.ndarray:
    """Nearest fp16 to (num_units * 2^-24) / den, ties to the even bit pattern.

    Works in integers: every finite fp16 is an integer multiple of 2^-24.
    """
    vals = _all_nonneg_finite_fp16()
    units = (vals.astype(np.float64) * 2.0 ** 24).astype(np.int64)   # exact
    scaled = units * den                                           # compare den*u with num
    idx = np.searchsorted(scaled, num_units, side="left")
    idx = np.clip(idx, 1, len(units) - 1)
    lo, hi = idx - 1, idx
    dlo = np.abs(num_units - scaled[lo])
    dhi = np.abs(scaled[hi] - num_units)
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    exact = scaled[np.clip(idx, 0, len(units) - 1)] == num_units
    pick = np.where(exact, np.clip(idx, 0, len(units) - 1), pick)
    return vals[pick]


def test_scale_exhaustive_against_exact_rational():
    """s = nearest fp16 to amax/127 (exact rational), for every finite amax >= 0."""
    amax = _all_nonneg_finite_fp16()
    got = quant.group_scales(amax.reshape(-1, 1), 1).reshape(-1)
    num = (amax.astype(np.float64) * 2.0 ** 24).astype(np.int64)
    want = _nearest_fp16_of_ratio(num, 127)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))


def _brute_codes(x16: np.ndarray, s: float) -> np.ndarray:
    """argmin_c |x - c s| over c in [-127, 127], ties to the even c (exact in fp64)."""
    x = x16.astype(np.float64)[:, None]
    c = np.arange(-127, 128, dtype=np.float64)[None, :]
    err = np.abs(x - c * s)          # exact: |x|, c*s and their difference fit in 53 bits
    best = err.min(axis=1, keepdims=True)
    cand = err == best
    even = cand & (np.abs(c.astype(np.int64)) % 2 == 0)
    choose = np.where(even.any(axis=1, keepdims=True), even, cand)
    return (np.argmax(choose, axis=1) - 127).astype(np.int8)


@pytest.mark.parametrize("s", [
    2.0 ** -24, 129 * 2.0 ** -24, 1000 * 2.0 ** -24, 2.0 ** -14, 0.00787353515625,
    0.0131072998046875, 0.333251953125, 1.0, 1.5009765625, 7.875, 127.0, 515.5,
])
def test_codes_exhaustive_against_brute_force(s):
    """Codes of every finite fp16 x under scale s equal the exact nearest code."""
    s16 = np.float16(s)
    assert float(s16) == s
    x = _all_finite_fp16()
    got = quant.quantize_with_scales(x.reshape(-1, 1), np.full((x.size, 1), s16), 1).reshape(-1)
    for lo in range(0, x.size, 8192):
        sl = slice(lo, lo + 8192)
        assert np.array_equal(got[sl], _brute_codes(x[sl], s)), f"s={s} block {lo}"


def test_error_bound_for_normal_scales():
    """|x - c s| <= s/2 whenever the group scale s is a normal fp16."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((4096, 64)) * rng.choice([1e-2, 1.0, 30.0], (4096, 1))).astype(np.float16)
    c, s = quant.quantize(x, 64)
    s64 = s.astype(np.float64)
    normal = s64 >= 2.0 ** -14
    assert normal.all()
    err = np.abs(x.astype(np.float64) - quant.dequantize(c, s, 64))
    assert (err <= s64[:, :1].repeat(64, 1) / 2).all()
    assert c.min() >= -127 and c.max() <= 127


def test_extreme_codes_and_zero_groups():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((512, 256)).astype(np.float16)
    x[5] = 0
    c, s = quant.quantize(x, 64)
    assert (s[5] == 0).all() and (c[5] == 0).all()
    g = np.abs(c.reshape(512, 4, 64)).max(axis=-1)
    assert (g[np.arange(512) != 5] == 127).all()    # the absmax element maps to +-127


def _read_golden_groups():
    recs, cur = [], {}
    with open(os.path.join(GOLDEN, "quant_groups.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            cur[key] = [float(v) for v in vals]
            if key == "c":
                recs.append(cur)
                cur = {}
    return recs


def test_golden_hand_computed_groups():
    recs = _read_golden_groups()
    assert len(recs) == 6
    for r in recs:
        x = np.array(r["x"], np.float64)
        x16 = x.astype(np.float16)
        assert np.array_equal(x16.astype(np.float64), x), "fixture values must be fp16-exact"
        c, s = quant.quantize(x16.reshape(1, -1), x.size)
        assert float(s[0, 0]) == r["s"][0], r
        assert c.reshape(-1).tolist() == [int(v) for v in r["c"]], r


def test_dequantize_exact():
    c = np.array([[-127, -1, 0, 1, 127, 64, -64, 3]], np.int8)
    s = np.array([[0.00787353515625, 2.0 ** -24]], np.float16)
    d = quant.dequantize(c, s, 4)
    want = np.array([-127, -1, 0, 1], np.float64) * 0.00787353515625
    assert np.array_equal(d[0, :4], want)
    assert np.array_equal(d[0, 4:], np.array([127, 64, -64, 3], np.float64) * 2.0 ** -24)


def test_tie_rows_are_rounding_ties():
    """The tie generator's groups get the intended scale, a third of its values are
    exact ties (x / s = k + 1/2), and those round to the even code."""
    x = inputs.tie_rows(64, 256, 64, 7).numpy()
    codes, scales = quant.quantize(x, 64)
    assert np.all(np.abs(x.astype(np.float64)).reshape(64, 4, 64).max(-1) ==
                  127 * scales.astype(np.float64))
    qt = x.astype(np.float32) / scales.astype(np.float32).repeat(64, axis=-1)
    ties = (qt - np.floor(qt)) == np.float32(0.5)
    assert 0.25 < ties.mean() < 0.42
    assert np.all(codes[ties] % 2 == 0)
    assert np.all(np.abs(codes[ties].astype(np.float64) - qt[ties]) == 0.5)

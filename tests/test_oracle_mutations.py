"""The quantization pins catch plausible mistakes planted in the oracle (CPU only).

Each case swaps one numpy routine the oracle's quantizer uses for a wrong one
(round-half-away instead of half-even, truncated scale, asymmetric clamp) and
checks that the exhaustive brute-force pins of test_oracle_quant now fail.
"""

import numpy as np
import pytest

import oracle.quant as q
from tests.test_oracle_quant import (_all_finite_fp16, _all_nonneg_finite_fp16, _brute_codes,
                                     _nearest_fp16_of_ratio)


class _NP:
    """numpy stand-in forwarding everything except the overridden names."""

    def __init__(self, **over):
        self.__dict__.update(over)

    def __getattr__(self, name):
        return getattr(np, name)


def _codes_pin_holds(s):
    x = _all_finite_fp16()
    got = q.quantize_with_scales(x.reshape(-1, 1), np.full((x.size, 1), np.float16(s)), 1).reshape(-1)
    return np.array_equal(got, _brute_codes(x, s))


def _scale_pin_holds():
    amax = _all_nonneg_finite_fp16()
    got = q.group_scales(amax.reshape(-1, 1), 1).reshape(-1)
    want = _nearest_fp16_of_ratio((amax.astype(np.float64) * 2.0 ** 24).astype(np.int64), 127)
    return np.array_equal(got.view(np.uint16), want.view(np.uint16))


def test_pins_hold_unmutated():
    assert _codes_pin_holds(1.0) and _scale_pin_holds()


def test_round_half_away_is_caught(monkeypatch):
    away = lambda r: np.trunc(r + np.copysign(np.float32(0.5), r))  # noqa: E731
    monkeypatch.setattr(q, "np", _NP(rint=away))
    assert not _codes_pin_holds(1.0)


def test_asymmetric_clamp_is_caught(monkeypatch):
    monkeypatch.setattr(q, "QMAX", 128)
    assert not _codes_pin_holds(2.0 ** -24)


def test_truncated_scale_is_caught(monkeypatch):
    real = q.group_scales

    def truncated(x16, gs):
        s = real(x16, gs)
        amax = np.max(np.abs(np.asarray(x16, np.float32)), axis=-1, keepdims=True)  # gs == 1 here
        exact = amax.astype(np.float64) / 127.0
        down = s.astype(np.float64) > exact               # RNE went up: truncation goes down
        bits = s.view(np.uint16).copy()
        bits[down] -= 1
        return bits.view(np.float16)

    monkeypatch.setattr(q, "group_scales", truncated)
    assert not _scale_pin_holds()

"""The oracle's pins catch plausible mistakes planted in the oracle (CPU only).

Quantization: each case swaps one numpy routine the oracle's quantizer uses for
a wrong one (round-half-away instead of half-even, truncated scale, asymmetric
clamp) and checks that the exhaustive brute-force pins of test_oracle_quant
now fail.  Attention: each case replaces one oracle function with a copy that
carries one mistake and checks that a pin of test_oracle_attention fails.
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


# --------------------------------------------------------------------------------------
# Attention: each case plants one plausible mistake in the oracle's attention (a
# dropped term, a wrong sign or index, a transposed operand, a bound off by one)
# and checks that one of the pins of test_oracle_attention now fails.

import functools  # noqa: E402
import math  # noqa: E402

import oracle.attention as oatt  # noqa: E402
from tests import test_oracle_attention as pins  # noqa: E402


def _decode_mutant(q16, khat, vhat, length, window=0, scale=None, *, interleaved=False,
                   lo_shift=0, normalise=True, k_is_v=False, sign=1.0, drop_scale=False):
    """The oracle's decode with one knob turned."""
    q = np.asarray(q16, np.float16).astype(np.float64)
    H, D = q.shape
    Hkv = khat.shape[1]
    G = H // Hkv
    sc = (1.0 if drop_scale else 1.0 / math.sqrt(D)) if scale is None else float(scale)
    lo = max(0, length - window + lo_shift) if window > 0 else 0
    keys = vhat if k_is_v else khat
    out = np.zeros((H, D), np.float64)
    for h in range(H):
        kvh = h % Hkv if interleaved else h // G
        z = sign * sc * (keys[lo:length, kvh, :] @ q[h])
        if z.shape[0] == 0:
            continue
        p = np.exp(z - np.max(z))
        o = p @ vhat[lo:length, kvh, :]
        out[h] = o / np.sum(p) if normalise else o
    return out


def _fails(pin, *args):
    try:
        pin(*args)
    except AssertionError:
        return True
    return False


@pytest.mark.parametrize("knob,pin", [
    (dict(), None),                                        # the unmutated copy passes them all
    (dict(drop_scale=True), pins.test_default_scale_is_inverse_sqrt_head_dim),
    (dict(interleaved=True), pins.test_context_one_returns_dequantized_v_row_and_gqa_mapping),
    (dict(lo_shift=1), pins.test_window_keeps_exactly_the_last_w_positions),
    (dict(lo_shift=-1), pins.test_window_keeps_exactly_the_last_w_positions),
    (dict(normalise=False), pins.test_identical_keys_return_mean_of_v),
    (dict(k_is_v=True), pins.test_dominant_key_selects_its_value),
    (dict(sign=-1.0), pins.test_dominant_key_selects_its_value),
])
def test_decode_mistakes_are_caught(monkeypatch, knob, pin):
    monkeypatch.setattr(oatt, "decode", functools.partial(_decode_mutant, **knob))
    if pin is None:
        for p in (pins.test_default_scale_is_inverse_sqrt_head_dim,
                  pins.test_context_one_returns_dequantized_v_row_and_gqa_mapping,
                  pins.test_window_keeps_exactly_the_last_w_positions,
                  pins.test_identical_keys_return_mean_of_v,
                  pins.test_dominant_key_selects_its_value,
                  pins.test_golden_two_keys_hand_computed):
            p()
    else:
        assert _fails(pin)


def test_combine_without_rescale_is_caught(monkeypatch):
    def combine_no_rescale(partials):
        live = [(m, l, o) for (m, l, o) in partials if l > 0.0]
        M = max(m for m, _, _ in live)
        Lsum = sum(l * math.exp(m - M) for m, l, _ in live)
        return sum(o for _, _, o in live) / Lsum          # o~_s not brought to the common max
    monkeypatch.setattr(oatt, "combine", combine_no_rescale)
    assert _fails(pins.test_combine_skips_empty_splits_and_matches_two_key_closed_form)
    assert _fails(pins.test_split_equals_single_pass, 4, 300, 0)


def test_split_bounds_rounding_down_is_caught(monkeypatch):
    def floor_bounds(lo, hi, n_splits, page_size):
        if hi <= lo:
            return [(lo, lo)] * n_splits
        p0 = lo // page_size
        per = ((hi - 1) // page_size + 1 - p0) // n_splits * page_size   # floor: drops the tail
        return [(max(lo, p0 * page_size + s * per), max(max(lo, p0 * page_size + s * per),
                                                          min(hi, p0 * page_size + (s + 1) * per)))
                for s in range(n_splits)]
    monkeypatch.setattr(oatt, "split_bounds", floor_bounds)
    assert _fails(pins.test_split_bounds_cover_the_range_once)


def test_prefill_without_the_current_position_is_caught(monkeypatch):
    def prefill_short(q16, khat, vhat, start, scale=None):
        q = np.asarray(q16, np.float16).astype(np.float64)
        n_new, H, D = q.shape
        G = H // khat.shape[1]
        sc = 1.0 / math.sqrt(D) if scale is None else float(scale)
        out = np.zeros((n_new, H, D), np.float64)
        for kvh in range(khat.shape[1]):
            heads = slice(kvh * G, (kvh + 1) * G)
            for i in range(n_new):
                n_vis = start + i                               # the query's own key left out
                z = sc * (q[i, heads, :] @ khat[:n_vis, kvh, :].T)
                p = np.exp(z - np.max(z, axis=1, keepdims=True))
                out[i, heads, :] = (p @ vhat[:n_vis, kvh, :]) / np.sum(p, axis=1, keepdims=True)
        return out
    monkeypatch.setattr(oatt, "prefill_chunk", prefill_short)
    assert _fails(pins.test_prefill_row_equals_decode_at_its_length_and_is_causal)


# ---- pool image: a layout mistake planted in the oracle's save must fail a pin
def _image_pins_hold():
    from tests import test_oracle_image as t
    try:
        t.test_image_matches_the_hand_assembled_bytes()
        t.test_sections_are_position_major_with_their_scales()
    except AssertionError:
        return False
    return True


def test_image_pins_hold_unmutated():
    assert _image_pins_hold()


def test_head_major_image_is_caught(monkeypatch):
    import oracle.image as im
    real_rows = im._rows

    def swapped_save(pool, lengths, page_table):
        parts = []
        for b, L in enumerate(int(x) for x in lengths):
            pages, slots = real_rows(pool, page_table[b], L)
            for layer in range(pool.n_layers):
                for _, region, nbytes in im._sections(pool, L):
                    rows = np.ascontiguousarray(region[layer, pages, :, slots, :].swapaxes(0, 1))
                    raw = rows.tobytes()
                    parts.append(raw + bytes(im._pad16(nbytes) - nbytes))
        payload = b"".join(parts)
        lens = np.asarray(lengths, "<i4").tobytes()
        head = im.HEADER.pack(im.MAGIC, im.VERSION, pool.variant, pool.n_layers, pool.n_kv_heads,
                              pool.head_dim, pool.gs, len(lengths), len(payload), 0)
        return head + lens + bytes(im._pad16(len(lens)) - len(lens)) + payload

    monkeypatch.setattr(im, "save", swapped_save)
    assert not _image_pins_hold()


def test_image_without_scales_is_caught(monkeypatch):
    import oracle.image as im
    real = im._sections
    monkeypatch.setattr(im, "_sections", lambda pool, L: real(pool, L)[:2])
    assert not _image_pins_hold()


# ---- 4-bit store: mistakes planted in the oracle's FWHT or Q4_0 must fail a pin
def _q4_pins_hold():
    from tests import test_oracle_q4 as t
    try:
        t.test_q4_0_hand_computed_blocks()
        t.test_fwht_hand_values()
        t.test_fwht_order_of_operations()
    except AssertionError:
        return False
    return True


def test_q4_pins_hold_unmutated():
    assert _q4_pins_hold()


def test_q4_last_largest_value_is_caught(monkeypatch):
    import oracle.q4 as m
    real = np.argmax
    monkeypatch.setattr(m, "np", _NP(argmax=lambda a, axis=None: a.shape[axis] - 1 - real(
        np.flip(a, axis=axis), axis=axis)))
    assert not _q4_pins_hold()


def test_q4_scale_sign_is_caught(monkeypatch):
    """d = m / 8 instead of m / -8: the largest value lands on the clamped end."""
    import oracle.q4 as m

    def plus_eighth(x32):
        x = np.asarray(x32, dtype=np.float32)
        g = x.reshape(x.shape[:-1] + (x.shape[-1] // 32, 32))
        first = np.argmax(np.abs(g), axis=-1)
        mx = np.take_along_axis(g, first[..., None], axis=-1)[..., 0]
        d = mx * np.float32(0.125)
        idv = np.where(d != 0, np.float32(1.0) / np.where(d != 0, d, 1), 0).astype(np.float32)
        t = ((g * idv[..., None]).astype(np.float32) + np.float32(8.5)).astype(np.float32)
        return np.minimum(np.floor(t), 15).astype(np.uint8).reshape(x.shape), d.astype(np.float16)

    monkeypatch.setattr(m, "q4_0_quantize", plus_eighth)
    assert not _q4_pins_hold()


def test_fwht_without_normalisation_is_caught(monkeypatch):
    import oracle.q4 as m
    real = m.fwht
    monkeypatch.setattr(m, "fwht", lambda x: real(x) * np.float32(np.sqrt(np.asarray(x).shape[-1])))
    assert not _q4_pins_hold()


def test_fwht_pairing_mistake_is_caught(monkeypatch):
    import oracle.q4 as m
    real = m.fwht

    def reversed_stages(x):     # the same butterflies, stages taken from the largest stride
        y = np.array(x, dtype=np.float32, copy=True)
        n = y.shape[-1]
        h = n // 2
        while h >= 1:
            v = y.reshape(y.shape[:-1] + (n // (2 * h), 2, h))
            a, b = v[..., 0, :].copy(), v[..., 1, :].copy()
            v[..., 0, :], v[..., 1, :] = a + b, a - b
            h //= 2
        return y * np.float32(1.0 / np.sqrt(n))

    monkeypatch.setattr(m, "fwht", reversed_stages)
    assert not _q4_pins_hold()
    monkeypatch.setattr(m, "fwht", real)

"""Pins for the oracle's 4-bit store (CPU only): the normalised FWHT over a row
and Q4_0 blocks (Strata pull request #2698, "Not in this PR": --kv q4_0 and
k8v4 with the Hadamard rotation over head_dim 256), and the k8v4 pool."""

import os

import numpy as np
import pytest

from oracle import attention as oatt
from oracle import pool as opool
from oracle import q4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q4_0_blocks.txt")


def _records():
    recs, cur = [], {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        tag, _, rest = line.partition(" ")
        if tag == "x" and cur:
            recs.append(cur)
            cur = {}
        cur[tag] = rest.split()
    recs.append(cur)
    return recs


def _sparse(items, default):
    out = np.full(32, default, np.float64)
    for it in items:
        i, v = it.split(":")
        out[int(i)] = float(v)
    return out


def test_q4_0_hand_computed_blocks():
    recs = _records()
    assert len(recs) == 4
    for r in recs:
        x = _sparse(r.get("x", []), 0.0).astype(np.float32)
        codes, d = q4.q4_0_quantize(x[None])
        assert np.float16(float(r["d"][0])).view(np.uint16) == d.view(np.uint16)[0, 0]
        assert codes[0].tolist() == _sparse(r.get("q", []), 8).astype(int).tolist()
        y = q4.q4_0_dequantize(codes, d)[0]
        want = _sparse(r.get("y", []), 0.0)
        assert np.array_equal(y, want), (y[:12], want[:12])


def test_q4_0_error_bound_and_extreme_value():
    """|x - y| <= |d|/2 (+ the fp16 rounding of d) below the clamp, <= |d| at it; the
    block's first largest value comes back within the rounding of d."""
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((4000, 32)) * np.exp(rng.uniform(-8, 8, (4000, 1)))).astype(np.float32)
    codes, d = q4.q4_0_quantize(x)
    y = q4.q4_0_dequantize(codes, d)
    dd = np.abs(d.astype(np.float64))
    err = np.abs(x.astype(np.float64) - y)
    tol_round = np.abs(x.astype(np.float64)) * 2.0 ** -10 + 1e-45
    clamped = codes == 15
    assert np.all(err[~clamped] <= 0.5 * dd.repeat(32, 1)[~clamped] * (1 + 2 ** -9) + tol_round[~clamped])
    assert np.all(err <= dd.repeat(32, 1) * (1 + 2 ** -9) + tol_round)
    first = np.argmax(np.abs(x), axis=1)
    assert np.all(codes[np.arange(4000), first] == 0)


def test_pack_layout_hand_placed():
    """Row of 64 values (2 blocks): byte 4r + 2g + h (chunks of 64/16 = 4 bytes)
    holds values 32g + 4r + 2h (low nibble) and + 1 (high nibble)."""
    c = np.zeros((1, 64), np.uint8)
    c[0, 0], c[0, 1] = 1, 2          # g 0, r 0, h 0 -> byte 0
    c[0, 2], c[0, 3] = 3, 4          # g 0, r 0, h 1 -> byte 1
    c[0, 4] = 5                      # g 0, r 1, h 0 -> byte 4 (low)
    c[0, 33] = 15                    # g 1, r 0, h 0 -> byte 2 (high)
    c[0, 63] = 9                     # g 1, r 7, h 1 -> byte 4*7 + 2 + 1 = 31 (high)
    b = q4.pack(c)[0]
    assert b[0] == 0x21 and b[1] == 0x43 and b[4] == 0x05 and b[2] == 0xF0 and b[31] == 0x90
    assert np.count_nonzero(b) == 5
    rng = np.random.default_rng(1)
    for D in (64, 128, 256):
        r = rng.integers(0, 16, (3, D)).astype(np.uint8)
        assert np.array_equal(q4.unpack(q4.pack(r)), r)
        # every byte of a row is written exactly once
        seen = sorted(q4.byte_of_value(v, D)[0] for v in range(0, D, 2))
        assert seen == list(range(D // 2))


def test_fwht_hand_values():
    assert q4.fwht(np.array([1, 2, 3, 4], np.float32)).tolist() == [5, -1, -2, 0]
    e0 = np.zeros(16, np.float32)
    e0[0] = 1
    assert q4.fwht(e0).tolist() == [0.25] * 16
    e5 = np.zeros(16, np.float32)
    e5[5] = 1                                   # column 5: (-1)^popcount(i & 5) / 4
    assert q4.fwht(e5).tolist() == [0.25 * (-1) ** bin(i & 5).count("1") for i in range(16)]


@pytest.mark.parametrize("n", [2, 8, 64, 256])
def test_fwht_equals_the_hadamard_matrix(n):
    scipy = pytest.importorskip("scipy.linalg")
    rng = np.random.default_rng(n)
    x = rng.standard_normal((5, n)).astype(np.float16).astype(np.float32)
    want = x.astype(np.float64) @ scipy.hadamard(n).T / np.sqrt(n)
    assert np.allclose(q4.fwht(x), want, rtol=0, atol=1e-5 * np.abs(x).max() * np.sqrt(n))
    assert np.allclose(q4.hadamard_fp64(x), want, rtol=0, atol=1e-12 * np.sqrt(n))
    assert np.allclose(q4.fwht(q4.fwht(x)), x, atol=1e-5)


def test_fwht_order_of_operations():
    """The butterflies in the stated order, one fp32 scalar at a time, give the
    same bits (the device kernels follow this order)."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(256) * np.exp(rng.uniform(-6, 6, 256))).astype(np.float16)
    y = [np.float32(v) for v in x]
    h = 1
    while h < 256:
        for i in range(256):
            if i & h == 0:
                a, b = y[i], y[i + h]
                y[i], y[i + h] = np.float32(a + b), np.float32(a - b)
        h *= 2
    y = np.array([np.float32(v * np.float32(0.0625)) for v in y], np.float32)
    assert np.array_equal(q4.fwht(x.astype(np.float32)).view(np.uint32), y.view(np.uint32))


def test_k8v4_pool_context_one_and_identical_keys():
    """k8v4: a single cached position returns its V row as stored (dequantized and
    rotated back); identical keys return the mean of the stored V rows; the V row
    comes back within the Q4_0 error of the rotated row (the rotation keeps L2 norms)."""
    rng = np.random.default_rng(9)
    P = opool.Pool(1, 2, 256, 64, 16, 4, opool.K8V4)
    k = rng.standard_normal((20, 2, 256)).astype(np.float16)
    k[:] = k[0]
    v = rng.standard_normal((20, 2, 256)).astype(np.float16)
    P.append_contiguous(0, k, v, 0, np.arange(2))
    kh, vh = P.gather(0, np.arange(2), 20)
    q = rng.standard_normal((8, 256)).astype(np.float16)
    o1 = oatt.decode(q, kh, vh, 1)
    assert np.allclose(o1, np.repeat(vh[0], 4, axis=0), atol=1e-12)
    o = oatt.decode(q, kh, vh, 20)
    assert np.allclose(o, np.repeat(vh.mean(axis=0), 4, axis=0), atol=1e-12)
    err = np.linalg.norm(vh - v.astype(np.float64), axis=-1) / np.linalg.norm(v.astype(np.float64), axis=-1)
    assert err.max() < 0.15 and err.mean() < 0.12          # 4-bit blocks of 32
    assert P.v_store.shape[-1] == 128 and P.v_scales.shape[-1] == 8
    # thread-chunk layout: chunk r of a row holds values 32g + 4r .. 32g + 4r + 3 of every block
    codes = q4.unpack(P.v_store[0, 0, 0, :1])[0]
    assert codes.shape == (256,)


def test_q4_0_pool_closed_forms_and_rotation_invariance():
    """q4_0: K and V both rotated and 4-bit.  Context 1 returns the stored V row;
    the scores equal those of the rotated query against the rotated, dequantized
    keys (what a kernel computes), because the rotation is orthonormal."""
    rng = np.random.default_rng(12)
    P = opool.Pool(1, 2, 128, 128, 16, 3, opool.Q4_0)
    assert P.k_store.dtype == np.uint8 and P.k_store.shape[-1] == 64 and P.k_scales.shape[-1] == 4
    k = rng.standard_normal((30, 2, 128)).astype(np.float16)
    v = rng.standard_normal((30, 2, 128)).astype(np.float16)
    P.append_contiguous(0, k, v, 0, np.arange(2))
    kh, vh = P.gather(0, np.arange(2), 30)
    q = rng.standard_normal((4, 128)).astype(np.float16)
    assert np.allclose(oatt.decode(q, kh, vh, 1), np.repeat(vh[0], 2, axis=0), atol=1e-12)
    rows = P.k_store[0, 0, 0, :16]                   # kv head 0, positions 0..15
    k_rot = q4.q4_0_dequantize(q4.unpack(rows), P.k_scales[0, 0, 0, :16])
    q_rot = q4.hadamard_fp64(q[0].astype(np.float64))
    assert np.allclose(k_rot @ q_rot, kh[:16, 0] @ q[0].astype(np.float64), atol=1e-9)

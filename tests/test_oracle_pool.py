"""Pins for the oracle's paged pool (CPU only): layout, placement, sizes."""

import numpy as np
import pytest

from oracle import pool as opool
from oracle import quant


def test_bytes_per_cell_matches_strata_figure():
    # Strata pull request #2698, "What it does": 528 B/cell (int8 codes plus one
    # fp16 scale per 64 values) against 2048 B/cell for the fp32 store, head_dim
    # 256, 2 kv heads -- "~3.9x smaller".
    assert opool.bytes_per_cell(2, 256, 64, int8=True) == 528
    assert 2 * 256 * 4 == 2048
    assert abs(2048 / 528 - 3.9) < 0.05
    # per (position, kv head) scales: one 2-byte scale per head_dim codes
    assert opool.bytes_per_cell(8, 128, 128, int8=True) == 8 * 128 + 8 * 2
    assert opool.bytes_per_cell(2, 256, 64, int8=False) == 1024


def test_placement_through_page_table_hand_computed():
    """Position 130 of a sequence with page table [7, 3, 5] lands on physical page 5, slot 2."""
    P = opool.Pool(n_layers=2, n_kv_heads=2, head_dim=8, gs=4, page_size=64, n_pages=8,
                   variant=opool.K8V8)
    k = np.zeros((1, 1, 2, 8), np.float16)
    v = np.zeros((1, 1, 2, 8), np.float16)
    k[0, 0, 1] = [127, 0, 0, 0, 0, 0, 0, 254]       # kv head 1: groups amax 127 and 254
    v[0, 0, 0] = [1, 2, 3, 4, 5, 6, 7, 8]
    P.append(1, k, v, seq_pos=[130], page_table=np.array([[7, 3, 5]]))
    raw = P.k_store.reshape(-1)
    # flat offset of [layer 1][page 5][head 1][slot 2][dim 0] in [2][8][2][64][8]
    off = (((1 * 8 + 5) * 2 + 1) * 64 + 2) * 8
    assert raw[off:off + 8].tolist() == [127, 0, 0, 0, 0, 0, 0, 127]
    assert np.count_nonzero(P.k_store) == 2
    sc = P.k_scales.reshape(-1)
    soff = (((1 * 8 + 5) * 2 + 1) * 64 + 2) * 2
    assert sc[soff:soff + 2].astype(np.float64).tolist() == [1.0, 2.0]
    # V head 0, groups amax 4 and 8 -> scales fp16(4/127), fp16(8/127)
    voff = (((1 * 8 + 5) * 2 + 0) * 64 + 2) * 8
    assert P.v_store.reshape(-1)[voff + 3] == 127 and P.v_store.reshape(-1)[voff + 7] == 127


@pytest.mark.parametrize("variant", [opool.K8V8, opool.K8V16, opool.K16V8])
def test_paged_equals_contiguous_and_loop_equals_vectorised(variant):
    rng = np.random.default_rng(11)
    L, Hkv, D, gs, ps = 200, 2, 64, 32, 16
    k = rng.standard_normal((L, Hkv, D)).astype(np.float16)
    v = rng.standard_normal((L, Hkv, D)).astype(np.float16)
    n = -(-L // ps)
    shuffled = rng.permutation(20)[:n]
    A = opool.Pool(1, Hkv, D, gs, ps, 20, variant)
    A.append_contiguous(0, k, v, 0, shuffled)
    B = opool.Pool(1, Hkv, D, gs, ps, n, variant)
    B.append(0, k[None], v[None], [0], np.arange(n)[None])      # per-token loop, identity pages
    ka, va = A.gather(0, shuffled, L)
    kb, vb = B.gather(0, np.arange(n), L)
    assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    k8, v8 = opool.store_is_int8(variant)
    if not k8:
        assert np.array_equal(ka, k.astype(np.float64))
    if not v8:
        assert np.array_equal(va, v.astype(np.float64))
    if k8:
        c, s = quant.quantize(k, gs)
        assert np.array_equal(ka, quant.dequantize(c, s, gs))


def test_append_overwrites_one_slot_only():
    P = opool.Pool(1, 1, 4, 4, 4, 3, opool.K8V8)
    ones = np.ones((1, 1, 1, 4), np.float16)
    P.append(0, ones, ones, [5], np.array([[2, 0]]))     # pos 5 -> page 0 slot 1
    assert P.k_store[0, 0, 0, 1].tolist() == [127] * 4
    assert np.count_nonzero(P.k_store) == 4
    assert np.count_nonzero(P.k_store[0, 2]) == 0

"""Pins for the oracle's pool image (CPU only): the format-3 save/load that carries
the scales region with the codes (genie-ai-runtime release v0.1.0-alpha.12,
"Path F (#45) interop guard"; release v0.1.0-alpha.11, "--int8-kv triage": a
save/load must persist the scales region, or refuse a cache whose int8 setting
differs)."""

import os
import struct

import numpy as np
import pytest

from oracle import image as oimage
from oracle import pool as opool

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pool_image_v3.txt")


def _golden():
    ks, vs, hexes = [], [], []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        tag, rest = line.split(None, 1)
        if tag == "k":
            ks.append([float(x) for x in rest.split()])
        elif tag == "v":
            vs.append([float(x) for x in rest.split()])
        elif tag == "hex":
            hexes.append(rest.replace(" ", ""))
    return (np.array(ks, np.float16), np.array(vs, np.float16), bytes.fromhex("".join(hexes)))


def test_image_matches_the_hand_assembled_bytes():
    k, v, want = _golden()
    P = opool.Pool(1, 1, 8, 4, 4, 3, opool.K8V8)
    pt = np.array([[2, 0]])
    P.append(0, k[None, :, None, :], v[None, :, None, :], [0], pt)
    got = oimage.save(P, [2], pt)
    assert got == want
    assert oimage.image_bytes(P, [2]) == len(want) == 48 + 16 + 64


def _random_pool(variant, L_list, ps, n_pages, seed, n_layers=2, Hkv=2, D=64, gs=32):
    rng = np.random.default_rng(seed)
    P = opool.Pool(n_layers, Hkv, D, gs, ps, n_pages, variant)
    need = [-(-L // ps) for L in L_list]
    ids = rng.permutation(n_pages)[:sum(need)]
    pt = np.full((len(L_list), max(need)), -1, np.int64)
    o = 0
    for b, n in enumerate(need):
        pt[b, :n] = ids[o:o + n]
        o += n
    for layer in range(n_layers):
        for b, L in enumerate(L_list):
            k = (rng.standard_normal((L, Hkv, D)) * (1 + layer)).astype(np.float16)
            vv = rng.standard_normal((L, Hkv, D)).astype(np.float16)
            P.append_contiguous(layer, k, vv, 0, pt[b])
    return P, pt


@pytest.mark.parametrize("variant", [opool.K8V8, opool.K8V16, opool.K16V8, opool.K8V4, opool.Q4_0])
def test_round_trip_into_another_paging(variant):
    """Saved from pages of 16 positions, loaded into pages of 64 through another
    permutation: every layer of every sequence reads back the same codes, scales
    and dequantized values."""
    lens = [37, 200, 1, 0]
    A, pta = _random_pool(variant, lens, 16, 40, seed=5)
    img = oimage.save(A, lens, pta)
    assert len(img) == oimage.image_bytes(A, lens)
    B, ptb = _random_pool(variant, [0, 0, 0, 0], 64, 17, seed=6)  # empty pool, other shape of paging
    rng = np.random.default_rng(7)
    ptb = rng.permutation(17)[:16].reshape(4, 4)
    assert oimage.load(B, img, ptb) == lens
    for layer in range(2):
        for b, L in enumerate(lens):
            ka, va = A.gather(layer, pta[b], L)
            kb, vb = B.gather(layer, ptb[b], L)
            assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    assert oimage.save(B, lens, ptb) == img          # the image does not depend on the paging


def test_scales_travel_with_the_codes():
    """An int8 image is larger than its codes by exactly the scales region:
    2 bytes per (position, kv head, group) and store, as Strata's 528 B/cell
    counts them (codes 512 + scales 16 at head_dim 256, 2 kv heads, groups of 64)."""
    P = opool.Pool(1, 2, 256, 64, 64, 4, opool.K8V8)
    L = 64
    n = oimage.image_bytes(P, [L]) - 48 - 16
    assert n == 2 * L * opool.bytes_per_cell(2, 256, 64, int8=True) == 2 * L * 528


def _header(img, **kw):
    fields = list(oimage.HEADER.unpack_from(img, 0))
    names = ["magic", "version", "variant", "n_layers", "n_kv_heads", "head_dim", "group_size",
             "n_seqs", "payload", "zero"]
    for k, val in kw.items():
        fields[names.index(k)] = val
    return oimage.HEADER.pack(*fields) + img[oimage.HEADER.size:]


def test_load_refuses_foreign_images():
    lens = [50, 3]
    A, pta = _random_pool(opool.K8V8, lens, 16, 10, seed=9)
    img = oimage.save(A, lens, pta)
    B, _ = _random_pool(opool.K8V8, [0, 0], 16, 10, seed=10)
    with pytest.raises(oimage.FormatError):          # a v2 image (no scales) is not read
        oimage.load(B, _header(img, version=2), pta)
    with pytest.raises(oimage.FormatError):
        oimage.load(B, _header(img, magic=b"XXXX"), pta)
    with pytest.raises(oimage.FormatError):          # int8 image into an fp16-V pool
        C, _ = _random_pool(opool.K8V16, [0, 0], 16, 10, seed=11)
        oimage.load(C, img, pta)
    with pytest.raises(oimage.FormatError):          # other group size
        oimage.load(B, _header(img, group_size=64), pta)
    with pytest.raises(oimage.FormatError):          # truncated
        oimage.load(B, img[:-1], pta)
    with pytest.raises(oimage.FormatError):          # a length beyond the page-table row
        oimage.load(B, img, pta[:, :1])
    with pytest.raises(oimage.FormatError):          # one row per sequence
        oimage.load(B, img, pta[:1])
    assert struct.unpack_from("<I", img, 4)[0] == 3


def _placement_pool():
    """Two kv heads, head_dim 8, one scale per row (group 8), one sequence of 3
    positions on pages of 2.  Row (p, h) of K is [127 * 2^e, 10p + h, 0 ...] with
    e = p + 2h, so its scale is 2^e and its codes are [127, (10p + h) / 2^e
    rounded, 0 ...]; V row (p, h) is [-(20p + h), 0 ...] (scale (20p + h)/127)."""
    P = opool.Pool(1, 2, 8, 8, 2, 4, opool.K8V8)
    k = np.zeros((1, 3, 2, 8), np.float16)
    v = np.zeros((1, 3, 2, 8), np.float16)
    for p in range(3):
        for h in range(2):
            k[0, p, h, 0] = 127 * 2.0 ** (p + 2 * h)
            k[0, p, h, 1] = 10 * p + h
            v[0, p, h, 0] = -(20 * p + h) if (p, h) != (0, 0) else -1
    pt = np.array([[3, 1]])
    P.append(0, k, v, [0], pt)
    return P, pt


def test_sections_are_position_major_with_their_scales():
    """Hand-computed offsets: section K holds row (p, h) at byte (p * 2 + h) * 8 of
    its 48 bytes; the K scales section follows the two 48-byte code sections
    (each padded to 48) at (p * 2 + h) * 2 and holds 2^(p + 2h)."""
    P, pt = _placement_pool()
    img = oimage.save(P, [3], pt)
    base = 48 + 16
    kcodes = np.frombuffer(img, np.int8, 48, base)
    for p in range(3):
        for h in range(2):
            row = kcodes[(p * 2 + h) * 8:(p * 2 + h + 1) * 8]
            assert row[0] == 127
            assert row[1] == int(np.rint((10 * p + h) / 2.0 ** (p + 2 * h)))
    vcodes = np.frombuffer(img, np.int8, 48, base + 48)
    assert vcodes[0] == -127 and vcodes[(2 * 2 + 1) * 8] == -127
    ks = np.frombuffer(img, np.float16, 6, base + 96)
    assert [float(x) for x in ks] == [2.0 ** (p + 2 * h) for p in range(3) for h in range(2)]
    vs = np.frombuffer(img, np.float16, 6, base + 96 + 16)
    assert float(vs[5]) == float(np.float16(np.float32(41) / np.float32(127)))
    assert len(img) == base + 48 + 48 + 16 + 16

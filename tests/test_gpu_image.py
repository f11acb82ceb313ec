"""Saved pool images on the GPU (kv_pool_save / kv_pool_load) against the oracle.

The image carries the int8 codes together with their scales (genie-ai-runtime
release v0.1.0-alpha.12, "Path F (#45) interop guard": format v2 lacked the
scales, format v3 persists them).  Checks: the device writes the oracle's image
byte for byte; loading it into a fresh pool through another page table (and
another page count) gives the oracle's loaded regions bit for bit and the same
decode output bit for bit; foreign images are refused before anything is
written.
"""

import numpy as np
import pytest
import torch

from int8_kv_cache_02_gb300 import inputs
from oracle import image as oimage
from oracle import pool as opool
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.lib_ready()


def _filled(seed, lens, n_layers, Hkv, D, gs, variant, n_pages_extra=3, outliers=False):
    from int8_kv_cache_02_gb300 import binding
    pt, n_pages = inputs.page_table(lens, 64, seed=seed)
    n_pages += n_pages_extra
    dev, orc = gu.make_pools(n_layers, Hkv, D, gs, 64, n_pages, variant)
    for layer in range(n_layers):
        q, ks, vs = inputs.random_case(seed + 17 * layer, len(lens), 8, Hkv, D, lens,
                                       outliers=outliers)
        for b in range(len(lens)):
            gu.fill_sequence(dev, orc, layer, ks[b], vs[b], pt[b])
    assert binding.kv_pool_read_device_error(dev) == 0
    return dev, orc, pt


@pytest.mark.parametrize("D,gs,variant", [(256, 64, 0), (128, 128, 1), (128, 64, 2), (256, 256, 0)])
def test_save_writes_the_oracle_image_and_load_restores_it(D, gs, variant):
    from int8_kv_cache_02_gb300 import binding
    lens = [700, 64, 1, 0, 1500]
    dev, orc, pt = _filled(40 + D + variant, lens, 2, 2, D, gs, variant, outliers=True)
    img = binding.kv_pool_save(dev, lens, pt.cuda())
    want = oimage.save(orc, lens, pt.numpy())
    assert len(img) == len(want) == binding.kv_pool_image_bytes(dev, lens)
    assert img == want

    # another paging: more pages, another permutation
    pt2, n2 = inputs.page_table(lens, 64, seed=99, n_pages_total=pt.shape[0] * pt.shape[1] + 7)
    dev2, orc2 = gu.make_pools(2, 2, D, gs, 64, n2, variant)
    assert binding.kv_pool_load(dev2, img, pt2.cuda()) == lens
    assert oimage.load(orc2, want, pt2.numpy()) == lens
    gu.regions_equal(dev2, orc2)
    assert binding.kv_pool_read_device_error(dev2) == 0

    # the reloaded cache decodes to the same bits
    q = inputs.normal_f16((len(lens), 16, D), torch.Generator().manual_seed(5)).cuda()
    lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
    for layer in (0, 1):
        a = torch.empty((len(lens), 16, D), dtype=torch.float32, device="cuda")
        b = torch.empty_like(a)
        binding.attn_decode_int8(dev, layer, q, lens_d, pt.cuda(), a, dev.decode_workspace(5, 16, 3),
                                 n_splits=3)
        binding.attn_decode_int8(dev2, layer, q, lens_d, pt2.cuda(), b,
                                 dev2.decode_workspace(5, 16, 3), n_splits=3)
        torch.cuda.synchronize()
        assert torch.equal(a, b)


@pytest.mark.slow
def test_grouped8k_workload_round_trip():
    """The 8K-context workload (16/2 heads, head_dim 256, 64-value groups, outlier K
    channels): saved, reloaded into a pool with pages in another order, byte-equal
    to the oracle's image and bit-equal when decoded."""
    from int8_kv_cache_02_gb300 import binding
    w = inputs.grouped8k()
    L = w["L"]
    pt, n = inputs.page_table([L], 64, seed=21)
    dev, orc = gu.make_pools(1, 2, 256, 64, 64, n, 0)
    gu.fill_sequence(dev, orc, 0, w["k"], w["v"], pt[0])
    img = binding.kv_pool_save(dev, [L], pt.cuda())
    assert img == oimage.save(orc, [L], pt.numpy())
    pt2, _ = inputs.page_table([L], 64, seed=22)
    dev2, orc2 = gu.make_pools(1, 2, 256, 64, 64, n, 0)
    assert binding.kv_pool_load(dev2, img, pt2.cuda()) == [L]
    oimage.load(orc2, img, pt2.numpy())
    gu.regions_equal(dev2, orc2)
    out = []
    for d, p in ((dev, pt), (dev2, pt2)):
        o = torch.empty((1, 16, 256), dtype=torch.float32, device="cuda")
        binding.attn_decode_int8(d, 0, w["q"].cuda(), torch.tensor([L], dtype=torch.int32,
                                                                    device="cuda"),
                                 p.cuda(), o, d.decode_workspace(1, 16, 16), n_splits=16)
        out.append(o)
    torch.cuda.synchronize()
    assert torch.equal(out[0], out[1])
    kh, vh = orc.gather(0, pt[0].numpy(), L)
    from oracle import attention as oatt
    gu.assert_attention_close(out[1][0].cpu().numpy(), oatt.decode(w["q"][0].numpy(), kh, vh, L),
                              "reloaded 8K")


def test_load_refuses_foreign_images_and_writes_nothing():
    from int8_kv_cache_02_gb300 import binding
    lens = [130, 5]
    dev, orc, pt = _filled(77, lens, 1, 2, 128, 64, 0)
    img = binding.kv_pool_save(dev, lens, pt.cuda())
    fresh, _ = gu.make_pools(1, 2, 128, 64, 64, pt.numel() + 2, 0)
    v2 = bytearray(img)
    v2[4] = 2                                                   # format version 2: no scales
    other, _ = gu.make_pools(1, 2, 128, 64, 64, pt.numel() + 2, 1)   # fp16 V store
    for bad, pool in ((bytes(v2), fresh), (img, other), (b"NOPE" + img[4:], fresh)):
        with pytest.raises(binding.Int8KVError) as e:
            binding.kv_pool_load(pool, bad, pt.cuda())
        assert e.value.status == binding.ERR_FORMAT
    torch.cuda.synchronize()
    assert int(fresh.k_store.abs().sum()) == 0 and int(fresh.k_scales.float().abs().sum()) == 0
    with pytest.raises(binding.Int8KVError):                    # truncated
        binding.kv_pool_load(fresh, img[:-16], pt.cuda())

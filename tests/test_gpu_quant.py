"""kv_quant_append on the GPU against the oracle: codes and scales bit-exact."""

import numpy as np
import pytest
import torch

from int8_kv_cache_02_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.lib_ready()


@pytest.mark.parametrize("variant", [0, 1, 2])
@pytest.mark.parametrize("D,gs,ps", [(128, 128, 64), (256, 64, 64), (64, 32, 16), (256, 16, 32),
                                     (128, 32, 128)])
def test_append_small_bit_exact(variant, D, gs, ps):
    Hkv, L = 2, 333
    q, ks, vs = inputs.random_case(100 + D + gs, 1, 2 * Hkv, Hkv, D, [L], outliers=True)
    pt, n_pages = inputs.page_table([L], ps, n_pages_total=-(-L // ps) + 5, seed=ps + D)
    dev, orc = gu.make_pools(2, Hkv, D, gs, ps, n_pages, variant)
    gu.fill_sequence(dev, orc, 1, ks[0], vs[0], pt[0], chunk=100)
    gu.regions_equal(dev, orc)


def test_append_every_finite_fp16_value():
    """All 63,488 finite fp16 values (shuffled into 64-value groups), plus groups of
    tiny values whose scale is a subnormal fp16, through the kernel."""
    bits = np.concatenate([np.arange(0, 0x7C00), np.arange(0x8000, 0xFC00)]).astype(np.uint16)
    rng = np.random.default_rng(0)
    vals = bits[rng.permutation(bits.size)].view(np.float16)
    tiny = (rng.standard_normal(256 * 64) * 1e-4).astype(np.float16)    # amax/127 < 2^-14
    x = np.concatenate([vals, tiny])
    n_rows = x.size // 256
    x = x[: n_rows * 256].reshape(n_rows, 1, 256)
    k = torch.from_numpy(x.copy())
    v = torch.from_numpy(x[::-1].copy())
    pt, n_pages = inputs.page_table([n_rows], 64, seed=1)
    dev, orc = gu.make_pools(1, 1, 256, 64, 64, n_pages, 0)
    gu.fill_sequence(dev, orc, 0, k, v, pt[0])
    gu.regions_equal(dev, orc)
    assert (orc.k_scales.astype(np.float64) < 2.0 ** -14).any()    # subnormal scales occurred


@pytest.mark.parametrize("D,gs", [(256, 64), (128, 128), (64, 32)])
def test_append_rounding_ties(D, gs):
    """Values whose quotient x / s is exactly k + 1/2 (round half to even) or one
    fp16 step from it, for scales from 2^-20 to 7 * 2^4."""
    n = 512
    k = inputs.tie_rows(n, D, gs, seed=D + gs).reshape(n, 1, D)
    v = inputs.tie_rows(n, D, gs, seed=D + gs + 1).reshape(n, 1, D)
    pt, n_pages = inputs.page_table([n], 64, seed=2)
    dev, orc = gu.make_pools(1, 1, D, gs, 64, n_pages, 0)
    gu.fill_sequence(dev, orc, 0, k, v, pt[0])
    gu.regions_equal(dev, orc)


def test_append_batch_of_sequences_at_different_positions():
    from int8_kv_cache_02_gb300 import binding
    B, n_new, Hkv, D, gs, ps = 5, 7, 4, 128, 64, 16
    starts = [0, 13, 64, 100, 250]
    lens = [s + n_new for s in starts]
    pt, n_pages = inputs.page_table(lens, ps, seed=9)
    g = torch.Generator().manual_seed(5)
    k = inputs.normal_f16((B, n_new, Hkv, D), g)
    v = inputs.normal_f16((B, n_new, Hkv, D), g)
    dev, orc = gu.make_pools(1, Hkv, D, gs, ps, n_pages, 0)
    binding.kv_quant_append(dev, 0, k.cuda(), v.cuda(),
                            torch.tensor(starts, dtype=torch.int32, device="cuda"), pt.cuda())
    orc.append(0, k.numpy(), v.numpy(), starts, pt.numpy())
    gu.regions_equal(dev, orc)


def test_bad_page_id_is_skipped_and_flagged():
    from int8_kv_cache_02_gb300 import binding
    dev, orc = gu.make_pools(1, 2, 128, 128, 64, 4, 0)
    pt = torch.tensor([[0, 99]], dtype=torch.int32, device="cuda")       # page 99 is outside
    k = torch.ones((1, 2, 2, 128), dtype=torch.float16, device="cuda")
    binding.kv_quant_append(dev, 0, k, k, torch.tensor([63], dtype=torch.int32, device="cuda"), pt)
    err = binding.kv_pool_read_device_error(dev)
    assert err & binding.DEVERR_PAGE_ID
    ks = dev.k_store.cpu()
    assert (ks[0, 0, :, 63] == 127).all() and int((ks != 0).sum()) == 2 * 128
    assert binding.kv_pool_read_device_error(dev) == 0                  # read clears the word


@pytest.mark.slow
@pytest.mark.parametrize("name", ["grouped8k", "prefill", "long128k"])
def test_append_full_size_workloads(name):
    """Whole caches of the measured workloads built by the kernel, compared byte for byte."""
    w = getattr(inputs, name)()
    n = w["k"].shape[0]
    pt, n_pages = inputs.page_table([n], 64, seed=3)
    dev, orc = gu.make_pools(1, w["Hkv"], w["D"], w["gs"], 64, n_pages, 0)
    gu.fill_sequence(dev, orc, 0, w["k"], w["v"], pt[0])
    gu.regions_equal(dev, orc)

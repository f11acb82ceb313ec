"""attn_prefill_chunk_int8 on the GPU against the fp64 oracle.

The chunk's K/V are appended first (kv_quant_append), then causal attention of
the chunk's queries runs over the whole int8 cache.  Tolerance as for decode:
max abs <= 2e-3, max rel-L2 per (position, head) vector <= 1e-4.
"""

import numpy as np
import pytest
import torch

from int8_kv_cache_02_gb300 import inputs
from oracle import attention as oatt
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.lib_ready()


def _run(seed, H, Hkv, D, gs, start, n_new, variant, n_splits=0, outliers=True, scale=0.0,
         spare=2, v=None):
    """v: the sequence's V rows [start + n_new][Hkv][D] (fp16) instead of random ones."""
    from int8_kv_cache_02_gb300 import binding
    L = start + n_new
    q_all, ks, vs = inputs.random_case(seed, n_new, H, Hkv, D, [L], outliers=outliers)
    if v is not None:
        vs = [v]
    q = q_all                                                   # [n_new][H][D]
    pt, n_pages = inputs.page_table([L], 64, n_pages_total=-(-L // 64) + spare, seed=seed)
    dev, orc = gu.make_pools(1, Hkv, D, gs, 64, n_pages, variant)
    if start:
        gu.fill_sequence(dev, orc, 0, ks[0][:start], vs[0][:start], pt[0])
    gu.fill_sequence(dev, orc, 0, ks[0][start:], vs[0][start:], pt[0], start=start)  # the chunk
    ns = n_splits or binding.attn_prefill_n_splits(dev, n_new, H, start)
    nb = binding.attn_prefill_workspace_bytes(n_new, H, Hkv, D, ns)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
    out = torch.full((n_new, H, D), float("nan"), dtype=torch.float32, device="cuda")
    binding.attn_prefill_chunk_int8(dev, 0, q.cuda(), start, pt[0].cuda(), out, ws,
                                    softmax_scale=scale, n_splits=ns)
    torch.cuda.synchronize()
    assert binding.kv_pool_read_device_error(dev) == 0
    kh, vh = orc.gather(0, pt[0].numpy(), L)
    ref = oatt.prefill_chunk(q.numpy(), kh, vh, start, scale=scale or None)
    return out.cpu().numpy(), ref, dev, pt, q


@pytest.mark.parametrize("start,n_new", [(0, 1), (0, 70), (100, 17), (1000, 200), (4000, 64)])
@pytest.mark.parametrize("n_splits", [1, 3, 20, 0])
def test_prefill_matches_oracle_grouped(start, n_new, n_splits):
    out, ref, *_ = _run(10 + start + n_new, 16, 2, 256, 64, start, n_new, 0, n_splits)
    gu.assert_attention_close(out, ref, f"start {start} n_new {n_new} ns {n_splits}")


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("variant", [0, 1, 2])
def test_prefill_head_counts_and_variants(G, variant):
    Hkv = 2
    out, ref, *_ = _run(200 + G + 10 * variant, G * Hkv, Hkv, 128, 128, 300, 45, variant, 2)
    gu.assert_attention_close(out, ref, f"G {G} variant {variant}")


@pytest.mark.parametrize("gs", [64, 128, 256])
@pytest.mark.parametrize("variant", [1, 2])
def test_prefill_group_sizes_fp16_stores(gs, variant):
    out, ref, *_ = _run(300 + gs + variant, 16, 2, 256, gs, 513, 33, variant, 4)
    gu.assert_attention_close(out, ref, f"gs {gs} variant {variant}")


def test_prefill_rows_agree_with_decode_at_their_length():
    """Row i of the chunk equals a decode of the same sequence at length start + i + 1."""
    from int8_kv_cache_02_gb300 import binding
    start, n_new = 700, 9
    out, ref, dev, pt, q = _run(41, 16, 2, 256, 64, start, n_new, 0, 2)
    lens = torch.tensor([start + i + 1 for i in range(n_new)], dtype=torch.int32, device="cuda")
    ptb = pt[0].repeat(n_new, 1).contiguous().cuda()
    dec = torch.empty((n_new, 16, 256), dtype=torch.float32, device="cuda")
    binding.attn_decode_int8(dev, 0, q.cuda(), lens, ptb, dec, dev.decode_workspace(n_new, 16, 1),
                             n_splits=1)
    torch.cuda.synchronize()
    assert np.max(np.abs(dec.cpu().numpy() - out)) <= 2e-5
    gu.assert_attention_close(out, ref, "prefill")


@pytest.mark.parametrize("vmag", [3e-6, 1e-3, 3e2, 6e4])
def test_prefill_value_magnitudes(vmag):
    """V from 3e-6 (fp16 subnormal scales of one or two units of 2^-24) to 6e4 (near
    fp16's largest value): the V range shift keeps the P.V factors and weights
    normal in fp16.  (Much smaller V rounds most groups' scales to zero; an output
    then made only of keys weighted below 2^-19 of the reference key is beyond
    the fp16 weight pairs' range.)"""
    start, n_new, Hkv, D = 600, 40, 2, 256
    g = torch.Generator().manual_seed(int(vmag * 1e6) % 1000 + 7)
    v = (torch.randn((start + n_new, Hkv, D), generator=g) * vmag).clamp(-65000, 65000)
    out, ref, *_ = _run(61, 16, Hkv, D, 64, start, n_new, 0, 3, v=v.to(torch.float16))
    gu.assert_attention_close(out / vmag, ref / vmag, f"vmag {vmag}")


def test_prefill_v_scales_growing_along_the_sequence():
    """V scales spanning 2^20 across positions, rising and falling, so that every
    group's power-of-two range is raised many times within a block's keys."""
    start, n_new, Hkv, D = 960, 64, 2, 256
    g = torch.Generator().manual_seed(78)
    ramp = torch.pow(2.0, torch.linspace(-12, 8, start + n_new)).roll(300)
    v = torch.randn((start + n_new, Hkv, D), generator=g) * ramp[:, None, None]
    for ns in (1, 4):
        out, ref, *_ = _run(62, 16, Hkv, D, 64, start, n_new, 0, ns, v=v.to(torch.float16))
        gu.assert_attention_close(out, ref, f"ramp ns {ns}")


def test_prefill_softmax_scale_override():
    out, ref, *_ = _run(51, 8, 2, 128, 64, 250, 30, 0, 2, scale=0.05)
    gu.assert_attention_close(out, ref, "scale")


@pytest.mark.slow
def test_prefill_workload_full_size():
    """32768 cached positions + a 256-query causal chunk, 16/2 heads, head_dim 256,
    64-value groups, outlier K channels; every output checked against the oracle."""
    from int8_kv_cache_02_gb300 import binding
    w = inputs.prefill()
    start, n_new = w["start"], w["n_new"]
    L = start + n_new
    pt, n_pages = inputs.page_table([L], 64, seed=6)
    dev, orc = gu.make_pools(1, 2, 256, 64, 64, n_pages, 0)
    gu.fill_sequence(dev, orc, 0, w["k"][:start], w["v"][:start], pt[0])
    gu.fill_sequence(dev, orc, 0, w["k"][start:], w["v"][start:], pt[0], start=start)
    gu.regions_equal(dev, orc)
    ns = binding.attn_prefill_n_splits(dev, n_new, 16, start)
    ws = torch.empty(max(16, binding.attn_prefill_workspace_bytes(n_new, 16, 2, 256, ns)),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((n_new, 16, 256), dtype=torch.float32, device="cuda")
    binding.attn_prefill_chunk_int8(dev, 0, w["q"].cuda(), start, pt[0].cuda(), out, ws,
                                    n_splits=ns)
    torch.cuda.synchronize()
    kh, vh = orc.gather(0, pt[0].numpy(), L)
    ref = oatt.prefill_chunk(w["q"].numpy(), kh, vh, start)
    gu.assert_attention_close(out.cpu().numpy(), ref, "prefill workload")


def test_prefill_rejects_unsupported_and_out_of_range():
    from int8_kv_cache_02_gb300 import binding
    dev, _ = gu.make_pools(1, 2, 128, 128, 64, 4, 0)
    q = torch.zeros((4, 6, 128), dtype=torch.float16, device="cuda")      # G = 3
    out = torch.zeros((4, 6, 128), dtype=torch.float32, device="cuda")
    pt = torch.arange(4, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.Int8KVError) as e:
        binding.attn_prefill_chunk_int8(dev, 0, q, 0, pt, out, None, n_splits=1)
    assert e.value.status == -6
    q = torch.zeros((4, 8, 128), dtype=torch.float16, device="cuda")
    out = torch.zeros((4, 8, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(binding.Int8KVError) as e:
        binding.attn_prefill_chunk_int8(dev, 0, q, 254, pt, out, None, n_splits=1)  # 258 > 256
    assert e.value.status == -5

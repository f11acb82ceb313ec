"""The tensor-memory decode kernel (tcgen05.mma, INT8KV_DECODE_TCGEN05) on the GPU
against the fp64 oracle over the dequantized cache.

Every pool here is switched to that kernel with kv_pool_set_decode_kernel, so the
cases below run it whatever the library would pick by itself.  Tolerance as for
every attention output: max abs error <= 2e-3 and max relative L2 error per
(sequence, query head) output vector <= 1e-4.
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


def _pools(n_layers, Hkv, D, gs, n_pages):
    from int8_kv_cache_02_gb300 import binding
    dev, orc = gu.make_pools(n_layers, Hkv, D, gs, 64, n_pages, binding.K8V8)
    dev.set_decode_kernel(binding.DECODE_TCGEN05)
    return dev, orc


def _setup(seed, B, H, Hkv, D, gs, lens, n_layers=1, layer=0, outliers=False, page_seed=1):
    q, ks, vs = inputs.random_case(seed, B, H, Hkv, D, lens, outliers=outliers)
    pt, n_pages = inputs.page_table([max(1, L) for L in lens], 64,
                                    n_pages_total=sum(-(-max(1, L) // 64) for L in lens) + 3,
                                    seed=page_seed)
    dev, orc = _pools(n_layers, Hkv, D, gs, n_pages)
    for b, L in enumerate(lens):
        if L:
            gu.fill_sequence(dev, orc, layer, ks[b], vs[b], pt[b])
    return q, pt, dev, orc


def _decode(dev, layer, q, lens, pt, window=0, n_splits=0, scale=0.0, ws=None):
    from int8_kv_cache_02_gb300 import binding
    B, H, D = q.shape
    if n_splits == 0:
        n_splits = binding.attn_decode_n_splits(dev, B, pt.shape[1] * dev.page_size)
    if ws is None:
        ws = dev.decode_workspace(B, H, n_splits)
    out = torch.full((B, H, D), float("nan"), dtype=torch.float32, device="cuda")
    binding.attn_decode_int8(dev, layer, q.cuda(), torch.tensor(lens, dtype=torch.int32,
                                                                  device="cuda"),
                             pt.cuda(), out, ws, window=window, softmax_scale=scale,
                             n_splits=n_splits)
    torch.cuda.synchronize()
    assert binding.kv_pool_read_device_error(dev) == 0
    return out.cpu().numpy()


def _oracle(orc, layer, q, lens, pt, window=0, scale=None):
    outs = []
    for b, L in enumerate(lens):
        kh, vh = orc.gather(layer, pt[b].numpy(), L)
        outs.append(oatt.decode(q[b].numpy(), kh, vh, L, window=window, scale=scale))
    return np.stack(outs)


CASES = [
    # seed, B, H, Hkv, D, gs, lens
    (1, 1, 8, 2, 128, 128, [512]),
    (2, 2, 16, 2, 256, 64, [700, 129]),
    (3, 3, 32, 8, 128, 128, [64, 1, 1000]),
    (4, 1, 16, 2, 256, 128, [1500]),
    (5, 2, 16, 2, 256, 256, [333, 65]),
    (6, 2, 8, 2, 128, 64, [257, 999]),
    (7, 1, 16, 2, 256, 64, [4100]),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"s{c[0]}")
@pytest.mark.parametrize("n_splits", [1, 3, 0])
def test_tc_decode_matches_oracle(case, n_splits):
    seed, B, H, Hkv, D, gs, lens = case
    q, pt, dev, orc = _setup(seed, B, H, Hkv, D, gs, lens, outliers=True)
    out = _decode(dev, 0, q, lens, pt, n_splits=n_splits)
    gu.assert_attention_close(out, _oracle(orc, 0, q, lens, pt), f"case {seed} ns {n_splits}")


@pytest.mark.parametrize("G", [1, 3, 5, 8])
def test_tc_head_counts(G):
    Hkv, lens = 2, [517, 64]
    q, pt, dev, orc = _setup(300 + G, 2, G * Hkv, Hkv, 256, 64, lens, outliers=True)
    for ns in (1, 5):
        gu.assert_attention_close(_decode(dev, 0, q, lens, pt, n_splits=ns),
                                  _oracle(orc, 0, q, lens, pt), f"G={G} ns={ns}")


@pytest.mark.parametrize("window,lens", [(512, [2000, 300, 513]), (100, [100, 101, 5000]),
                                         (1, [7, 64])])
def test_tc_sliding_window(window, lens):
    q, pt, dev, orc = _setup(90 + window, len(lens), 16, 2, 256, 64, lens)
    for ns in (1, 2, 0):
        out = _decode(dev, 0, q, lens, pt, window=window, n_splits=ns)
        gu.assert_attention_close(out, _oracle(orc, 0, q, lens, pt, window=window),
                                  f"window {window} ns {ns}")


def test_tc_context_one_returns_the_dequantized_v_row():
    q, pt, dev, orc = _setup(31, 2, 16, 2, 256, 64, [1, 1])
    out = _decode(dev, 0, q, [1, 1], pt, n_splits=1)
    for b in range(2):
        _, vh = orc.gather(0, pt[b].numpy(), 1)
        for h in range(16):
            assert np.array_equal(out[b, h].astype(np.float64), vh[0, h // 8])


def test_tc_identical_keys_return_the_mean_of_v():
    L, Hkv, D = 300, 2, 128
    g = torch.Generator().manual_seed(41)
    k = inputs.normal_f16((1, Hkv, D), g).expand(L, Hkv, D).contiguous()
    v = inputs.normal_f16((L, Hkv, D), g)
    q = inputs.normal_f16((1, 8, D), g)
    pt, n_pages = inputs.page_table([L], 64, seed=2)
    dev, orc = _pools(1, Hkv, D, 128, n_pages)
    gu.fill_sequence(dev, orc, 0, k, v, pt[0])
    out = _decode(dev, 0, q, [L], pt, n_splits=3)
    _, vh = orc.gather(0, pt[0].numpy(), L)
    for h in range(8):
        assert np.allclose(out[0, h], vh[:, h // 4].mean(axis=0), rtol=0, atol=2e-6)


def test_tc_split_equals_single_pass():
    q, pt, dev, orc = _setup(33, 1, 16, 2, 256, 64, [3000], outliers=True)
    one = _decode(dev, 0, q, [3000], pt, n_splits=1)
    for ns in (2, 7, 47):
        many = _decode(dev, 0, q, [3000], pt, n_splits=ns)
        assert np.max(np.abs(one - many)) <= 1e-5, ns


def test_tc_empty_sequences_and_more_splits_than_pages():
    lens = [0, 130, 0, 65]
    q, pt, dev, orc = _setup(51, 4, 8, 2, 128, 128, lens)
    for ns in (4, 9):
        out = _decode(dev, 0, q, lens, pt, n_splits=ns)
        assert (out[0] == 0).all() and (out[2] == 0).all()
        gu.assert_attention_close(out[[1, 3]], _oracle(orc, 0, q[[1, 3]], [130, 65],
                                                       pt[[1, 3]]), f"ns {ns}")


def test_tc_workspace_reuse_is_deterministic_and_scale_override():
    q, pt, dev, orc = _setup(71, 1, 16, 2, 256, 64, [1000], n_layers=2, layer=1, outliers=True)
    ws = dev.decode_workspace(1, 16, 6)
    a = _decode(dev, 1, q, [1000], pt, n_splits=6, ws=ws)
    b = _decode(dev, 1, q, [1000], pt, n_splits=6, ws=ws)
    assert np.array_equal(a, b)
    gu.assert_attention_close(a, _oracle(orc, 1, q, [1000], pt), "layer 1")
    sc = 0.3
    gu.assert_attention_close(_decode(dev, 1, q, [1000], pt, n_splits=2, scale=sc),
                              _oracle(orc, 1, q, [1000], pt, scale=sc), "scale")


@pytest.mark.parametrize("vmag", [1e-6, 1e-3, 3e2, 6e4])
def test_tc_value_magnitudes(vmag):
    """V from 1e-6 to 6e4: the power-of-two range of P' keeps its hi/lo parts normal."""
    L, Hkv, D = 700, 2, 128
    g = torch.Generator().manual_seed(int(vmag * 1e6) % 1000 + 7)
    q = inputs.normal_f16((1, 8, D), g)
    k = inputs.normal_f16((L, Hkv, D), g)
    v = (torch.randn((L, Hkv, D), generator=g) * vmag).clamp(-65000, 65000).to(torch.float16)
    pt, n_pages = inputs.page_table([L], 64, seed=4)
    dev, orc = _pools(1, Hkv, D, 64, n_pages)
    gu.fill_sequence(dev, orc, 0, k, v, pt[0])
    ref = _oracle(orc, 0, q, [L], pt)
    for ns in (1, 4):
        gu.assert_attention_close(_decode(dev, 0, q, [L], pt, n_splits=ns) / vmag, ref / vmag,
                                  f"vmag {vmag}")


def test_tc_v_scales_and_scores_growing_along_the_sequence():
    """V scales spanning 2^20 and score maxima rising page after page, so the block's
    V ranges and reference maxima move many times (O rescaled in tensor memory)."""
    L, Hkv, D = 2048, 2, 256
    g = torch.Generator().manual_seed(77)
    q = (inputs.normal_f16((1, 16, D), g).float() * 4).to(torch.float16)
    kramp = torch.linspace(0.05, 3.0, L)
    k = (torch.randn((L, Hkv, D), generator=g) * kramp[:, None, None]).to(torch.float16)
    vramp = torch.pow(2.0, torch.linspace(-12, 8, L)).roll(700)
    v = (torch.randn((L, Hkv, D), generator=g) * vramp[:, None, None]).to(torch.float16)
    pt, n_pages = inputs.page_table([L], 64, seed=5)
    dev, orc = _pools(1, Hkv, D, 64, n_pages)
    gu.fill_sequence(dev, orc, 0, k, v, pt[0])
    ref = _oracle(orc, 0, q, [L], pt)
    for ns in (1, 2, 7):
        gu.assert_attention_close(_decode(dev, 0, q, [L], pt, n_splits=ns), ref, f"ns {ns}")


def test_tc_ignores_garbage_scales_beyond_the_context():
    """Scale slots past the sequence end hold NaN / Inf bit patterns and the code
    slots random bytes: the output depends on positions < L only."""
    L = 100
    q, pt, dev, orc = _setup(501, 1, 16, 2, 256, 64, [L])
    last = int(pt[0, 1])
    for sc in (dev.k_scales, dev.v_scales):
        raw = sc.view(torch.int16)
        raw[0, last, :, L - 64:, :] = 0x7E00
        raw[0, last, :, L - 64 + 20:, :] = 0x7C00
    g = torch.Generator().manual_seed(3)
    junk = torch.randint(-128, 128, (2, 64 - (L - 64), 256), generator=g, dtype=torch.int8)
    dev.k_store[0, last, :, L - 64:, :] = junk.cuda()
    dev.v_store[0, last, :, L - 64:, :] = junk.flip(0).cuda()
    out = _decode(dev, 0, q, [L], pt, n_splits=1)
    assert np.isfinite(out).all()
    gu.assert_attention_close(out, _oracle(orc, 0, q, [L], pt), "garbage")


def test_tc_decode_append_equals_append_then_decode():
    """The tensor-memory kernel has no fused append: attn_decode_append_int8 appends
    first; the pool and the output equal kv_quant_append then attn_decode_int8."""
    from int8_kv_cache_02_gb300 import binding
    lens = [300, 65]
    q, ks, vs = inputs.random_case(17, 2, 16, 2, 256, lens, outliers=True)
    pt, n_pages = inputs.page_table([L + 1 for L in lens], 64, n_pages_total=12, seed=9)
    outs, pools = [], []
    for fused in (True, False):
        dev, orc = _pools(1, 2, 256, 64, n_pages)
        for b, L in enumerate(lens):
            gu.fill_sequence(dev, orc, 0, ks[b][:L - 1], vs[b][:L - 1], pt[b], oracle=False)
        newk = torch.stack([ks[b][L - 1] for b, L in enumerate(lens)]).cuda()
        newv = torch.stack([vs[b][L - 1] for b, L in enumerate(lens)]).cuda()
        seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
        ws = dev.decode_workspace(2, 16, 3)
        out = torch.empty((2, 16, 256), dtype=torch.float32, device="cuda")
        if fused:
            binding.attn_decode_append_int8(dev, 0, q.cuda(), newk, newv, seq, pt.cuda(), out, ws,
                                            n_splits=3)
        else:
            binding.kv_quant_append(dev, 0, newk.unsqueeze(1), newv.unsqueeze(1), seq - 1,
                                    pt.cuda())
            binding.attn_decode_int8(dev, 0, q.cuda(), seq, pt.cuda(), out, ws, n_splits=3)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
        pools.append(dev)
    assert np.array_equal(outs[0], outs[1])
    for a, b in ((pools[0].k_store, pools[1].k_store), (pools[0].v_store, pools[1].v_store),
                 (pools[0].k_scales, pools[1].k_scales), (pools[0].v_scales, pools[1].v_scales)):
        assert torch.equal(a, b)


def test_tc_selector_refuses_what_it_cannot_serve():
    from int8_kv_cache_02_gb300 import binding
    for variant in (binding.K8V16, binding.K16V8):
        dev, _ = gu.make_pools(1, 2, 256, 64, 64, 4, variant)
        with pytest.raises(binding.Int8KVError):
            dev.set_decode_kernel(binding.DECODE_TCGEN05)
        dev.set_decode_kernel(binding.DECODE_WARP_MMA)
    dev, _ = gu.make_pools(1, 2, 64, 64, 16, 4, binding.K8V8)
    with pytest.raises(binding.Int8KVError):
        dev.set_decode_kernel(binding.DECODE_TCGEN05)
    with pytest.raises(binding.Int8KVError):
        dev.set_decode_kernel(7)
    dev.set_decode_kernel(binding.DECODE_SIMT)


@pytest.mark.slow
def test_tc_long128k_workload():
    w = inputs.long128k()
    L = 131072
    pt, n_pages = inputs.page_table([L], 64, seed=8)
    dev, orc = _pools(1, 2, 256, 64, n_pages)
    gu.fill_sequence(dev, orc, 0, w["k"], w["v"], pt[0])
    ref = _oracle(orc, 0, w["q"], [L], pt)
    gu.assert_attention_close(_decode(dev, 0, w["q"], [L], pt), ref, "128k tc")

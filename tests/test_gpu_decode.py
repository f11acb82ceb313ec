"""attn_decode_int8 on the GPU against the fp64 oracle over the dequantized cache.

Tolerance (fp32 kernel vs fp64 oracle): max abs error <= 2e-3 and max relative
L2 error per (sequence, query head) output vector <= 1e-4.
"""

import math

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


def _setup(seed, B, H, Hkv, D, gs, lens, variant, ps=64, n_layers=1, layer=0, outliers=False,
           page_seed=1, spare_pages=3):
    q, ks, vs = inputs.random_case(seed, B, H, Hkv, D, lens, outliers=outliers)
    pt, n_pages = inputs.page_table([max(1, L) for L in lens], ps,
                                    n_pages_total=sum(-(-max(1, L) // ps) for L in lens) + spare_pages,
                                    seed=page_seed)
    dev, orc = gu.make_pools(n_layers, Hkv, D, gs, ps, n_pages, variant)
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
    return out.cpu().numpy()


def _oracle(orc, layer, q, lens, pt, window=0, scale=None):
    outs = []
    for b, L in enumerate(lens):
        kh, vh = orc.gather(layer, pt[b].numpy(), L)
        outs.append(oatt.decode(q[b].numpy(), kh, vh, L, window=window, scale=scale))
    return np.stack(outs)


CASES = [
    # seed, B, H, Hkv, D, gs, lens, variant, ps
    (1, 1, 8, 2, 128, 128, [512], 0, 64),
    (2, 2, 16, 2, 256, 64, [700, 129], 0, 64),
    (3, 3, 32, 8, 128, 128, [64, 1, 1000], 0, 64),
    (4, 2, 8, 1, 64, 32, [300, 77], 0, 16),
    (5, 1, 16, 2, 256, 64, [1500], 1, 64),
    (6, 1, 16, 2, 256, 64, [1500], 2, 64),
    (7, 2, 4, 4, 128, 64, [333, 65], 0, 32),
    (8, 2, 12, 2, 128, 32, [257, 999], 1, 128),
    (9, 1, 10, 2, 64, 64, [200], 2, 64),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"s{c[0]}")
@pytest.mark.parametrize("n_splits", [1, 4, 0])
def test_decode_matches_oracle(case, n_splits):
    seed, B, H, Hkv, D, gs, lens, variant, ps = case
    q, pt, dev, orc = _setup(seed, B, H, Hkv, D, gs, lens, variant, ps=ps, outliers=True)
    out = _decode(dev, 0, q, lens, pt, n_splits=n_splits)
    ref = _oracle(orc, 0, q, lens, pt)
    gu.assert_attention_close(out, ref, f"case {seed} n_splits {n_splits}")


@pytest.mark.parametrize("window,lens", [(512, [2000, 300, 513]), (100, [100, 101, 5000]),
                                         (1, [7, 1])])
def test_sliding_window(window, lens):
    q, pt, dev, orc = _setup(21, len(lens), 32, 8, 128, 128, lens, 0)
    for ns in (1, 3, 0):
        out = _decode(dev, 0, q, lens, pt, window=window, n_splits=ns)
        gu.assert_attention_close(out, _oracle(orc, 0, q, lens, pt, window=window),
                                  f"window {window} n_splits {ns}")


def test_split_equals_single_pass_tiny_workload():
    """genie-ai-runtime v1.3.0: split-K is exact against the single-block kernel.
    The tiny workload (512 positions, GQA 4): n_splits 4 against 1."""
    w = inputs.tiny()
    pt, n_pages = inputs.page_table([512], 64)
    dev, orc = gu.make_pools(1, 2, 128, 128, 64, n_pages, 0)
    gu.fill_sequence(dev, orc, 0, w["k"], w["v"], pt[0])
    one = _decode(dev, 0, w["q"], [512], pt, n_splits=1)
    four = _decode(dev, 0, w["q"], [512], pt, n_splits=4)
    assert np.max(np.abs(one - four)) <= 1e-6
    gu.assert_attention_close(four, _oracle(orc, 0, w["q"], [512], pt), "tiny")


def test_context_one_returns_the_dequantized_v_row():
    q, pt, dev, orc = _setup(31, 2, 16, 2, 256, 64, [1, 1], 0)
    out = _decode(dev, 0, q, [1, 1], pt, n_splits=1)
    for b in range(2):
        _, vh = orc.gather(0, pt[b].numpy(), 1)
        for h in range(16):
            assert np.array_equal(out[b, h].astype(np.float64), vh[0, h // 8])


def test_identical_keys_return_the_mean_of_v():
    from int8_kv_cache_02_gb300 import binding
    L, Hkv, D = 300, 2, 128
    g = torch.Generator().manual_seed(41)
    k = inputs.normal_f16((1, Hkv, D), g).expand(L, Hkv, D).contiguous()
    v = inputs.normal_f16((L, Hkv, D), g)
    q = inputs.normal_f16((1, 8, D), g)
    pt, n_pages = inputs.page_table([L], 64, seed=2)
    dev, orc = gu.make_pools(1, Hkv, D, 128, 64, n_pages, 0)
    gu.fill_sequence(dev, orc, 0, k, v, pt[0])
    out = _decode(dev, 0, q, [L], pt, n_splits=3)
    _, vh = orc.gather(0, pt[0].numpy(), L)
    for h in range(8):
        assert np.allclose(out[0, h], vh[:, h // 4].mean(axis=0), rtol=0, atol=2e-6)
    assert binding.kv_pool_read_device_error(dev) == 0


def test_empty_sequences_give_zero_rows():
    q, pt, dev, orc = _setup(51, 3, 8, 2, 128, 128, [0, 130, 0], 0)
    out = _decode(dev, 0, q, [0, 130, 0], pt, n_splits=4)
    assert (out[0] == 0).all() and (out[2] == 0).all()
    gu.assert_attention_close(out[1:2], _oracle(orc, 0, q[1:2], [130], pt[1:2]), "mid")


def test_paged_equals_contiguous_bitwise_and_workspace_reuse():
    L = 1000
    q, ks, vs = inputs.random_case(61, 1, 16, 2, 256, [L], outliers=True)
    res = []
    for seed in (None, 5):
        pt, n_pages = inputs.page_table([L], 64, n_pages_total=40, seed=seed)
        dev, orc = gu.make_pools(1, 2, 256, 64, 64, n_pages, 0)
        gu.fill_sequence(dev, orc, 0, ks[0], vs[0], pt[0], oracle=False)
        ws = dev.decode_workspace(1, 16, 6)
        a = _decode(dev, 0, q, [L], pt, n_splits=6, ws=ws)
        b = _decode(dev, 0, q, [L], pt, n_splits=6, ws=ws)        # same workspace again
        assert np.array_equal(a, b)
        res.append(a)
    assert np.array_equal(res[0], res[1])


def test_softmax_scale_override_and_second_layer():
    q, pt, dev, orc = _setup(71, 1, 8, 2, 128, 64, [400], 0, n_layers=2, layer=1)
    sc = 0.3
    out = _decode(dev, 1, q, [400], pt, n_splits=2, scale=sc)
    gu.assert_attention_close(out, _oracle(orc, 1, q, [400], pt, scale=sc), "scale")
    out0 = _decode(dev, 0, q, [400], pt, n_splits=2)            # layer 0 is empty: all codes 0
    assert np.isfinite(out0).all()


def test_length_beyond_the_page_table_is_clamped_and_flagged():
    from int8_kv_cache_02_gb300 import binding
    q, pt, dev, orc = _setup(81, 1, 8, 2, 128, 128, [128], 0)      # page table holds 2 pages
    out = _decode(dev, 0, q, [5000], pt, n_splits=2)
    assert binding.kv_pool_read_device_error(dev) & binding.DEVERR_LENGTH
    gu.assert_attention_close(out, _oracle(orc, 0, q, [128], pt), "clamped")


@pytest.mark.slow
def test_grouped8k_workload_with_append():
    """8192-position context, 64-value groups with outlier K channels: 8191 cached
    positions, the step appends the last token and decodes over all 8192."""
    from int8_kv_cache_02_gb300 import binding
    w = inputs.grouped8k()
    pt, n_pages = inputs.page_table([8192], 64, seed=7)
    dev, orc = gu.make_pools(1, 2, 256, 64, 64, n_pages, 0)
    gu.fill_sequence(dev, orc, 0, w["k"][:8191], w["v"][:8191], pt[0])
    binding.kv_quant_append(dev, 0, w["k"][8191:].reshape(1, 1, 2, 256).cuda(),
                            w["v"][8191:].reshape(1, 1, 2, 256).cuda(),
                            torch.tensor([8191], dtype=torch.int32, device="cuda"), pt.cuda())
    orc.append(0, w["k"][8191:].numpy()[None], w["v"][8191:].numpy()[None], [8191], pt.numpy())
    gu.regions_equal(dev, orc)
    ref = _oracle(orc, 0, w["q"], [8192], pt)
    for ns in (0, 1, 16):
        gu.assert_attention_close(_decode(dev, 0, w["q"], [8192], pt, n_splits=ns), ref,
                                  f"8k n_splits {ns}")


@pytest.mark.slow
@pytest.mark.parametrize("variant", [0, 1])
def test_long128k_workload(variant):
    w = inputs.long128k()
    L = 131072
    pt, n_pages = inputs.page_table([L], 64, seed=8)
    dev, orc = gu.make_pools(1, 2, 256, 64, 64, n_pages, variant)
    gu.fill_sequence(dev, orc, 0, w["k"], w["v"], pt[0])
    ref = _oracle(orc, 0, w["q"], [L], pt)
    gu.assert_attention_close(_decode(dev, 0, w["q"], [L], pt), ref, f"128k v{variant}")


# --------------------------------------------------------------------------------------
# Tensor-core path specifics (page size 64, head_dim 128/256, groups of >= 64 values)

@pytest.mark.parametrize("G", [1, 3, 5, 8])
@pytest.mark.parametrize("variant", [0, 1, 2])
def test_mma_path_head_counts(G, variant):
    Hkv = 2
    lens = [517, 64]
    q, pt, dev, orc = _setup(300 + G + 10 * variant, 2, G * Hkv, Hkv, 256, 64, lens, variant,
                             outliers=True)
    for ns in (1, 5):
        out = _decode(dev, 0, q, lens, pt, n_splits=ns)
        gu.assert_attention_close(out, _oracle(orc, 0, q, lens, pt), f"G={G} v={variant} ns={ns}")


@pytest.mark.parametrize("gs", [64, 128, 256])
def test_mma_path_group_sizes(gs):
    lens = [1000]
    q, pt, dev, orc = _setup(400 + gs, 1, 16, 2, 256, gs, lens, 0, outliers=True)
    out = _decode(dev, 0, q, lens, pt, n_splits=3)
    gu.assert_attention_close(out, _oracle(orc, 0, q, lens, pt), f"gs={gs}")


@pytest.mark.parametrize("vmag", [1e-6, 1e-3, 3e2, 6e4])
@pytest.mark.parametrize("variant", [0, 2])
def test_mma_path_value_magnitudes(vmag, variant):
    """V from 1e-6 (fp16 subnormal range) to 6e4 (near fp16 max): the P' range shift
    keeps the hi/lo weights normal whatever the V scale."""
    L, Hkv, D = 700, 2, 128
    g = torch.Generator().manual_seed(int(vmag * 1e6) % 1000 + variant)
    q = inputs.normal_f16((1, 8, D), g)
    k = inputs.normal_f16((L, Hkv, D), g)
    v = (torch.randn((L, Hkv, D), generator=g) * vmag).clamp(-65000, 65000).to(torch.float16)
    pt, n_pages = inputs.page_table([L], 64, seed=4)
    dev, orc = gu.make_pools(1, Hkv, D, 64, 64, n_pages, variant)
    gu.fill_sequence(dev, orc, 0, k, v, pt[0])
    ref = _oracle(orc, 0, q, [L], pt)
    for ns in (1, 4):
        gu.assert_attention_close(_decode(dev, 0, q, [L], pt, n_splits=ns) / vmag, ref / vmag,
                                  f"vmag {vmag}")


def test_mma_path_v_scales_growing_along_the_sequence():
    """V scales spanning 2^20 across positions, growing and shrinking, so the running
    power-of-two range of every warp is raised many times."""
    L, Hkv, D = 1024, 2, 256
    g = torch.Generator().manual_seed(77)
    q = inputs.normal_f16((1, 16, D), g)
    k = inputs.normal_f16((L, Hkv, D), g)
    ramp = torch.pow(2.0, torch.linspace(-12, 8, L)).roll(300)
    v = (torch.randn((L, Hkv, D), generator=g) * ramp[:, None, None]).to(torch.float16)
    pt, n_pages = inputs.page_table([L], 64, seed=5)
    dev, orc = gu.make_pools(1, Hkv, D, 64, 64, n_pages, 0)
    gu.fill_sequence(dev, orc, 0, k, v, pt[0])
    ref = _oracle(orc, 0, q, [L], pt)
    for ns in (1, 2, 7):
        gu.assert_attention_close(_decode(dev, 0, q, [L], pt, n_splits=ns), ref, f"ns {ns}")


@pytest.mark.parametrize("variant", [1, 2])
def test_mma_path_ignores_garbage_beyond_the_context(variant):
    """Slots past the sequence end of an fp16 store hold NaN / Inf bit patterns."""
    from int8_kv_cache_02_gb300 import binding
    L = 100
    q, pt, dev, orc = _setup(501, 1, 16, 2, 256, 64, [L], variant)
    store = dev.v_store if variant == 1 else dev.k_store
    raw = store.view(torch.int16)
    last = int(pt[0, 1])
    raw[0, last, :, L - 64:, :] = 0x7E00            # NaN in fp16, in the unwritten slots
    raw[0, last, :, 60 + L - 64:, :] = 0x7C00       # +Inf
    out = _decode(dev, 0, q, [L], pt, n_splits=1)
    assert np.isfinite(out).all()
    gu.assert_attention_close(out, _oracle(orc, 0, q, [L], pt), "garbage")
    assert binding.kv_pool_read_device_error(dev) == 0


@pytest.mark.slow
def test_batched_workload_full_size_every_sequence():
    """64 sequences of 1024..32768 positions (8 kv heads, head_dim 128, one scale per
    (position, kv head), pages of 64), two layers: layer 0 full context, layer 1 a
    512-position window.  The whole pool is built through the kernel; every
    sequence of both layers is checked against the oracle: its codes and scales
    bit for bit (SHA-256 of the position-major rows against the oracle's), and
    its attention output at the split count the library picks and at a single
    split.  The oracle runs in spawned worker processes, one sequence per job."""
    import concurrent.futures as cf
    import multiprocessing as mp
    import os

    from int8_kv_cache_02_gb300 import binding
    from tests import batched_oracle as bo
    lens, qs = inputs.batched_lengths_and_q()
    lens = [int(x) for x in lens]
    windows = {0: 0, 1: 512}
    workers = max(1, min(16, (os.cpu_count() or 2) - 1))
    one_thread = {k: "1" for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    saved = {k: os.environ.get(k) for k in one_thread}
    os.environ.update(one_thread)          # inherited by the workers only (spawned below)
    try:
        ex = cf.ProcessPoolExecutor(workers, mp_context=mp.get_context("spawn"))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    with ex:
        jobs = {(layer, b): ex.submit(bo.oracle_sequence, layer, b, L, windows[layer])
                for layer in (0, 1) for b, L in enumerate(lens)}
        pt, n_pages = inputs.page_table(lens, 64, seed=11)
        dev = binding.KVPool(2, 8, 128, 128, 64, n_pages, binding.K8V8)
        ptd = pt.cuda()
        zero = torch.zeros(1, dtype=torch.int32, device="cuda")
        for layer in (0, 1):
            for b, L in enumerate(lens):
                k, v = inputs.batched_kv(layer, b, L)
                binding.kv_quant_append(dev, layer, k.reshape(1, L, 8, 128).cuda(),
                                        v.reshape(1, L, 8, 128).cuda(), zero, ptd[b:b + 1])
        lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
        outs = {}
        for layer, window in windows.items():
            ns = binding.attn_decode_n_splits(dev, 64, window + 64 if window else pt.shape[1] * 64)
            for n in sorted({ns, 1}):
                out = torch.empty((64, 32, 128), dtype=torch.float32, device="cuda")
                binding.attn_decode_int8(dev, layer, qs[layer].cuda(), lens_d, ptd, out,
                                         dev.decode_workspace(64, 32, n), window=window,
                                         n_splits=n)
                torch.cuda.synchronize()
                outs[(layer, n)] = out.cpu().numpy()
        assert binding.kv_pool_read_device_error(dev) == 0
        for layer in (0, 1):
            kst, vst = dev.k_store[layer].cpu().numpy(), dev.v_store[layer].cpu().numpy()
            ksc, vsc = dev.k_scales[layer].cpu().numpy(), dev.v_scales[layer].cpu().numpy()
            for b, L in enumerate(lens):
                pos = np.arange(L)
                pages, slots = pt[b].numpy()[pos // 64], pos % 64
                got = bo.codes_digest(kst[pages, :, slots, :], ksc[pages, :, slots, :],
                                      vst[pages, :, slots, :], vsc[pages, :, slots, :])
                want, ref = jobs[(layer, b)].result()
                assert got == want, f"layer {layer} seq {b}: codes or scales differ"
                for (ly, n), out in outs.items():
                    if ly == layer:
                        gu.assert_attention_close(out[b], ref, f"layer {layer} seq {b} L {L} ns {n}")


@pytest.mark.parametrize("D,gs,ps,variant", [(256, 64, 64, 0), (128, 128, 64, 1), (256, 128, 64, 2),
                                             (64, 32, 16, 0)])
@pytest.mark.parametrize("window", [0, 100])
def test_decode_append_equals_append_then_decode(D, gs, ps, variant, window):
    """attn_decode_append_int8 (append fused into the decode kernel where the tensor-core
    path serves the shape) is bit-identical to kv_quant_append + attn_decode_int8."""
    from int8_kv_cache_02_gb300 import binding
    lens = [777, 64, 1, 300]
    B, H, Hkv = len(lens), 8, 2
    q, ks, vs = inputs.random_case(611 + D + variant, B, H, Hkv, D, lens, outliers=True)
    pt, n_pages = inputs.page_table(lens, ps, seed=21)
    outs, pools = [], []
    for fused in (False, True):
        dev, orc = gu.make_pools(1, Hkv, D, gs, ps, n_pages, variant)
        for b, L in enumerate(lens):
            if L > 1:
                gu.fill_sequence(dev, orc, 0, ks[b][:L - 1], vs[b][:L - 1], pt[b], oracle=False)
        kn = torch.stack([ks[b][L - 1] for b, L in enumerate(lens)]).cuda()   # [B][Hkv][D]
        vn = torch.stack([vs[b][L - 1] for b, L in enumerate(lens)]).cuda()
        lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
        ns = 4
        ws = dev.decode_workspace(B, H, ns)
        out = torch.full((B, H, D), float("nan"), dtype=torch.float32, device="cuda")
        if fused:
            binding.attn_decode_append_int8(dev, 0, q.cuda(), kn, vn, lens_d, pt.cuda(), out, ws,
                                            window=window, n_splits=ns)
        else:
            binding.kv_quant_append(dev, 0, kn[:, None].contiguous(), vn[:, None].contiguous(),
                                    lens_d - 1, pt.cuda())
            binding.attn_decode_int8(dev, 0, q.cuda(), lens_d, pt.cuda(), out, ws, window=window,
                                     n_splits=ns)
        torch.cuda.synchronize()
        assert binding.kv_pool_read_device_error(dev) == 0
        outs.append(out.cpu().numpy())
        pools.append(dev)
    assert np.array_equal(outs[0], outs[1])
    for name in ("k_store", "v_store", "k_scales", "v_scales"):
        a, b = getattr(pools[0], name), getattr(pools[1], name)
        assert (a is None and b is None) or torch.equal(a, b), name
    # and against the oracle
    orc = gu.opool.Pool(1, Hkv, D, gs, ps, n_pages, variant)
    for b, L in enumerate(lens):
        orc.append_contiguous(0, ks[b].numpy(), vs[b].numpy(), 0, pt[b].numpy())
    gu.assert_attention_close(outs[1], _oracle(orc, 0, q, lens, pt, window=window), "fused")


@pytest.mark.parametrize("D,gs,variant", [(256, 64, 0), (256, 256, 0), (128, 64, 0), (256, 64, 2)])
@pytest.mark.parametrize("ns", [4, 16])
def test_decode_append_rounds_ties_like_the_oracle(D, gs, variant, ns):
    """The fused append on rows of rounding ties (x / s = k + 1/2) and their fp16
    neighbours: the pool rows it writes equal the oracle's, byte for byte, with the
    new position the last row of a page issued at once or of one refilled later."""
    from int8_kv_cache_02_gb300 import binding
    lens = [2000, 129, 64, 1]
    B, H, Hkv = len(lens), 8, 2
    q, ks, vs = inputs.random_case(915 + D + gs + ns, B, H, Hkv, D, lens)
    kn = inputs.tie_rows(B * Hkv, D, gs, seed=D + gs).reshape(B, Hkv, D)
    vn = inputs.tie_rows(B * Hkv, D, gs, seed=D + gs + 5).reshape(B, Hkv, D)
    for b, L in enumerate(lens):
        ks[b][L - 1] = kn[b]
        vs[b][L - 1] = vn[b]
    pt, n_pages = inputs.page_table(lens, 64, seed=23)
    dev, orc = gu.make_pools(1, Hkv, D, gs, 64, n_pages, variant)
    for b, L in enumerate(lens):
        if L > 1:
            gu.fill_sequence(dev, orc, 0, ks[b][:L - 1], vs[b][:L - 1], pt[b])
    orc.append(0, kn[:, None].numpy(), vn[:, None].numpy(), [L - 1 for L in lens], pt.numpy())
    out = torch.empty((B, H, D), dtype=torch.float32, device="cuda")
    binding.attn_decode_append_int8(dev, 0, q.cuda(), kn.cuda(), vn.cuda(),
                                    torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                    pt.cuda(), out, dev.decode_workspace(B, H, ns), n_splits=ns)
    torch.cuda.synchronize()
    assert binding.kv_pool_read_device_error(dev) == 0
    gu.regions_equal(dev, orc)
    gu.assert_attention_close(out.cpu().numpy(), _oracle(orc, 0, q, lens, pt), "ties")


@pytest.mark.parametrize("n_splits", [2, 3, 5, 7, 8, 9, 13])
def test_split_counts_around_the_cluster_size(n_splits):
    """Up to 8 splits combine inside the kernel (one cluster, any size); more go through
    the combine kernel.  Cluster sizes that do not divide head_dim included."""
    lens = [1500, 700]
    q, pt, dev, orc = _setup(900 + n_splits, 2, 16, 2, 256, 64, lens, 0, outliers=True)
    out = _decode(dev, 0, q, lens, pt, n_splits=n_splits)
    gu.assert_attention_close(out, _oracle(orc, 0, q, lens, pt), f"n_splits {n_splits}")
    q, pt, dev, orc = _setup(950 + n_splits, 1, 8, 2, 128, 128, [900], 1)
    out = _decode(dev, 0, q, [900], pt, n_splits=n_splits)
    gu.assert_attention_close(out, _oracle(orc, 0, q, [900], pt), f"D128 n_splits {n_splits}")


@pytest.mark.parametrize("n_splits", [9, 16, 40, 100])
def test_many_splits_twice_on_one_workspace(n_splits):
    """More than 8 splits go through the combine kernel; a second call on the same
    workspace gives the same bits."""
    lens = [6000, 2500]
    q, pt, dev, orc = _setup(970 + n_splits, 2, 16, 2, 256, 64, lens, 0, outliers=True)
    ws = dev.decode_workspace(2, 16, n_splits)
    first = _decode(dev, 0, q, lens, pt, n_splits=n_splits, ws=ws)
    second = _decode(dev, 0, q, lens, pt, n_splits=n_splits, ws=ws)
    assert np.array_equal(first, second)
    from int8_kv_cache_02_gb300 import binding
    assert binding.kv_pool_read_device_error(dev) == 0
    gu.assert_attention_close(first, _oracle(orc, 0, q, lens, pt), f"n_splits {n_splits}")


def test_many_splits_on_a_grid_larger_than_the_gpu():
    """64 sequences x 8 kv heads x 16 splits: more blocks than the GPU holds at once,
    ragged lengths; the result matches the oracle."""
    g = torch.Generator().manual_seed(12)
    lens = torch.randint(1, 700, (64,), generator=g).tolist()
    q, pt, dev, orc = _setup(77, 64, 32, 8, 128, 128, lens, 0)
    out = _decode(dev, 0, q, lens, pt, n_splits=16)
    from int8_kv_cache_02_gb300 import binding
    assert binding.kv_pool_read_device_error(dev) == 0
    gu.assert_attention_close(out, _oracle(orc, 0, q, lens, pt), "combine kernel")


@pytest.mark.parametrize("D,gs,variant", [(256, 64, 0), (128, 128, 0), (256, 128, 1), (128, 64, 2)])
def test_every_decode_kernel_matches_the_oracle(D, gs, variant):
    """kv_pool_set_decode_kernel: each kernel that serves the pool gives the oracle's
    result; AUTO is the warp-level tensor-core kernel, bit for bit."""
    from int8_kv_cache_02_gb300 import binding
    lens = [700, 129, 64]
    q, pt, dev, orc = _setup(600 + D + gs + variant, 3, 16, 2, D, gs, lens, variant, outliers=True)
    ref = _oracle(orc, 0, q, lens, pt)
    kinds = [binding.DECODE_WARP_MMA, binding.DECODE_SIMT]
    outs = {}
    for kind in kinds:
        dev.set_decode_kernel(kind)
        for ns in (1, 5):
            out = _decode(dev, 0, q, lens, pt, n_splits=ns)
            gu.assert_attention_close(out, ref, f"kind {kind} ns {ns}")
            outs[(kind, ns)] = out
    dev.set_decode_kernel(binding.DECODE_AUTO)
    for ns in (1, 5):
        assert np.array_equal(_decode(dev, 0, q, lens, pt, n_splits=ns),
                              outs[(binding.DECODE_WARP_MMA, ns)])
    assert binding.kv_pool_read_device_error(dev) == 0


@pytest.mark.parametrize("row_len,n_splits", [(313, 1), (2500, 1), (2500, 4), (2048, 3)])
def test_page_table_rows_read_with_the_length_or_per_page(row_len, n_splits):
    """Page-table rows longer than the 256 entries a block reads whole with the length:
    the block's page ids are read page by page, and a block whose range holds more than
    256 pages reads the rest of them from memory when it refills.  Entries past the
    sequence's pages are never used."""
    from int8_kv_cache_02_gb300 import binding
    L = 20000   # 313 pages
    q, pt, dev, orc = _setup(1300 + row_len + n_splits, 1, 16, 2, 256, 64, [L], 0, outliers=True)
    wide = torch.zeros((1, row_len), dtype=torch.int32)
    wide[:, :pt.shape[1]] = pt
    out = _decode(dev, 0, q, [L], wide, n_splits=n_splits)
    assert binding.kv_pool_read_device_error(dev) == 0
    gu.assert_attention_close(out, _oracle(orc, 0, q, [L], pt), f"row {row_len} ns {n_splits}")


# --------------------------------------------------------------------------------------
# Query windows (attn_decode_multi_int8): q_len queries per sequence, causal within the
# window; the oracle is decode at each query's own length (a pinned prefill row).

@pytest.mark.parametrize("D,gs,variant,H,Hkv,q_len,n_splits", [
    (256, 64, 0, 16, 2, 1, 0),     # q_len 1: attn_decode_int8, bit for bit
    (256, 64, 0, 16, 2, 2, 0),     # G 8 x 2 queries: two column groups
    (256, 64, 0, 8, 2, 2, 4),      # G 4 x 2 queries: the 8 columns of one block
    (128, 128, 1, 8, 4, 4, 13),    # G 2 x 4 queries; fp16 V; the combine kernel
    (256, 64, 2, 16, 4, 3, 1),     # G 4 x 3 = 12 columns: groups of 8 and 4; fp16 K; one split
    (128, 64, 0, 32, 8, 4, 5),     # G 4 x 4: two column groups; a cluster of 5 splits
])
def test_query_window_matches_the_oracle(D, gs, variant, H, Hkv, q_len, n_splits):
    from int8_kv_cache_02_gb300 import binding
    lens = [700, 129, 3]           # the last: fewer positions than queries
    B = len(lens)
    q0, pt, dev, orc = _setup(1400 + D + q_len + variant, B, H, Hkv, D, gs, lens, variant,
                              outliers=True)
    g = torch.Generator().manual_seed(1450 + q_len)
    q = inputs.normal_f16((B, q_len, H, D), g)
    ns = n_splits or binding.attn_decode_n_splits(dev, B * (-(-q_len * (H // Hkv) // 8)),
                                                  pt.shape[1] * 64)
    ws = dev.decode_workspace(B * q_len, H, ns)
    out = torch.full((B, q_len, H, D), float("nan"), dtype=torch.float32, device="cuda")
    binding.attn_decode_multi_int8(dev, 0, q.cuda(), torch.tensor(lens, dtype=torch.int32,
                                                                   device="cuda"),
                                   pt.cuda(), out, ws, n_splits=ns)
    torch.cuda.synchronize()
    assert binding.kv_pool_read_device_error(dev) == 0
    got = out.cpu().numpy()
    ref = np.zeros((B, q_len, H, D))
    for b, L in enumerate(lens):
        kh, vh = orc.gather(0, pt[b].numpy(), L)
        for i in range(q_len):
            pos = L - q_len + i
            if pos >= 0:
                ref[b, i] = oatt.decode(q[b, i].numpy(), kh, vh, pos + 1)
    gu.assert_attention_close(got.reshape(B * q_len, H, D), ref.reshape(B * q_len, H, D),
                              f"window {q_len}")
    if q_len == 1:
        single = _decode(dev, 0, q[:, 0], lens, pt, n_splits=ns)
        assert np.array_equal(got[:, 0], single)


def test_query_window_needs_the_tensor_core_kernel():
    from int8_kv_cache_02_gb300 import binding
    q0, pt, dev, orc = _setup(1490, 1, 8, 2, 64, 64, [100], 0)     # head_dim 64: CUDA-core kernel
    q = torch.zeros((1, 2, 8, 64), dtype=torch.float16, device="cuda")
    out = torch.zeros((1, 2, 8, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(binding.Int8KVError) as e:
        binding.attn_decode_multi_int8(dev, 0, q, torch.tensor([100], dtype=torch.int32,
                                                                device="cuda"),
                                       pt.cuda(), out, dev.decode_workspace(2, 8, 4), n_splits=4)
    assert e.value.status == -6

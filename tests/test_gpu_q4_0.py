"""q4_0 on the GPU against the oracle: K and V both rotated by the normalised
FWHT and stored as Q4_0 (Strata pull request #2698, "Not in this PR": --kv q4_0
with the Hadamard rotation; rotate K and V before they are stored, the queries
before the scores and the output back).

Codes and scales must equal the oracle's bit for bit; attention outputs must be
within the usual tolerance of the oracle's fp64 attention over the dequantized
cache rotated back (the oracle never rotates a query: the transform is
orthonormal, so its scores are the rotated ones).
"""

import numpy as np
import pytest
import torch

from int8_kv_cache_02_gb300 import inputs
from oracle import attention as oatt
from oracle import image as oimage
from tests import gpu_util as gu
from tests.test_gpu_k8v4 import _tricky_rows

pytestmark = pytest.mark.gpu

Q4_0 = 4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gu.lib_ready()


@pytest.mark.parametrize("D,gs", [(256, 64), (128, 128), (64, 32)])
def test_append_is_bit_exact(D, gs):
    from int8_kv_cache_02_gb300 import binding
    lens = [333, 64, 1]
    pt, n_pages = inputs.page_table(lens, 64, seed=12, n_pages_total=9)
    dev, orc = gu.make_pools(2, 2, D, gs, 64, n_pages, Q4_0)
    for layer in range(2):
        for b, L in enumerate(lens):
            k = _tricky_rows(L, 2, D, 20 * layer + b)
            v = _tricky_rows(L, 2, D, 200 + 20 * layer + b)
            gu.fill_sequence(dev, orc, layer, k, v, pt[b])
    gu.regions_equal(dev, orc)
    assert binding.kv_pool_read_device_error(dev) == 0


def _decode(dev, q, lens, pt, n_splits, window=0, kind=0):
    from int8_kv_cache_02_gb300 import binding
    dev.set_decode_kernel(kind)
    B, H, D = q.shape
    out = torch.full((B, H, D), float("nan"), dtype=torch.float32, device="cuda")
    binding.attn_decode_int8(dev, 0, q.cuda(), torch.tensor(lens, dtype=torch.int32, device="cuda"),
                             pt.cuda(), out, dev.decode_workspace(B, H, n_splits), window=window,
                             n_splits=n_splits)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("D,gs,H,Hkv", [(256, 64, 16, 2), (128, 128, 8, 2), (64, 32, 12, 4),
                                        (128, 64, 32, 8), (256, 32, 12, 4), (256, 256, 8, 8)])
@pytest.mark.parametrize("n_splits", [1, 4, 16])
def test_decode_matches_oracle(D, gs, H, Hkv, n_splits):
    from int8_kv_cache_02_gb300 import binding
    lens = [1500, 130, 1]
    q, ks, vs = inputs.random_case(500 + D + H, len(lens), H, Hkv, D, lens, outliers=(D == 256))
    pt, n_pages = inputs.page_table(lens, 64, seed=15)
    dev, orc = gu.make_pools(1, Hkv, D, gs, 64, n_pages, Q4_0)
    for b in range(len(lens)):
        gu.fill_sequence(dev, orc, 0, ks[b], vs[b], pt[b])
    # head_dim 256: the tensor-core kernel (AUTO) and the CUDA-core one; else CUDA cores
    kinds = [binding.DECODE_AUTO, binding.DECODE_SIMT] if D == 256 else [binding.DECODE_AUTO]
    for window in (0, 200):
        ref = np.stack([oatt.decode(q[b].numpy(), *orc.gather(0, pt[b].numpy(), L), L, window=window)
                        for b, L in enumerate(lens)])
        for kind in kinds:
            got = _decode(dev, q, lens, pt, n_splits, window, kind)
            gu.assert_attention_close(got, ref, f"q4_0 D{D} H{H} ns{n_splits} w{window} kind{kind}")
    assert binding.kv_pool_read_device_error(dev) == 0


@pytest.mark.parametrize("D", [128, 256])
def test_closed_forms(D):
    """Context 1 returns the stored V row (rotated back); identical keys give the
    mean of the stored V rows, whatever the query."""
    from int8_kv_cache_02_gb300 import binding
    H, Hkv = 4, 1
    g = torch.Generator().manual_seed(9)
    k_row = inputs.normal_f16((1, Hkv, D), g)
    ks = k_row.expand(40, Hkv, D).contiguous()
    vs = inputs.normal_f16((40, Hkv, D), g)
    q = inputs.normal_f16((1, H, D), g)
    pt, n_pages = inputs.page_table([40], 64, seed=3)
    dev, orc = gu.make_pools(1, Hkv, D, D, 64, n_pages, Q4_0)
    gu.fill_sequence(dev, orc, 0, ks, vs, pt[0])
    _, vh = orc.gather(0, pt[0].numpy(), 40)
    for L, want in ((1, vh[0, 0]), (40, vh[:, 0].mean(axis=0))):
        got = _decode(dev, q, [L], pt, 1)
        gu.assert_attention_close(got[0], np.broadcast_to(want, (H, D)), f"q4_0 closed form L{L}")
    assert binding.kv_pool_read_device_error(dev) == 0


def test_fused_step_and_image_round_trip():
    """attn_decode_append_int8 on a q4_0 pool equals kv_quant_append followed by
    attn_decode_int8 (bits of the pool and of the output), and a saved image of the
    pool is the oracle's byte for byte and reloads to the same regions."""
    from int8_kv_cache_02_gb300 import binding
    lens = [900, 257]
    q, ks, vs = inputs.random_case(604, 2, 16, 2, 256, lens, outliers=True, extra_pos=1)
    pt, n_pages = inputs.page_table([L + 1 for L in lens], 64, seed=18)
    a_dev, a_orc = gu.make_pools(1, 2, 256, 64, 64, n_pages, Q4_0)
    b_dev, _ = gu.make_pools(1, 2, 256, 64, 64, n_pages, Q4_0)
    for b, L in enumerate(lens):
        for d in (a_dev, b_dev):
            gu.fill_sequence(d, a_orc if d is a_dev else None, 0, ks[b][:L], vs[b][:L], pt[b],
                             oracle=d is a_dev)
    k_new = torch.stack([ks[b][L] for b, L in enumerate(lens)]).cuda()
    v_new = torch.stack([vs[b][L] for b, L in enumerate(lens)]).cuda()
    lens1 = [L + 1 for L in lens]
    lens_d = torch.tensor(lens1, dtype=torch.int32, device="cuda")
    out_a = torch.empty((2, 16, 256), dtype=torch.float32, device="cuda")
    binding.attn_decode_append_int8(a_dev, 0, q.cuda(), k_new, v_new, lens_d, pt.cuda(), out_a,
                                    a_dev.decode_workspace(2, 16, 8), n_splits=8)
    binding.kv_quant_append(b_dev, 0, k_new[:, None], v_new[:, None],
                            torch.tensor(lens, dtype=torch.int32, device="cuda"), pt.cuda())
    out_b = torch.empty_like(out_a)
    binding.attn_decode_int8(b_dev, 0, q.cuda(), lens_d, pt.cuda(), out_b,
                             b_dev.decode_workspace(2, 16, 8), n_splits=8)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    for b, L in enumerate(lens):
        a_orc.append(0, k_new[b][None, None].cpu().numpy(), v_new[b][None, None].cpu().numpy(), [L],
                     pt[b:b + 1].numpy())
    gu.regions_equal(a_dev, a_orc)
    ref = np.stack([oatt.decode(q[b].numpy(), *a_orc.gather(0, pt[b].numpy(), L), L)
                    for b, L in enumerate(lens1)])
    gu.assert_attention_close(out_a.cpu().numpy(), ref, "fused q4_0 step")
    img = binding.kv_pool_save(a_dev, lens1, pt.cuda())
    assert img == oimage.save(a_orc, lens1, pt.numpy())
    c_dev, c_orc = gu.make_pools(1, 2, 256, 64, 64, n_pages, Q4_0)
    assert binding.kv_pool_load(c_dev, img, pt.cuda()) == lens1
    oimage.load(c_orc, img, pt.numpy())
    gu.regions_equal(c_dev, c_orc)


def test_q4_0_kernel_choice_and_refusals():
    """head_dim 256 decodes on the tensor-core kernel (a row of either store is one
    128-byte box); head_dim 128 only on the CUDA cores, which serve no query
    windows; the prefill chunk refuses q4_0 (UNSUPPORTED, not served another way)."""
    from int8_kv_cache_02_gb300 import binding
    dev, _ = gu.make_pools(1, 2, 256, 64, 64, 4, Q4_0)
    dev.set_decode_kernel(binding.DECODE_WARP_MMA)
    small, _ = gu.make_pools(1, 2, 128, 64, 64, 4, Q4_0)
    with pytest.raises(binding.Int8KVError):
        small.set_decode_kernel(binding.DECODE_WARP_MMA)
    q = torch.zeros((8, 16, 256), dtype=torch.float16, device="cuda")
    out = torch.zeros((8, 16, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(binding.Int8KVError) as e:
        binding.attn_prefill_chunk_int8(dev, 0, q, 0, torch.zeros(4, dtype=torch.int32,
                                                                  device="cuda"), out, None)
    assert e.value.status == -6
    qw = torch.zeros((1, 2, 16, 128), dtype=torch.float16, device="cuda")
    ow = torch.zeros((1, 2, 16, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(binding.Int8KVError) as e:
        binding.attn_decode_multi_int8(small, 0, qw, torch.tensor([10], dtype=torch.int32,
                                                                  device="cuda"),
                                       torch.zeros((1, 4), dtype=torch.int32, device="cuda"), ow,
                                       small.decode_workspace(2, 16, 1), n_splits=1)
    assert e.value.status == -6


@pytest.mark.parametrize("q_len,n_splits", [(3, 1), (2, 5), (4, 12)])
def test_query_windows_q4_0(q_len, n_splits):
    """Query windows over a q4_0 pool (tensor-core kernel): query i of a window at
    position L - q_len + i sees keys 0 .. L - q_len + i; every query is rotated."""
    from int8_kv_cache_02_gb300 import binding
    lens = [700, 90]
    B, H = 2, 16
    g = torch.Generator().manual_seed(80 + q_len)
    qw = inputs.normal_f16((B, q_len, H, 256), g)
    _, ks, vs = inputs.random_case(81 + q_len, B, H, 2, 256, lens, outliers=True)
    pt, n_pages = inputs.page_table(lens, 64, seed=19)
    dev, orc = gu.make_pools(1, 2, 256, 64, 64, n_pages, Q4_0)
    for b in range(B):
        gu.fill_sequence(dev, orc, 0, ks[b], vs[b], pt[b])
    out = torch.full((B, q_len, H, 256), float("nan"), dtype=torch.float32, device="cuda")
    binding.attn_decode_multi_int8(dev, 0, qw.cuda(), torch.tensor(lens, dtype=torch.int32,
                                                                     device="cuda"),
                                   pt.cuda(), out, dev.decode_workspace(B * q_len, H, n_splits),
                                   n_splits=n_splits)
    torch.cuda.synchronize()
    ref = np.zeros((B, q_len, H, 256))
    for b, L in enumerate(lens):
        kh, vh = orc.gather(0, pt[b].numpy(), L)
        for i in range(q_len):
            ref[b, i] = oatt.decode(qw[b, i].numpy(), kh, vh, L - q_len + i + 1)
    gu.assert_attention_close(out.cpu().numpy(), ref, f"q4_0 window {q_len}")
    assert binding.kv_pool_read_device_error(dev) == 0


@pytest.mark.slow
def test_grouped8k_workload_q4_0():
    """The 8K-context workload (16/2 heads, head_dim 256, outlier K channels) in a
    q4_0 pool: codes and scales bit-exact, decode within the tolerance at the
    library's split count."""
    from int8_kv_cache_02_gb300 import binding
    w = inputs.grouped8k()
    L = w["L"]
    pt, n = inputs.page_table([L], 64, seed=41)
    dev, orc = gu.make_pools(1, 2, 256, 64, 64, n, Q4_0)
    gu.fill_sequence(dev, orc, 0, w["k"], w["v"], pt[0])
    gu.regions_equal(dev, orc)
    ns = binding.attn_decode_n_splits(dev, 1, L)
    got = _decode(dev, w["q"], [L], pt, ns)
    ref = oatt.decode(w["q"][0].numpy(), *orc.gather(0, pt[0].numpy(), L), L)
    gu.assert_attention_close(got[0], ref, "q4_0 8K")

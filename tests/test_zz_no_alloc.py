"""The allocation-free decode entry point (attn_decode_int8_noalloc).

Callers that cannot allocate device memory where they decode use this entry
point: it keeps the split partials in a fixed scratch array inside the library
instead of a caller workspace.  These tests call it through the C ABI and check
that two calls in a row give the output of attn_decode_int8 (which takes a
workspace) within the attention tolerance of the other tests (2e-3 max abs,
1e-4 max rel-L2), and that an oversized request is refused.  The file is named
to be collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

from int8_kv_cache_02_gb300 import inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _case(L=3000, seed=901):
    q, ks, vs = inputs.random_case(seed, 2, 16, 2, 256, [L, L // 3], outliers=True)
    lens = [L, L // 3]
    pt, n_pages = inputs.page_table(lens, 64, seed=3)
    dev, orc = gu.make_pools(1, 2, 256, 64, 64, n_pages, 0)
    for b in range(2):
        gu.fill_sequence(dev, orc, 0, ks[b], vs[b], pt[b], oracle=False)
    return q.cuda(), torch.tensor(lens, dtype=torch.int32, device="cuda"), pt.cuda(), dev


def _raw_noalloc(L, dev, q, lens, pt, out, n_splits, window=0):
    return L.attn_decode_int8_noalloc(dev.handle, 0, ctypes.c_void_p(q.data_ptr()), q.shape[0],
                                      q.shape[1], ctypes.c_void_p(lens.data_ptr()),
                                      ctypes.c_void_p(pt.data_ptr()), pt.shape[1], window,
                                      ctypes.c_float(0.0), n_splits,
                                      ctypes.c_void_p(out.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("n_splits", [16, 0, 1])
def test_noalloc_matches_the_workspace_entry_point_on_two_calls(n_splits):
    from int8_kv_cache_02_gb300 import binding
    gu.lib_ready()
    L = binding.lib()
    q, lens, pt, dev = _case()
    ns = n_splits or binding.attn_decode_n_splits(dev, 2, pt.shape[1] * 64)
    ref = torch.empty((2, 16, 256), dtype=torch.float32, device="cuda")
    binding.attn_decode_int8(dev, 0, q, lens, pt, ref, dev.decode_workspace(2, 16, ns), n_splits=ns)
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full((2, 16, 256), float("nan"), dtype=torch.float32, device="cuda")
        assert _raw_noalloc(L, dev, q, lens, pt, out, n_splits) == 0
        torch.cuda.synchronize()
        gu.assert_attention_close(out.cpu().numpy(), ref.cpu().numpy().astype(np.float64),
                                  f"call {call}")
    assert binding.kv_pool_read_device_error(dev) == 0


def test_noalloc_refuses_a_workspace_beyond_its_scratch():
    from int8_kv_cache_02_gb300 import binding
    gu.lib_ready()
    L = binding.lib()
    # 64 sequences x 32 heads x 16 splits x 128 dims x 4 B = 16 MiB of partials > 4 MiB
    dev, _ = gu.make_pools(1, 8, 128, 128, 64, 64, 0)
    q = torch.zeros((64, 32, 128), dtype=torch.float16, device="cuda")
    lens = torch.full((64,), 64, dtype=torch.int32, device="cuda")
    pt = torch.zeros((64, 1), dtype=torch.int32, device="cuda")
    out = torch.zeros((64, 32, 128), dtype=torch.float32, device="cuda")
    assert _raw_noalloc(L, dev, q, lens, pt, out, 16) == -5          # INT8KV_ERR_CAPACITY
    assert binding.int8kv_status_string(-5).startswith("request exceeds")


def test_noalloc_windowed_auto_split_matches_the_workspace_entry_point():
    """With a sliding window and n_splits = 0 the split count is the one
    attn_decode_int8 picks for the same call (sized to the window, not to the
    page table), so the two entry points give the same bits."""
    from int8_kv_cache_02_gb300 import binding
    gu.lib_ready()
    L = binding.lib()
    q, lens, pt, dev = _case(L=9000, seed=902)
    ref = torch.empty((2, 16, 256), dtype=torch.float32, device="cuda")
    ns = binding.attn_decode_n_splits(dev, 2, 512 + 64)
    assert ns < binding.attn_decode_n_splits(dev, 2, pt.shape[1] * 64)
    binding.attn_decode_int8(dev, 0, q, lens, pt, ref, dev.decode_workspace(2, 16, ns), window=512)
    for call in range(2):
        out = torch.full((2, 16, 256), float("nan"), dtype=torch.float32, device="cuda")
        assert _raw_noalloc(L, dev, q, lens, pt, out, 0, window=512) == 0
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {call}"
    assert binding.kv_pool_read_device_error(dev) == 0


def test_noalloc_auto_split_fits_the_scratch():
    """n_splits = 0 on a batch whose heuristic split count would need more than
    the scratch: the call picks the best count that fits instead of refusing,
    and its output matches attn_decode_int8 at that count within the tolerance."""
    from int8_kv_cache_02_gb300 import binding
    gu.lib_ready()
    L = binding.lib()
    # 64 sequences, 32/8 heads, head_dim 128, page-table rows of 512 pages (the
    # shape of the 64-sequence batch, short contexts): the heuristic's count for
    # 32K positions needs far more than the 4 MiB scratch
    B, H, Hkv, D = 64, 32, 8, 128
    lens_l = [200 + 9 * b for b in range(B)]
    qh, ks, vs = inputs.random_case(903, B, H, Hkv, D, lens_l)
    pt, n_pages = inputs.page_table(lens_l, 64, seed=4, max_pages=512)
    dev, _ = gu.make_pools(1, Hkv, D, 128, 64, n_pages, 0)
    for b in range(B):
        gu.fill_sequence(dev, None, 0, ks[b], vs[b], pt[b], oracle=False)
    q, lens, ptd = qh.cuda(), torch.tensor(lens_l, dtype=torch.int32, device="cuda"), pt.cuda()
    ns_ws = binding.attn_decode_n_splits(dev, B, pt.shape[1] * 64)
    need = binding.attn_decode_workspace_bytes(B, H, Hkv, D, ns_ws)
    assert need > 4 << 20
    out = torch.full((B, H, D), float("nan"), dtype=torch.float32, device="cuda")
    assert _raw_noalloc(L, dev, q, lens, ptd, out, 0) == 0
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    fits = [n for n in range(1, 257)
            if binding.attn_decode_workspace_bytes(B, H, Hkv, D, n) <= 4 << 20]
    ref = torch.empty_like(out)
    ns = max(fits)
    binding.attn_decode_int8(dev, 0, q, lens, ptd, ref, dev.decode_workspace(B, H, ns), n_splits=ns)
    torch.cuda.synchronize()
    gu.assert_attention_close(out.cpu().numpy(), ref.cpu().numpy().astype(np.float64), "auto fit")
    assert binding.kv_pool_read_device_error(dev) == 0


def test_noalloc_in_a_captured_graph_as_lengths_grow():
    """After a warm call, a noalloc decode recorded into a CUDA graph replays with
    the lengths read on the device: each replay, after the host advances the
    lengths, matches the oracle's decode at those lengths."""
    from int8_kv_cache_02_gb300 import binding
    from oracle import attention as oatt
    gu.lib_ready()
    L = binding.lib()
    lens0 = [1200, 300]
    q, ks, vs = inputs.random_case(904, 2, 16, 2, 256, [x + 8 for x in lens0], outliers=True)
    pt, n_pages = inputs.page_table([x + 8 for x in lens0], 64, seed=5)
    dev, orc = gu.make_pools(1, 2, 256, 64, 64, n_pages, 0)
    for b in range(2):
        gu.fill_sequence(dev, orc, 0, ks[b], vs[b], pt[b])
    qd, ptd = q.cuda(), pt.cuda()
    lens = torch.tensor(lens0, dtype=torch.int32, device="cuda")
    out = torch.zeros((2, 16, 256), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        assert _raw_noalloc(L, dev, qd, lens, ptd, out, 8) == 0   # warm: the scratch address
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        assert _raw_noalloc(L, dev, qd, lens, ptd, out, 8) == 0
    for step in range(4):
        now = [x + 2 * step for x in lens0]
        lens.copy_(torch.tensor(now, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        ref = np.stack([oatt.decode(q[b].numpy(), *orc.gather(0, pt[b].numpy(), n), n)
                        for b, n in enumerate(now)])
        gu.assert_attention_close(out.cpu().numpy(), ref, f"replay {step}")
    assert binding.kv_pool_read_device_error(dev) == 0

"""Decode steps captured in a CUDA graph and replayed, on the GPU.

genie-ai-runtime v1.3.0 "Details" bakes the split count into a captured graph
and reads the position on the device.  Here the sequence lengths are read on
the device and the split count is fixed when the graph is captured, so one
captured run of steps (bump the lengths, append one token, decode) replays
correctly while the contexts grow: every step's output matches the oracle at
that step's length, and the appended codes and scales match the oracle's pool
bit for bit.
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


@pytest.mark.parametrize("D,gs,variant,n_splits", [
    (256, 64, 0, 0),      # int8 K and V, 64-value groups, the heuristic's split count
    (128, 128, 1, 5),     # fp16 V, per-(position, kv head) scales, one cluster of 5 splits
    (256, 64, 2, 12),     # fp16 K, 12 splits through the combine kernel
])
def test_captured_append_decode_steps_replay_as_lengths_grow(D, gs, variant, n_splits):
    from int8_kv_cache_02_gb300 import binding
    B, H, Hkv, S, R = 2, 16, 2, 4, 2          # S steps per graph, R replays
    L0 = [700, 130]
    total = [L + S * R for L in L0]
    seed = 1500 + D + variant
    _, ks, vs = inputs.random_case(seed, B, H, Hkv, D, total, outliers=True)
    g = torch.Generator().manual_seed(seed + 1)
    qs = inputs.normal_f16((R, S, B, H, D), g)
    pt, n_pages = inputs.page_table(total, 64, n_pages_total=sum(-(-L // 64) for L in total) + 2,
                                    seed=seed)
    dev, orc = gu.make_pools(1, Hkv, D, gs, 64, n_pages, variant)
    for b in range(B):
        gu.fill_sequence(dev, orc, 0, ks[b][:L0[b]], vs[b][:L0[b]], pt[b])

    ptd = pt.cuda()
    lens = torch.tensor(L0, dtype=torch.int32, device="cuda")
    ns = n_splits or binding.attn_decode_n_splits(dev, B, pt.shape[1] * 64)
    ws = dev.decode_workspace(B, H, ns)
    q_in = torch.zeros((S, B, H, D), dtype=torch.float16, device="cuda")
    k_in = torch.zeros((S, B, Hkv, D), dtype=torch.float16, device="cuda")
    v_in = torch.zeros((S, B, Hkv, D), dtype=torch.float16, device="cuda")
    out = torch.full((S, B, H, D), float("nan"), dtype=torch.float32, device="cuda")

    # one eager call on a scratch pool of the same shape sets the kernel's launch
    # attributes before the capture
    scratch, _ = gu.make_pools(1, Hkv, D, gs, 64, n_pages, variant)
    binding.attn_decode_int8(scratch, 0, q_in[0], lens, ptd, out[0], ws, n_splits=ns)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for s in range(S):
            lens.add_(1)                        # the new token sits at lens[b] - 1
            binding.attn_decode_append_int8(dev, 0, q_in[s], k_in[s], v_in[s], lens, ptd,
                                            out[s], ws, n_splits=ns)
    torch.cuda.synchronize()

    for r in range(R):
        for s in range(S):
            step = r * S + s
            q_in[s].copy_(qs[r, s])
            for b in range(B):
                k_in[s, b].copy_(ks[b][L0[b] + step])
                v_in[s, b].copy_(vs[b][L0[b] + step])
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert binding.kv_pool_read_device_error(dev) == 0
        got = out.cpu().numpy()
        for s in range(S):
            step = r * S + s
            ref = []
            for b in range(B):
                pos = L0[b] + step
                orc.append_contiguous(0, ks[b][pos:pos + 1].numpy(), vs[b][pos:pos + 1].numpy(),
                                      pos, pt[b].numpy())
                kh, vh = orc.gather(0, pt[b].numpy(), pos + 1)
                ref.append(oatt.decode(qs[r, s, b].numpy(), kh, vh, pos + 1))
            gu.assert_attention_close(got[s], np.stack(ref), f"replay {r} step {s}")
    assert lens.cpu().tolist() == total
    gu.regions_equal(dev, orc)

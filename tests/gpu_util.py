"""Helpers for the GPU parity tests: fill a device pool through the library and
the oracle's pool from the same fp16 inputs, and compare the results."""

import numpy as np
import torch

from oracle import pool as opool

ATOL = 2e-3      # max abs error of an fp32 attention output against the fp64 oracle
RTOL_L2 = 1e-4   # max relative L2 error per (sequence, query head) output vector


def lib_ready():
    from int8_kv_cache_02_gb300 import binding, build
    build.build()
    binding.lib()


def make_pools(n_layers, Hkv, D, gs, ps, n_pages, variant):
    from int8_kv_cache_02_gb300 import binding
    dev = binding.KVPool(n_layers, Hkv, D, gs, ps, n_pages, variant)
    orc = opool.Pool(n_layers, Hkv, D, gs, ps, n_pages, variant)
    return dev, orc


def fill_sequence(dev, orc, layer, k, v, page_row, start=0, chunk=16384, oracle=True):
    """Append fp16 K/V [n][Hkv][D] of one sequence at positions start.. on both pools."""
    from int8_kv_cache_02_gb300 import binding
    n = k.shape[0]
    pt = torch.as_tensor(np.asarray(page_row, np.int32)).reshape(1, -1).cuda()
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        kd = k[a:b].reshape(1, b - a, *k.shape[1:]).cuda()
        vd = v[a:b].reshape(1, b - a, *v.shape[1:]).cuda()
        pos = torch.tensor([start + a], dtype=torch.int32, device="cuda")
        binding.kv_quant_append(dev, layer, kd, vd, pos, pt)
    if oracle:
        orc.append_contiguous(layer, k.numpy(), v.numpy(), start, np.asarray(page_row))


def regions_equal(dev, orc):
    """Bit-exact comparison of every region of the two pools."""
    torch.cuda.synchronize()
    pairs = [(dev.k_store, orc.k_store), (dev.v_store, orc.v_store),
             (dev.k_scales, orc.k_scales), (dev.v_scales, orc.v_scales)]
    for d, o in pairs:
        if o is None:
            assert d is None
            continue
        dn = d.cpu().numpy()
        if dn.dtype == np.float16:
            dn, o = dn.view(np.uint16), o.view(np.uint16)
        if not np.array_equal(dn, o):
            bad = np.argwhere(dn != o)
            raise AssertionError(f"{bad.shape[0]} mismatches, first at {bad[0].tolist()}: "
                                 f"device {dn[tuple(bad[0])]} oracle {o[tuple(bad[0])]}")


def attention_errors(out, ref):
    """(max abs error, max relative L2 error per output vector) of fp32 `out` vs fp64 `ref`
    shaped [..., D].  A zero reference vector must be matched exactly."""
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = out - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    nd = np.linalg.norm(diff.reshape(-1, diff.shape[-1]), axis=1)
    nr = np.linalg.norm(ref.reshape(-1, ref.shape[-1]), axis=1)
    zero = nr == 0
    assert np.all(nd[zero] == 0), "nonzero output where the oracle gives 0"
    rel = float(np.max(nd[~zero] / nr[~zero])) if (~zero).any() else 0.0
    return max_abs, rel


def assert_attention_close(out, ref, what=""):
    ma, rl = attention_errors(out, ref)
    assert ma <= ATOL and rl <= RTOL_L2, f"{what}: max abs {ma:.3e}, max rel-L2 {rl:.3e}"
    return ma, rl

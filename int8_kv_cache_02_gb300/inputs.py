"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the method: it draws fp16 normal samples
and builds page tables.  Everything is drawn on the CPU from
``torch.Generator().manual_seed(seed)`` so that the oracle and the device see
the same bytes.  Draw order within a generator is fixed and documented below.

Workloads (decode over an INT8 KV cache; sizes are the ones the kernels are
measured on):

* ``tiny``      batch 1, 8 query heads, 2 kv heads, head_dim 128, 512 cached
                positions, one scale per (position, kv head); seed 0.
                Draws: q [1][8][128], K [512][2][128], V [512][2][128].
* ``grouped8k`` batch 1, 16 query heads, 2 kv heads, head_dim 256, one scale
                per 64 values, context 8192 = 8191 cached + 1 appended by the
                step; seed 1.  Draws: q [1][16][256], K [8192][2][256],
                V [8192][2][256], then per kv head ``randperm(256)[:4]``: those
                K channels are multiplied by 20 before the fp16 cast.
* ``long128k``  batch 1, 16/2 heads, head_dim 256, 64-value groups, context
                131072; seed 2; draws q, K, V as ``tiny`` (no outliers).
* ``batched``   batch 64, 32 query heads, 8 kv heads, head_dim 128, one scale
                per (position, kv head), pages of 64 positions, two layers
                (layer 1 uses a 512-position sliding window).  Seed 3 draws the
                lengths first: ``randint(1024, 32769, (64,))``, then q for
                layer 0 and layer 1 ([64][32][128] each).  K/V of (layer, seq b)
                come from their own generator, seed ``3_000_000 + 1000*layer + b``,
                drawing K [L_b][8][128] then V, so any sequence can be rebuilt
                alone.
* ``tie_rows``  rows whose every group of gs values has the absmax 127*s0 for
                an s0 = m * 2^e (m odd, < 8), so that the group's scale is s0
                exactly, and whose other values are +-(k + 1/2) * s0 (x / s a
                rounding tie) or one fp16 step away from it.
* ``prefill``   batch 1, 16/2 heads, head_dim 256, 64-value groups; 32768
                cached positions plus a causal chunk of 256 new queries; seed 4.
                Draws: q [256][16][256], K [33024][2][256], V, then the outlier
                channels as in ``grouped8k``.
"""

import torch

F16 = torch.float16


def normal_f16(shape, gen):
    """N(0, 1) samples drawn in fp32 from ``gen`` and rounded to fp16."""
    return torch.randn(shape, dtype=torch.float32, generator=gen).to(F16)


def _outlier_channels(x32, n_kv_heads, head_dim, gen, n_out=4, factor=20.0):
    for h in range(n_kv_heads):
        ch = torch.randperm(head_dim, generator=gen)[:n_out]
        x32[:, h, ch] *= factor
    return x32


def kv_with_outliers(n_pos, n_kv_heads, head_dim, gen):
    """K with 4 outlier channels per kv head (x20), V plain; both fp16."""
    k32 = torch.randn((n_pos, n_kv_heads, head_dim), dtype=torch.float32, generator=gen)
    v = normal_f16((n_pos, n_kv_heads, head_dim), gen)
    k = _outlier_channels(k32, n_kv_heads, head_dim, gen).to(F16)
    return k, v


def page_table(lengths, page_size, n_pages_total=None, seed=None, max_pages=None):
    """Page table int32 [B][max_pages]: sequence b's logical page p -> physical id.

    Physical ids are a seeded permutation of 0..sum(pages)-1 when ``seed`` is
    given (exercises the paging), else consecutive.  Unused entries are -1.
    """
    need = [-(-int(L) // page_size) for L in lengths]
    total = sum(need)
    n_pages_total = total if n_pages_total is None else n_pages_total
    assert n_pages_total >= total
    if seed is None:
        ids = torch.arange(total, dtype=torch.int32)
    else:
        g = torch.Generator().manual_seed(seed)
        ids = torch.randperm(n_pages_total, generator=g)[:total].to(torch.int32)
    mp = max(max(need), 1) if max_pages is None else max_pages
    pt = torch.full((len(lengths), mp), -1, dtype=torch.int32)
    o = 0
    for b, n in enumerate(need):
        pt[b, :n] = ids[o:o + n]
        o += n
    return pt, n_pages_total


def tiny():
    g = torch.Generator().manual_seed(0)
    q = normal_f16((1, 8, 128), g)
    k = normal_f16((512, 2, 128), g)
    v = normal_f16((512, 2, 128), g)
    return dict(name="tiny", B=1, H=8, Hkv=2, D=128, gs=128, L=512, q=q, k=k, v=v)


def grouped8k():
    g = torch.Generator().manual_seed(1)
    q = normal_f16((1, 16, 256), g)
    k32 = torch.randn((8192, 2, 256), dtype=torch.float32, generator=g)
    v = normal_f16((8192, 2, 256), g)
    k = _outlier_channels(k32, 2, 256, g).to(F16)
    return dict(name="grouped8k", B=1, H=16, Hkv=2, D=256, gs=64, L=8192, q=q, k=k, v=v)


def long128k():
    g = torch.Generator().manual_seed(2)
    q = normal_f16((1, 16, 256), g)
    k = normal_f16((131072, 2, 256), g)
    v = normal_f16((131072, 2, 256), g)
    return dict(name="long128k", B=1, H=16, Hkv=2, D=256, gs=64, L=131072, q=q, k=k, v=v)


def batched_lengths_and_q():
    g = torch.Generator().manual_seed(3)
    lens = torch.randint(1024, 32769, (64,), generator=g)
    q = [normal_f16((64, 32, 128), g) for _ in range(2)]
    return lens, q


def batched_kv(layer, b, length):
    g = torch.Generator().manual_seed(3_000_000 + 1000 * layer + b)
    k = normal_f16((length, 8, 128), g)
    v = normal_f16((length, 8, 128), g)
    return k, v


def prefill():
    g = torch.Generator().manual_seed(4)
    q = normal_f16((256, 16, 256), g)
    k32 = torch.randn((33024, 2, 256), dtype=torch.float32, generator=g)
    v = normal_f16((33024, 2, 256), g)
    k = _outlier_channels(k32, 2, 256, g).to(F16)
    return dict(name="prefill", H=16, Hkv=2, D=256, gs=64, start=32768, n_new=256,
                q=q, k=k, v=v)


def random_case(seed, B, H, Hkv, D, lengths, outliers=False, extra_pos=0):
    """Generic small case: q [B][H][D], per-sequence K/V [L_b + extra_pos][Hkv][D]."""
    g = torch.Generator().manual_seed(seed)
    q = normal_f16((B, H, D), g)
    ks, vs = [], []
    for L in lengths:
        n = int(L) + extra_pos
        if outliers:
            k, v = kv_with_outliers(n, Hkv, D, g)
        else:
            k = normal_f16((n, Hkv, D), g)
            v = normal_f16((n, Hkv, D), g)
        ks.append(k)
        vs.append(v)
    return q, ks, vs


def tie_rows(n_rows, D, gs, seed):
    """fp16 [n_rows][D] of values on and next to the code rounding boundaries.

    Group (row, j): s0 = m * 2^e, m in {1, 3, 5, 7}, e in [-20, 4]; one value is
    +-127*s0, every other one +-(k + 1/2)*s0 with k in [0, 126], two thirds of them
    moved one fp16 step up or down.  All of these are exact fp16 values: (2k+1)*m
    < 2^11 and the smallest, 2^-21, is a multiple of the subnormal step 2^-24.
    """
    g = torch.Generator().manual_seed(seed)
    ng = D // gs
    m = torch.tensor([1, 3, 5, 7])[torch.randint(0, 4, (n_rows, ng), generator=g)]
    e = torch.randint(-20, 5, (n_rows, ng), generator=g)
    s0 = m.double() * torch.pow(2.0, e.double())                       # [rows][ng]
    k = torch.randint(0, 127, (n_rows, ng, gs), generator=g).double()
    sign = torch.randint(0, 2, (n_rows, ng, gs), generator=g).double() * 2 - 1
    x = sign * (k + 0.5) * s0[..., None]
    top = torch.randint(0, gs, (n_rows, ng), generator=g)
    x.scatter_(2, top[..., None], (sign.gather(2, top[..., None]) * 127.0) * s0[..., None])
    bits = x.to(F16).view(torch.int16)
    step = torch.randint(-1, 2, (n_rows, ng, gs), generator=g).to(torch.int16)
    step.scatter_(2, top[..., None], torch.zeros((n_rows, ng, 1), dtype=torch.int16))
    return (bits + step).view(F16).reshape(n_rows, D)

"""Oracle side of the full-size batched-pool parity test, one sequence per call,
run in worker processes (test infrastructure only).

For (layer, sequence b) of the 64-sequence workload (8 kv heads, head_dim 128,
one scale per (position, kv head), layer 1 with a 512-position window) it
rebuilds the sequence's fp16 K/V from their own seed, quantizes them with the
oracle, and returns a SHA-256 digest of the codes and scales (bytes in
position-major [L][8][128] and [L][8][1] order, K then V) together with the
oracle's fp64 decode output.
"""

import hashlib

import numpy as np


def codes_digest(kc, ks, vc, vs):
    h = hashlib.sha256()
    for a in (kc, ks, vc, vs):
        a = np.ascontiguousarray(a)
        h.update(a.view(np.uint16).tobytes() if a.dtype == np.float16 else a.tobytes())
    return h.hexdigest()


def oracle_sequence(layer, b, L, window):
    import torch

    from int8_kv_cache_02_gb300 import inputs
    torch.set_num_threads(1)
    from oracle import attention as oatt
    from oracle import quant
    k, v = inputs.batched_kv(layer, b, L)
    _, qs = inputs.batched_lengths_and_q()
    kc, ks = quant.quantize(k.numpy(), 128)
    vc, vs = quant.quantize(v.numpy(), 128)
    ref = oatt.decode(qs[layer][b].numpy(), quant.dequantize(kc, ks, 128),
                      quant.dequantize(vc, vs, 128), L, window=window)
    return codes_digest(kc, ks, vc, vs), ref

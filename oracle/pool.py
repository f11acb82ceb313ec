"""Oracle: the paged KV pool with a separate scales region (test infrastructure only).

The genie-ai-runtime INT8 KV cache (release v0.1.0-alpha.12, "Path I series",
row I1) keeps the int8 K/V body in the pool and the per-head scales in a
separate region allocated only in INT8 mode; the attention finds the scale of
a cached row by (position, kv head) (row I3).  Strata pull request #2698
("What it does") keeps one store per tensor (K and V) and lets either be int8
or full precision (``k8v8``, ``k8v32``, ``k32v8``); here the full-precision
store is fp16 (variants k8v8, k8v16, k16v8).

Layout (the device pool uses the same one, so bytes compare directly):

  int8 store   codes  int8 [n_layers][n_pages][n_kv_heads][page_size][head_dim]
  fp16 store   values fp16 [n_layers][n_pages][n_kv_heads][page_size][head_dim]
  scales       fp16        [n_layers][n_pages][n_kv_heads][page_size][head_dim // gs]
               (present only for an int8 store)

Position ``p`` of a sequence lives on physical page ``page_table[p // page_size]``
at slot ``p % page_size``.
"""

import numpy as np

from . import q4, quant

K8V8, K8V16, K16V8, K8V4, Q4_0 = 0, 1, 2, 3, 4
VARIANT_NAMES = {K8V8: "k8v8", K8V16: "k8v16", K16V8: "k16v8", K8V4: "k8v4", Q4_0: "q4_0"}


def store_is_int8(variant: int):
    """(K is int8, V is int8) for a store variant (k8v4: K int8, V 4-bit; q4_0: both 4-bit)."""
    return {K8V8: (True, True), K8V16: (True, False), K16V8: (False, True),
            K8V4: (True, False), Q4_0: (False, False)}[variant]


def store_is_q4(variant: int):
    """(K is 4-bit, V is 4-bit) for a store variant."""
    return {K8V4: (False, True), Q4_0: (True, True)}.get(variant, (False, False))


def bytes_per_cell(n_kv_heads: int, head_dim: int, gs: int, int8: bool) -> int:
    """Bytes one position occupies in one store (K or V) over all kv heads.

    int8: one code per value plus one 2-byte scale per group; fp16: 2 bytes per
    value.  (Strata #2698 quotes 528 B/cell at head_dim 256 with 2 kv heads and
    64-value groups, against 2048 B for its fp32 store.)
    """
    if int8:
        return n_kv_heads * head_dim + n_kv_heads * (head_dim // gs) * 2
    return n_kv_heads * head_dim * 2


class Pool:
    """Host model of the paged pool; arrays are the raw regions.

    k8v4 (Strata pull request #2698, "Not in this PR": the 4-bit store with the
    FWHT-256 rotation, see oracle/q4.py): V rows are rotated, then Q4_0; the V
    store is uint8 [..., head_dim / 2] (two codes per byte) and the V scales
    fp16 [..., head_dim / 32].  q4_0 (the same page's --kv q4_0): K and V both.
    gather returns rows rotated back in fp64, so attention over them is
    attention with the rotated queries over the rotated keys (the rotation is
    orthonormal)."""

    def __init__(self, n_layers, n_kv_heads, head_dim, gs, page_size, n_pages, variant):
        assert head_dim % gs == 0
        self.n_layers, self.n_kv_heads, self.head_dim = n_layers, n_kv_heads, head_dim
        self.gs, self.ng = gs, head_dim // gs
        self.page_size, self.n_pages, self.variant = page_size, n_pages, variant
        self.k_int8, self.v_int8 = store_is_int8(variant)
        self.k_q4, self.v_q4 = store_is_q4(variant)
        body = (n_layers, n_pages, n_kv_heads, page_size, head_dim)
        sc = (n_layers, n_pages, n_kv_heads, page_size, self.ng)
        self.k_store = np.zeros(body, np.int8 if self.k_int8 else np.float16)
        self.v_store = np.zeros(body, np.int8 if self.v_int8 else np.float16)
        self.k_scales = np.zeros(sc, np.float16) if self.k_int8 else None
        self.v_scales = np.zeros(sc, np.float16) if self.v_int8 else None
        if self.k_q4 or self.v_q4:
            assert head_dim % q4.BLOCK == 0 and head_dim & (head_dim - 1) == 0
        if self.k_q4:
            self.k_store = np.zeros(body[:-1] + (head_dim // 2,), np.uint8)
            self.k_scales = np.zeros(body[:-1] + (head_dim // q4.BLOCK,), np.float16)
        if self.v_q4:
            self.v_store = np.zeros(body[:-1] + (head_dim // 2,), np.uint8)
            self.v_scales = np.zeros(body[:-1] + (head_dim // q4.BLOCK,), np.float16)

    def _slot(self, page_table_row, pos):
        return int(page_table_row[pos // self.page_size]), pos % self.page_size

    def append(self, layer, k_new, v_new, seq_pos, page_table):
        """Quantize and write new tokens.

        k_new, v_new: fp16 [n_seqs][n_new][n_kv_heads][head_dim]; token i of
        sequence b goes to position seq_pos[b] + i.  page_table: int [n_seqs][max_pages].
        """
        k_new = np.asarray(k_new, np.float16)
        v_new = np.asarray(v_new, np.float16)
        n_seqs, n_new = k_new.shape[:2]
        for b in range(n_seqs):
            for i in range(n_new):
                page, slot = self._slot(page_table[b], int(seq_pos[b]) + i)
                for new, store, scales, is8, is4 in (
                    (k_new, self.k_store, self.k_scales, self.k_int8, self.k_q4),
                    (v_new, self.v_store, self.v_scales, self.v_int8, self.v_q4),
                ):
                    x = new[b, i]                              # [n_kv_heads][head_dim]
                    if is4:
                        c, s = q4.quantize_rows(x)
                        store[layer, page, :, slot, :] = c
                        scales[layer, page, :, slot, :] = s
                    elif is8:
                        c, s = quant.quantize(x, self.gs)
                        store[layer, page, :, slot, :] = c
                        scales[layer, page, :, slot, :] = s
                    else:
                        store[layer, page, :, slot, :] = x

    def append_contiguous(self, layer, k_seq, v_seq, start, page_table_row):
        """Vectorised append of one sequence's tokens start..start+n-1.

        Same result as ``append`` with one sequence; k_seq, v_seq: fp16
        [n][n_kv_heads][head_dim].
        """
        k_seq = np.asarray(k_seq, np.float16)
        v_seq = np.asarray(v_seq, np.float16)
        n = k_seq.shape[0]
        pos = np.arange(start, start + n)
        pages = np.asarray(page_table_row)[pos // self.page_size]
        slots = pos % self.page_size
        for x, store, scales, is8, is4 in (
            (k_seq, self.k_store, self.k_scales, self.k_int8, self.k_q4),
            (v_seq, self.v_store, self.v_scales, self.v_int8, self.v_q4),
        ):
            if is4:
                c, s = q4.quantize_rows(x)
                store[layer, pages, :, slots, :] = c
                scales[layer, pages, :, slots, :] = s
            elif is8:
                c, s = quant.quantize(x, self.gs)
                store[layer, pages, :, slots, :] = c
                scales[layer, pages, :, slots, :] = s
            else:
                store[layer, pages, :, slots, :] = x

    def gather(self, layer, page_table_row, length):
        """Exact fp64 K^, V^ [length][n_kv_heads][head_dim] of positions 0..length-1."""
        return self.gather_range(layer, page_table_row, 0, length)

    def gather_range(self, layer, page_table_row, start, stop):
        """Exact fp64 K^, V^ [stop-start][n_kv_heads][head_dim] of positions start..stop-1."""
        pos = np.arange(start, stop)
        pages = np.asarray(page_table_row)[pos // self.page_size] if stop > start else np.zeros(0, int)
        slots = pos % self.page_size
        out = []
        for store, scales, is8, is4 in (
            (self.k_store, self.k_scales, self.k_int8, self.k_q4),
            (self.v_store, self.v_scales, self.v_int8, self.v_q4),
        ):
            rows = store[layer, pages, :, slots, :]             # [L][Hkv][D]
            if is4:   # dequantized and rotated back to the original basis
                out.append(q4.dequantize_rows(rows, scales[layer, pages, :, slots, :]))
            elif is8:
                out.append(quant.dequantize(rows, scales[layer, pages, :, slots, :], self.gs))
            else:
                out.append(rows.astype(np.float64))
        return out[0], out[1]

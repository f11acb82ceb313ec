"""Oracle: the saved image of a pool's used positions, codes and scales together
(test infrastructure only).

genie-ai-runtime release v0.1.0-alpha.12 ("Path F (#45) interop guard", and
"Not in this release") records that its persistent-KV format v2 (F4a) stored
the int8 bytes without the per-head scales that attention needs when a cache
is hydrated again, so int8 saves had to be skipped; format v3 (#67) is to
persist the scales region as well.  Release v0.1.0-alpha.11 ("--int8-kv
triage", the list of what a proper fix needs) says the same: save/load must
persist the scales region too, or refuse caches whose int8 setting differs.
The Path F table of alpha.10 adds that a save packs only the used tokens
(F3b).  The byte layout below is this library's own; the pages fix only what
it must carry.

Image layout (little-endian; every section starts on a 16-byte boundary):

  header, 48 bytes:
     0  4 bytes  magic b"I8KV"
     4  u32      format version, 3
     8  u32      store variant (0 k8v8, 1 k8v16, 2 k16v8, 3 k8v4, 4 q4_0)
    12  u32      n_layers
    16  u32      n_kv_heads
    20  u32      head_dim
    24  u32      group_size
    28  u32      n_seqs
    32  u64      payload bytes (everything after the lengths)
    40  u64      0
  lengths: int32 [n_seqs], padded with zeros to a multiple of 16 bytes
  payload: for each sequence b, for each layer l, four sections (the scales
  sections only for a quantized store), each padded with zeros to 16 bytes:
     K store   [L_b][n_kv_heads][head_dim]  int8 codes or fp16 values  (q4_0: as V of k8v4)
     V store   [L_b][n_kv_heads][head_dim]  (k8v4: [head_dim / 2] bytes of 4-bit codes)
     K scales  [L_b][n_kv_heads][head_dim / group_size] fp16
     V scales  [L_b][n_kv_heads][head_dim / group_size] fp16  (k8v4: [head_dim / 32])

The payload is position-major, so an image does not depend on the page size
or the physical pages of the pool it came from: it can be loaded into any
pool of the same variant and shape, through any page table.
"""

import struct

import numpy as np

MAGIC = b"I8KV"
VERSION = 3
HEADER = struct.Struct("<4sIIIIIIIQQ")
assert HEADER.size == 48


class FormatError(ValueError):
    """An image that is not a format-3 image of a pool of this variant and shape."""


def _pad16(n):
    return (n + 15) // 16 * 16


def _sections(pool, L):
    """(name, region, bytes) of the sections of one (sequence, layer): K store, V
    store, then the scales region of each store that has one.  A section holds
    the region's rows of positions 0..L-1, so its bytes are L x kv heads x the
    region's row bytes."""
    out = []
    for name, region in (("k", pool.k_store), ("v", pool.v_store), ("ks", pool.k_scales),
                         ("vs", pool.v_scales)):
        if region is not None:
            out.append((name, region, L * pool.n_kv_heads * region.shape[-1] * region.itemsize))
    return out


def image_bytes(pool, lengths):
    """Size of the image of sequences of these lengths."""
    n = HEADER.size + _pad16(4 * len(lengths))
    for L in lengths:
        for _layer in range(pool.n_layers):
            n += sum(_pad16(b) for _, _, b in _sections(pool, int(L)))
    return n


def _rows(pool, page_table_row, L):
    """(pages, slots) of positions 0..L-1 of a sequence."""
    pos = np.arange(L)
    pages = np.asarray(page_table_row, np.int64)[pos // pool.page_size] if L else np.zeros(0, np.int64)
    return pages, pos % pool.page_size


def save(pool, lengths, page_table):
    """The image (bytes) of positions 0..L_b-1 of every layer of each sequence b.

    page_table: int [n_seqs][max_pages] of the pool."""
    lengths = [int(x) for x in lengths]
    parts = []
    for b, L in enumerate(lengths):
        pages, slots = _rows(pool, page_table[b], L)
        for layer in range(pool.n_layers):
            for _, region, nbytes in _sections(pool, L):
                rows = region[layer, pages, :, slots, :]          # [L][Hkv][width]
                raw = np.ascontiguousarray(rows).tobytes()
                assert len(raw) == nbytes
                parts.append(raw + bytes(_pad16(nbytes) - nbytes))
    payload = b"".join(parts)
    lens = np.asarray(lengths, "<i4").tobytes()
    head = HEADER.pack(MAGIC, VERSION, pool.variant, pool.n_layers, pool.n_kv_heads,
                       pool.head_dim, pool.gs, len(lengths), len(payload), 0)
    return head + lens + bytes(_pad16(len(lens)) - len(lens)) + payload


def read_header(image):
    """(version, variant, n_layers, n_kv_heads, head_dim, group_size, lengths, payload offset,
    payload bytes); raises FormatError on a wrong magic or a truncated image."""
    if len(image) < HEADER.size:
        raise FormatError("image shorter than its header")
    magic, ver, var, nl, hkv, d, gs, ns, pay, _ = HEADER.unpack_from(image, 0)
    if magic != MAGIC:
        raise FormatError("not a pool image")
    off = HEADER.size + _pad16(4 * ns)
    if len(image) < off:
        raise FormatError("image shorter than its lengths")
    lengths = np.frombuffer(image, "<i4", ns, HEADER.size).astype(np.int64)
    return ver, var, nl, hkv, d, gs, lengths, off, pay


def load(pool, image, page_table):
    """Write an image into the pool through page_table (int [n_seqs][max_pages]);
    returns the sequences' lengths.  Raises FormatError when the image is not
    format 3, was saved from a pool of another variant or shape, has a length
    that does not fit its page-table row, or is truncated."""
    ver, var, nl, hkv, d, gs, lengths, off, pay = read_header(image)
    if ver != VERSION:
        raise FormatError(f"format version {ver}, expected {VERSION}")
    if (var, nl, hkv, d, gs) != (pool.variant, pool.n_layers, pool.n_kv_heads, pool.head_dim,
                                 pool.gs):
        raise FormatError("image of a pool of another variant or shape")
    if len(lengths) != len(page_table):
        raise FormatError("one page-table row per saved sequence is needed")
    if np.any(lengths < 0):
        raise FormatError("negative length")
    if pay != image_bytes(pool, lengths) - off or len(image) < off + pay:
        raise FormatError("payload size does not match the lengths")
    cap = len(page_table[0]) * pool.page_size if len(page_table) else 0
    if np.any(lengths > cap):
        raise FormatError("a length beyond its page-table row")
    for b, L in enumerate(int(x) for x in lengths):
        pages, slots = _rows(pool, page_table[b], L)
        for layer in range(pool.n_layers):
            for _, region, nbytes in _sections(pool, L):
                width = region.shape[-1]
                rows = np.frombuffer(image, region.dtype, L * pool.n_kv_heads * width, off)
                region[layer, pages, :, slots, :] = rows.reshape(L, pool.n_kv_heads, width)
                off += _pad16(nbytes)
    return [int(x) for x in lengths]

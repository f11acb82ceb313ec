"""Oracle: the 4-bit value store of the k8v4 variant (test infrastructure only).

Strata pull request #2698 ("Not in this PR") names the next variants of its
cache: ``--kv q4_0`` and ``k8v4``, with "PR #21's Hadamard rotation over
head_dim 256" (fast Walsh-Hadamard transform, FWHT-256) and the Q4_0 format:
rotate K (after RoPE) and V before they are stored, rotate the queries, and
rotate the output back.  k8v4 keeps K as int8 codes with 64-value fp16 scales
and stores V in 4 bits; the rotation is applied where the 4-bit store is, so
the rows of V are rotated before quantization and the attention output is
rotated back.  The pages fix neither the transform's normalisation nor Q4_0's
rounding; the readings below are this library's:

FWHT over a row of n = 256 values (x as fp32):
    for h = 1, 2, 4, ..., n/2:  for every pair (i, i + h) with i & h == 0:
        (x_i, x_{i+h}) <- (x_i + x_{i+h}, x_i - x_{i+h})          (fp32)
    then x <- x * (1/16)                                          (exact)
  i.e. y = H x / sqrt(n) with H the Sylvester Hadamard matrix (entries
  (-1)^popcount(i & j)); orthonormal and its own inverse.

Q4_0 (the ggml 4-bit format: blocks of 32 values, one fp16 scale each):
    m  = the block's first value of largest magnitude (sign kept)
    d  = m * (-1/8)               (fp32, exact)
    id = 1 / d   (fp32 IEEE division; 0 when d == 0)
    q  = min(15, floor(fp32(fp32(x * id) + 8.5)))   -- a product, then a sum, each rounded
    stored: q (4 bits, 0..15) and fp16_rne(d); value (q - 8) * fp16(d)
  so the block's largest value maps to code 0 (-8 d), and codes run 0..15.

Store layout (this library's own; the pages give none): a row of D values is
D/2 bytes in 8 chunks of D/16 bytes.  Chunk r holds two bytes per block g of
32 values: byte (D/16)*r + 2g + h holds value 32g + 4r + 2h in its low nibble
and value 32g + 4r + 2h + 1 in its high nibble (r = 0..7, h = 0, 1).  So the
8 chunks each carry 4 values of every block, which the tensor-core decode
loads as one 16-byte piece per row and thread.  Scales: fp16 [D/32] per row.
"""

import numpy as np

BLOCK = 32


def fwht(x):
    """Normalised FWHT along the last axis (length a power of two), in fp32,
    butterfly by butterfly in the order above; returns fp32."""
    y = np.array(x, dtype=np.float32, copy=True)
    n = y.shape[-1]
    assert n & (n - 1) == 0
    h = 1
    while h < n:
        v = y.reshape(y.shape[:-1] + (n // (2 * h), 2, h))
        a = v[..., 0, :].copy()
        b = v[..., 1, :].copy()
        v[..., 0, :] = a + b
        v[..., 1, :] = a - b
        h *= 2
    return y * np.float32(1.0 / np.sqrt(n))


def q4_0_quantize(x32):
    """Q4_0 of fp32 rows [..., D] (D a multiple of 32): (codes uint8 [..., D] in
    0..15, scales fp16 [..., D // 32])."""
    x = np.asarray(x32, dtype=np.float32)
    D = x.shape[-1]
    assert D % BLOCK == 0
    g = x.reshape(x.shape[:-1] + (D // BLOCK, BLOCK))
    first = np.argmax(np.abs(g), axis=-1)             # first index of the largest |x|
    m = np.take_along_axis(g, first[..., None], axis=-1)[..., 0]
    d = m * np.float32(-0.125)                         # exact
    with np.errstate(divide="ignore"):
        idv = np.where(d != 0, np.float32(1.0) / d, np.float32(0.0)).astype(np.float32)
    t = (g * idv[..., None]).astype(np.float32)        # one rounding
    t = (t + np.float32(8.5)).astype(np.float32)       # a second one
    q = np.minimum(np.floor(t), 15).astype(np.uint8)
    return q.reshape(x.shape), d.astype(np.float16)


def q4_0_dequantize(codes, d16):
    """Exact fp64 values (q - 8) * d of codes [..., D] with fp16 scales [..., D // 32]."""
    q = np.asarray(codes).astype(np.float64)
    D = q.shape[-1]
    d = np.asarray(d16, dtype=np.float16).astype(np.float64)[..., None]
    return ((q.reshape(q.shape[:-1] + (D // BLOCK, BLOCK)) - 8.0) * d).reshape(q.shape)


def byte_of_value(v, D):
    """(byte, nibble) of value v in a packed row of D values (layout above)."""
    g, w = divmod(v, BLOCK)
    r, j = divmod(w, 4)
    return (D // 16) * r + 2 * g + j // 2, j % 2


def pack(codes):
    """uint8 codes [..., D] (0..15) -> bytes [..., D // 2] in the layout above."""
    c = np.asarray(codes, dtype=np.uint8)
    D = c.shape[-1]
    assert D % BLOCK == 0
    out = np.zeros(c.shape[:-1] + (D // 2,), np.uint8)
    for v in range(0, D, 2):          # values v (low nibble) and v + 1 (high) share a byte
        byte, nib = byte_of_value(v, D)
        assert nib == 0 and byte_of_value(v + 1, D) == (byte, 1)
        out[..., byte] = c[..., v] | (c[..., v + 1] << 4)
    return out


def unpack(packed):
    """bytes [..., D // 2] -> codes [..., D]."""
    p = np.asarray(packed, dtype=np.uint8)
    D = 2 * p.shape[-1]
    out = np.empty(p.shape[:-1] + (D,), np.uint8)
    for v in range(D):
        byte, nib = byte_of_value(v, D)
        out[..., v] = (p[..., byte] >> (4 * nib)) & 0x0F
    return out


def quantize_rows(x16):
    """The stored form of fp16 V rows [..., D]: (packed codes [..., D // 2], scales
    [..., D // 32]) of Q4_0 over the rotated rows."""
    codes, d = q4_0_quantize(fwht(np.asarray(x16, np.float16).astype(np.float32)))
    return pack(codes), d


def dequantize_rows(packed, d16):
    """fp64 V rows [..., D] in the original (unrotated) basis: the exact orthonormal
    rotation applied to the dequantized rotated values."""
    r = q4_0_dequantize(unpack(packed), d16)
    return hadamard_fp64(r)


_H = {}


def hadamard_fp64(x):
    """H x / sqrt(n) in fp64 along the last axis, straight from the definition
    H_ij = (-1)^popcount(i & j)."""
    x = np.asarray(x, np.float64)
    n = x.shape[-1]
    if n not in _H:
        i = np.arange(n)
        pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
        _H[n] = np.where(pc % 2 == 0, 1.0, -1.0) / np.sqrt(n)
    return x @ _H[n].T

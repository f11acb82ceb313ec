"""Oracle: attention over the dequantized INT8 KV cache, in fp64 (test infrastructure only).

Decode (genie-ai-runtime release v0.1.0-alpha.12, "Path I series" row I3: the
attention dequantizes each cached row with its own (position, kv head) scale;
Strata pull request #2698, "What it does": decode dequantizes on the fly):

  for query head h of sequence b, with kv head  kvh = h // G  (G = H / Hkv,
  consecutive query heads share a kv head) and visible keys j in [lo, L):
      z_j = scale * sum_d q[h, d] * K^[j, kvh, d]
      p_j = exp(z_j - max_j z_j)
      o[h] = sum_j p_j V^[j, kvh] / sum_j p_j

  ``scale`` defaults to 1 / sqrt(head_dim).  ``lo = max(0, L - window)`` with a
  sliding window (genie-ai-runtime v1.3.0 "Details": the kernels honour the
  sliding-window mask; the window is read as the last ``window`` positions,
  the current one included), else 0.  A sequence with no visible key yields 0.

Split-K (genie-ai-runtime v1.3.0, "split-K decode attention"): the key range
is cut into splits; each split returns the online-softmax partial
(m, l, o~) = (max z, sum exp(z - m), sum exp(z - m) v); the reduce combines them
per head:  M = max m_s,  L = sum l_s e^{m_s - M},  O = sum o~_s e^{m_s - M} / L;
a split with no key contributes (m = -inf, l = 0) and is skipped.

Prefill chunk (Strata #2698: the prompt chunk reads the int8 cache through a
dequantizing step; genie-ai-runtime v1.3.1: query-tiled causal attention for
short chunks): the chunk's new K/V are appended first, then query i at absolute
position start + i sees keys 0 .. start + i.

Softmax is evaluated two-pass (max, then sums) in fp64.
"""

import math

import numpy as np


def _softmax_weighted(z: np.ndarray, vals: np.ndarray) -> np.ndarray:
    """sum_j softmax(z)_j vals[j] in fp64 (two-pass); 0 when there are no keys."""
    if z.shape[0] == 0:
        return np.zeros(vals.shape[1:], np.float64)
    p = np.exp(z - np.max(z))
    return (p @ vals) / np.sum(p)


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def decode(q16, khat, vhat, length, window=0, scale=None):
    """Decode attention of one sequence.

    q16: fp16 [H][D]; khat, vhat: fp64 [>= length][Hkv][D] (position-major);
    returns fp64 [H][D].
    """
    q = np.asarray(q16, np.float16).astype(np.float64)
    H, D = q.shape
    Hkv = khat.shape[1]
    G = H // Hkv
    sc = default_scale(D) if scale is None else float(scale)
    lo = max(0, length - window) if window > 0 else 0
    out = np.zeros((H, D), np.float64)
    for h in range(H):
        kvh = h // G
        if h % G == 0:   # the visible keys and values of this kv head, as rows
            kh = np.ascontiguousarray(khat[lo:length, kvh, :])
            vh = np.ascontiguousarray(vhat[lo:length, kvh, :])
        z = sc * (kh @ q[h])
        out[h] = _softmax_weighted(z, vh)
    return out


def split_bounds(lo: int, hi: int, n_splits: int, page_size: int):
    """Page-aligned split of the key range [lo, hi): split s covers keys
    [lo_page + s * c, lo_page + (s + 1) * c) ∩ [lo, hi) with
    c = page_size * ceil(n_range_pages / n_splits)."""
    if hi <= lo:
        return [(lo, lo)] * n_splits
    p0 = lo // page_size
    n_pages = (hi - 1) // page_size + 1 - p0
    per = -(-n_pages // n_splits) * page_size
    out = []
    for s in range(n_splits):
        a = max(lo, p0 * page_size + s * per)
        b = min(hi, p0 * page_size + (s + 1) * per)
        out.append((a, max(a, b)))
    return out


def split_partial(q_row, khat_h, vhat_h, a, b, scale):
    """Online-softmax partial (m, l, o~) of one query head over keys [a, b)."""
    if b <= a:
        return -math.inf, 0.0, np.zeros(vhat_h.shape[1], np.float64)
    z = scale * (khat_h[a:b] @ q_row)
    m = float(np.max(z))
    p = np.exp(z - m)
    return m, float(np.sum(p)), p @ vhat_h[a:b]


def combine(partials):
    """Per-head reduce of split partials [(m, l, o~), ...] -> normalised output."""
    live = [(m, l, o) for (m, l, o) in partials if l > 0.0]
    if not live:
        return np.zeros_like(partials[0][2])
    M = max(m for m, _, _ in live)
    Lsum = sum(l * math.exp(m - M) for m, l, _ in live)
    O = sum(o * math.exp(m - M) for m, _, o in live)
    return O / Lsum


def decode_split(q16, khat, vhat, length, n_splits, page_size=64, window=0, scale=None):
    """Decode attention through split partials and the combine (fp64)."""
    q = np.asarray(q16, np.float16).astype(np.float64)
    H, D = q.shape
    G = H // khat.shape[1]
    sc = default_scale(D) if scale is None else float(scale)
    lo = max(0, length - window) if window > 0 else 0
    out = np.zeros((H, D), np.float64)
    for h in range(H):
        kvh = h // G
        parts = [split_partial(q[h], khat[:, kvh, :], vhat[:, kvh, :], a, b, sc)
                 for (a, b) in split_bounds(lo, length, n_splits, page_size)]
        out[h] = combine(parts)
    return out


def prefill_chunk(q16, khat, vhat, start, scale=None):
    """Causal attention of a chunk of queries at absolute positions start + i.

    q16: fp16 [n_new][H][D]; khat, vhat: fp64 [>= start + n_new][Hkv][D];
    returns fp64 [n_new][H][D].
    """
    q = np.asarray(q16, np.float16).astype(np.float64)
    n_new, H, D = q.shape
    G = H // khat.shape[1]
    sc = default_scale(D) if scale is None else float(scale)
    out = np.zeros((n_new, H, D), np.float64)
    for kvh in range(khat.shape[1]):
        heads = slice(kvh * G, (kvh + 1) * G)
        kh = khat[:, kvh, :]
        vh = vhat[:, kvh, :]
        for i in range(n_new):
            n_vis = start + i + 1
            z = sc * (q[i, heads, :] @ kh[:n_vis].T)          # [G][n_vis]
            p = np.exp(z - np.max(z, axis=1, keepdims=True))
            out[i, heads, :] = (p @ vh[:n_vis]) / np.sum(p, axis=1, keepdims=True)
    return out

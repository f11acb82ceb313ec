// Device helpers shared by the kernels.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

#include "internal.h"

namespace int8kv {

__device__ __forceinline__ void flag_error(int32_t* err, int bits) {
  if (err) atomicOr(err, bits);
}

// Physical page of logical page `lp` of a sequence, or -1 (flagged) when the
// table entry or the index is outside the pool.
// A page-table entry, or -1 (flagged) when it names no page of the pool.
__device__ __forceinline__ int check_page(int pg, const PoolView& p) {
  if (pg < 0 || pg >= p.n_pages) {
    flag_error(p.err, INT8KV_DEVERR_PAGE_ID);
    return -1;
  }
  return pg;
}

__device__ __forceinline__ int lookup_page(const int32_t* row, int lp, int max_pages,
                                           const PoolView& p) {
  if (lp < 0 || lp >= max_pages) {
    flag_error(p.err, INT8KV_DEVERR_LENGTH);
    return -1;
  }
  return check_page(__ldg(row + lp), p);
}

// Row index (in units of head_dim values) of (page, kv head, slot).
__device__ __forceinline__ size_t row_index(const PoolView& p, int page, int kvh, int slot) {
  return ((size_t)page * p.Hkv + kvh) * p.ps + slot;
}

__device__ __forceinline__ float h2f(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

// Sequence length read on the device, clamped to what its page-table row can
// hold (a longer length is flagged).
__device__ __forceinline__ int clamp_length(int L, int max_pages, const PoolView& p) {
  const int cap = max_pages * p.ps;
  if (L > cap) {
    flag_error(p.err, INT8KV_DEVERR_LENGTH);
    L = cap;
  }
  return L < 0 ? 0 : L;
}

// Page-aligned, balanced split of the key range [lo, hi): with P pages from
// page p0 = lo / ps on, split s covers pages [p0 + s*P/S, p0 + (s+1)*P/S)
// (integer division: page counts differ by at most one), clipped to [lo, hi).
__device__ __forceinline__ void split_range(int lo, int hi, int s, int n_splits, int ps,
                                            int* a, int* b) {
  if (hi <= lo) {
    *a = *b = lo;
    return;
  }
  const int p0 = lo / ps;
  const int pages = (hi - 1) / ps + 1 - p0;
  const int pa = p0 + (int)(((long long)s * pages) / n_splits);
  const int pb = p0 + (int)(((long long)(s + 1) * pages) / n_splits);
  int x = pa * ps, y = pb * ps;
  x = x < lo ? lo : x;
  y = y > hi ? hi : y;
  *a = x;
  *b = y > x ? y : x;
}

}  // namespace int8kv

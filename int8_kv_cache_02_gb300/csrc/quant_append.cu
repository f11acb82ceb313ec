// kv_quant_append: fp16 K/V rows of new tokens -> int8 codes + fp16 absmax/127
// scales, written through the page table into the paged pool.
//
// Method: genie-ai-runtime release v0.1.0-alpha.12, "Path I series" rows I1-I2
// (per-head conversion with scale capture into a separate scales region) and
// Strata pull request #2698, "What it does" (one FP16 scale per 64 values,
// group absmax / 127).  Rounding: s = fp16_rn(fp32(absmax) / 127.0f) with an
// IEEE division; code = round-half-even(fp32(x) / fp32(s)), clamped to ±127;
// s == 0 gives code 0.
//
// One warp per (sequence, new token, kv head) row; lane l holds the head_dim/32
// consecutive values [l*VPL, (l+1)*VPL), loaded and stored with one vector
// access each, so a row is one coalesced read and one coalesced write.  The
// absmax of a group of gs values is a butterfly max over the gs/VPL lanes that
// hold it.  HBM-bound: per row 2*D bytes in, D + 2*D/gs bytes out per store.

#include <cmath>

#include <cuda_fp16.h>

#include "common.cuh"
#include "q4_row.cuh"
#include "quant_row.cuh"

namespace int8kv {
namespace {

template <int VPL>
__global__ void __launch_bounds__(256) quant_append_kernel(
    PoolView p, const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
    int n_seqs, int n_new, const int32_t* __restrict__ seq_pos,
    const int32_t* __restrict__ page_table, int max_pages, bool k_int8, bool v_int8,
    int pos_offset, float fwht_norm) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long long n_rows = (long long)n_seqs * n_new * p.Hkv;
  if (row >= n_rows) return;
  const int kvh = (int)(row % p.Hkv);
  const long long bi = row / p.Hkv;      // b * n_new + i
  const int i = (int)(bi % n_new);
  const int b = (int)(bi / n_new);
  const int pos = __ldg(seq_pos + b) + pos_offset + i;
  if (pos < 0) {
    if (lane == 0) flag_error(p.err, INT8KV_DEVERR_LENGTH);
    return;
  }
  const int page = lookup_page(page_table + (size_t)b * max_pages, pos / p.ps, max_pages, p);
  if (page < 0) return;
  const size_t dst_row = row_index(p, page, kvh, pos % p.ps);
  const size_t src_off = (size_t)row * p.D;
  const int lpg = p.gs / VPL;  // lanes per scale group
  if (p.k4)   // q4_0: K rotated, then Q4_0
    quantize_row_q4<VPL>(k_new + src_off, (uint8_t*)p.k + dst_row * (p.D / 2),
                         (uint16_t*)p.ks + dst_row * (p.D / 32), lane, fwht_norm);
  else if (k_int8)
    quantize_row<VPL>(k_new + src_off, (int8_t*)p.k + dst_row * p.D,
                      (uint16_t*)p.ks + dst_row * p.ng, lane, lpg);
  else
    copy_row<VPL>(k_new + src_off, (uint16_t*)p.k + dst_row * p.D, lane);
  if (p.v4)   // k8v4, q4_0: rotated, then Q4_0 (D/2 bytes and D/32 scales per row)
    quantize_row_q4<VPL>(v_new + src_off, (uint8_t*)p.v + dst_row * (p.D / 2),
                         (uint16_t*)p.vs + dst_row * (p.D / 32), lane, fwht_norm);
  else if (v_int8)
    quantize_row<VPL>(v_new + src_off, (int8_t*)p.v + dst_row * p.D,
                      (uint16_t*)p.vs + dst_row * p.ng, lane, lpg);
  else
    copy_row<VPL>(v_new + src_off, (uint16_t*)p.v + dst_row * p.D, lane);
}

}  // namespace

cudaError_t launch_quant_append(const PoolView& pool, const uint16_t* k_new, const uint16_t* v_new,
                                int n_seqs, int n_new, const int32_t* seq_pos,
                                const int32_t* page_table, int max_pages, bool k_int8,
                                bool v_int8, cudaStream_t stream, int pos_offset) {
  const long long rows = (long long)n_seqs * n_new * pool.Hkv;
  if (rows == 0) return cudaSuccess;
  const int warps = 8;
  const unsigned grid = (unsigned)((rows + warps - 1) / warps);
  const float norm = (float)(1.0 / std::sqrt((double)pool.D));   // FWHT scaling of the 4-bit store
  switch (pool.D) {
    case 64:
      quant_append_kernel<2><<<grid, warps * 32, 0, stream>>>(pool, k_new, v_new, n_seqs, n_new,
                                                              seq_pos, page_table, max_pages,
                                                              k_int8, v_int8, pos_offset, norm);
      break;
    case 128:
      quant_append_kernel<4><<<grid, warps * 32, 0, stream>>>(pool, k_new, v_new, n_seqs, n_new,
                                                              seq_pos, page_table, max_pages,
                                                              k_int8, v_int8, pos_offset, norm);
      break;
    case 256:
      quant_append_kernel<8><<<grid, warps * 32, 0, stream>>>(pool, k_new, v_new, n_seqs, n_new,
                                                              seq_pos, page_table, max_pages,
                                                              k_int8, v_int8, pos_offset, norm);
      break;
    default:
      return cudaErrorNotSupported;
  }
  return cudaGetLastError();
}

}  // namespace int8kv

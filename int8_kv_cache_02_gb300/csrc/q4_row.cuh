// The 4-bit value store of the k8v4 variant, one row per warp: the normalised
// fast Walsh-Hadamard transform of the row, then Q4_0 blocks of 32 values.
//
// Method: Strata pull request #2698, "Not in this PR": --kv q4_0 / k8v4 with
// the Hadamard rotation over head_dim 256 (rotate V before it is stored,
// rotate the output back).  Readings of what the pages leave open:
//   FWHT: for h = 1, 2, 4, ..., D/2, every pair (i, i + h) with i & h == 0
//         becomes (x_i + x_{i+h}, x_i - x_{i+h}) in fp32; then x * fp32(1/sqrt(D)).
//   Q4_0 (ggml's 4-bit block format): m = the block's first value of largest
//         magnitude, d = m * (-1/8), id = 1/d (IEEE; 0 when d == 0), code =
//         min(15, floor(fl(fl(x * id) + 8.5))) -- the product and the sum each
//         rounded (no fused multiply-add) -- stored as fp16(d) and a nibble.
// Lane l holds values [l*VPL, (l+1)*VPL) of the row: butterflies with h < VPL
// stay in the lane, larger ones pair lane l with lane l ^ (h / VPL); a block of
// 32 values spans 32 / VPL lanes.  Every operation is the one the definition
// names, in its order, so the codes and scales are bit-exact.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

#include "quant_row.cuh"

namespace int8kv {

// In-place normalised FWHT of a row held VPL values per lane (D = 32 * VPL).
template <int VPL>
__device__ __forceinline__ void fwht_row(float (&x)[VPL], int lane, float norm) {
#pragma unroll
  for (int h = 1; h < VPL; h <<= 1)
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if ((i & h) == 0) {
        const float a = x[i], b = x[i + h];
        x[i] = __fadd_rn(a, b);
        x[i + h] = __fsub_rn(a, b);
      }
#pragma unroll
  for (int bit = 1; bit < 32; bit <<= 1) {   // h = bit * VPL
    const bool upper = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const float y = __shfl_xor_sync(0xffffffffu, x[i], bit);
      x[i] = upper ? __fsub_rn(y, x[i]) : __fadd_rn(x[i], y);   // lower: a + b; upper: a - b
    }
  }
#pragma unroll
  for (int i = 0; i < VPL; ++i) x[i] = __fmul_rn(x[i], norm);
}

// Byte of a packed 4-bit row of D values that holds value v (v even: low
// nibble, v + 1: high nibble): the row is 8 chunks of D/16 bytes, byte
// (D/16)*r + 2g + h holding values 32g + 4r + 2h and 32g + 4r + 2h + 1.
__host__ __device__ __forceinline__ int q4_byte_of(int v, int D) {
  const int g = v >> 5, w = v & 31;
  return (D / 16) * (w >> 2) + 2 * g + ((w & 3) >> 1);
}

// Q4_0 codes (VPL nibbles packed two per byte, low nibble first) and the fp16
// scale of the lane's block (every lane of the block gets it).
template <int VPL>
__device__ __forceinline__ uint32_t q4_0_regs(const float (&x)[VPL], int lane, uint16_t& scale) {
  constexpr int LPB = 32 / VPL;   // lanes per block of 32 values
  // the block's first value of largest magnitude: (|m|, m, its index)
  float ma = fabsf(x[0]), mv = x[0];
  int mi = lane * VPL;
#pragma unroll
  for (int i = 1; i < VPL; ++i)
    if (fabsf(x[i]) > ma) {
      ma = fabsf(x[i]);
      mv = x[i];
      mi = lane * VPL + i;
    }
#pragma unroll
  for (int off = 1; off < LPB; off <<= 1) {
    const float oa = __shfl_xor_sync(0xffffffffu, ma, off);
    const float ov = __shfl_xor_sync(0xffffffffu, mv, off);
    const int oi = __shfl_xor_sync(0xffffffffu, mi, off);
    if (oa > ma || (oa == ma && oi < mi)) {
      ma = oa;
      mv = ov;
      mi = oi;
    }
  }
  const float d = __fmul_rn(mv, -0.125f);
  const float id = d != 0.f ? __fdiv_rn(1.0f, d) : 0.f;
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const float t = __fadd_rn(__fmul_rn(x[i], id), 8.5f);
    const int q = min(15, (int)floorf(t));
    packed |= (uint32_t)q << (4 * i);
  }
  scale = __half_as_ushort(__float2half_rn(d));
  return packed;
}

// One fp16 row (lane's VPL values at src + lane * VPL) into the 4-bit store:
// codes to dst_codes (D/2 bytes), scales to dst_scales (D/32 fp16).
template <int VPL>
__device__ __forceinline__ void quantize_row_q4(const uint16_t* src, uint8_t* dst_codes,
                                                uint16_t* dst_scales, int lane, float norm) {
  float x[VPL];
  load_halves<VPL>(src + lane * VPL, x);
  fwht_row<VPL>(x, lane, norm);
  uint16_t scale;
  const uint32_t packed = q4_0_regs<VPL>(x, lane, scale);
  constexpr int D = 32 * VPL;
#pragma unroll
  for (int p = 0; p < VPL / 2; ++p)   // the lane's value pairs, each one byte of the row
    dst_codes[q4_byte_of(lane * VPL + 2 * p, D)] = (uint8_t)(packed >> (8 * p));
  if (lane % (32 / VPL) == 0) dst_scales[lane * VPL / 32] = scale;
}

}  // namespace int8kv

// Pieces shared by the tensor-core decode and prefill kernels: the staged page
// layout in shared memory, the TMA issue of one page, exact int8 -> fp16
// conversion, and power-of-two helpers.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace int8kv {
namespace mma {

constexpr int kPage = 64;                  // page size served by the tensor-core kernels
constexpr int kBoxBytes = kPage * 128;     // one swizzled TMA box: 64 rows x 128 B
constexpr uint32_t kMaxPolls = 1u << 22;   // bounded mbarrier waits (well over any copy time)

// One staged page of one kv head: K rows, V rows (int8: 128-dim boxes; fp16:
// 64-dim boxes; 4-bit (VQ4 / KQ4, head_dim 256): one 128-byte box of packed
// codes per row; each box 64 rows x 128 B, 128-byte swizzle), then the K and V
// scales rows ([64][ng] fp16 of an int8 store; [64][D/32] of a 4-bit store).
template <int D, bool KI8, bool VI8, bool VQ4 = false, bool KQ4 = false>
struct StagedPage {
  static constexpr int KBYTES = KQ4 ? D / 2 * kPage : (KI8 ? D * kPage : 2 * D * kPage);
  static constexpr int VBYTES = VQ4 ? D / 2 * kPage : (VI8 ? D * kPage : 2 * D * kPage);
  static constexpr int KBOXES = KBYTES / kBoxBytes;
  static constexpr int VBOXES = VBYTES / kBoxBytes;
  static constexpr int SCALE_BYTES = kPage * 4 * 2;   // up to 4 groups per row
  static constexpr int VQ4_SCALE_BYTES = kPage * (D / 32) * 2;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = KBYTES;
  static constexpr int KS_OFF = KBYTES + VBYTES;
  static constexpr int VS_OFF = KS_OFF + (KI8 ? SCALE_BYTES : (KQ4 ? VQ4_SCALE_BYTES : 0));
  static constexpr int RAW = VS_OFF + (VI8 ? SCALE_BYTES : (VQ4 ? VQ4_SCALE_BYTES : 0));
  static constexpr int STAGE = (RAW + 1023) / 1024 * 1024;
};

// Bytes 0 and 2 of x (int8 codes c) -> fp16 pair holding 1152 + c: the fp16 with
// bit pattern 0x6400 | u is 1024 + u for u in [0, 255] (the magic-number method
// of Kim et al., "Who Says Elephants Can't Run", 2022), u = c ^ 0x80 = c + 128.
__device__ __forceinline__ uint32_t lop_i8pair(uint32_t x) {
  return (x & 0x00FF00FFu) ^ 0x64806480u;
}

// (1152 + c) - 1152 = c, exact in fp16.
__device__ __forceinline__ uint32_t sub1152(uint32_t h2) {
  const __half2 r =
      __hsub2(*reinterpret_cast<const __half2*>(&h2), __half2half2(__ushort_as_half(0x6480)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ float pow2f(int e) {   // 2^e for e in [-126, 127]
  return __uint_as_float((uint32_t)(127 + e) << 23);
}

__device__ __forceinline__ int exponent_of(float x) {   // floor(log2 x), x > 0 normal
  return (int)((__float_as_uint(x) >> 23) & 0xFF) - 127;
}

// Softmax weights p0, p1 >= 0 (below 2^16; the kernels pass p * 2^5 <= 2^13) as
// fp16 hi + lo pairs: hi keeps each weight's 11 leading bits (its 13 low mantissa
// bits cleared: exact in fp16 from 2^-14 up), lo the remainder rounded to fp16.
__device__ __forceinline__ void split_pair(float p0, float p1, uint32_t& hi, uint32_t& lo) {
  const float h0 = __uint_as_float(__float_as_uint(p0) & 0xFFFFE000u);
  const float h1 = __uint_as_float(__float_as_uint(p1) & 0xFFFFE000u);
  hi = ptx::pack_f16x2(h0, h1);
  lo = ptx::pack_f16x2(p0 - h0, p1 - h1);
}

// The same pair formed directly (one factor w for both): P' = p * w in fp32,
// hi = fl16(P'), lo = fl16(P' - hi).  Fewer operations than split_pair followed by
// weight_pair when a tile has a single V group.
__device__ __forceinline__ void weight_pair_f32(float p0, float p1, float w, uint32_t& hi,
                                                uint32_t& lo) {
  const float w0 = p0 * w, w1 = p1 * w;
  hi = ptx::pack_f16x2(w0, w1);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  lo = ptx::pack_f16x2(w0 - f.x, w1 - f.y);
}

// The P.V weights P' = p * s of two keys (p as the hi + lo pairs of split_pair, s
// an fp16 factor per key) as a new fp16 hi + lo pair, in half-precision
// arithmetic: hi = fl(ph s); ph s - hi, an 11-bit by 11-bit product less its
// rounding to 11 bits, is exact in fp16 outside the subnormal range, so
// lo = fl(pl s + (ph s - hi)) leaves P' within ~2^-21 of p * s.  Exact only
// while p and s are normal in fp16 (callers split p scaled up by 2^5 and scale s
// down by as much).
__device__ __forceinline__ void weight_pair(uint32_t ph, uint32_t pl, uint32_t s, uint32_t& hi,
                                            uint32_t& lo) {
  const __half2 a = *reinterpret_cast<const __half2*>(&ph);
  const __half2 b = *reinterpret_cast<const __half2*>(&pl);
  const __half2 f = *reinterpret_cast<const __half2*>(&s);
  const __half2 h = __hmul2_rn(a, f);
  const __half2 l = __hfma2(b, f, __hfma2(a, f, __hneg2(h)));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Issue the copies of one page (or, for a page id flagged invalid, complete the
// stage's barrier with no bytes) into stage `st`.  kStream: the page is read
// once (decode), so its L2 lines go first; otherwise (prefill: every query tile
// of the kv head reads it) the default policy keeps it for the other blocks.
template <int D, bool KI8, bool VI8, bool kStream = false, bool VQ4 = false, bool KQ4 = false>
__device__ __forceinline__ void issue_page(unsigned char* stage, uint64_t* full_bar, int* stage_page,
                                           int page, int row, const PoolView& p, int kvh,
                                           const CUtensorMap* tmk, const CUtensorMap* tmv) {
  using SP = StagedPage<D, KI8, VI8, VQ4, KQ4>;
  *stage_page = page;
  if (page < 0) {
    ptx::mbar_arrive(full_bar);
    return;
  }
  const int ng = p.ng;
  constexpr uint32_t VSB = VQ4 ? SP::VQ4_SCALE_BYTES : 0;   // 4-bit store: D/32 scales a row
  constexpr uint32_t KSB = KQ4 ? SP::VQ4_SCALE_BYTES : 0;
  const uint32_t tx = SP::KBYTES + SP::VBYTES + (KI8 ? kPage * ng * 2 : KSB) +
                      (VI8 ? kPage * ng * 2 : VSB);
  ptx::mbar_arrive_expect_tx(full_bar, tx);
  const size_t srow = ((size_t)page * p.Hkv + kvh) * kPage * ng;
  const size_t vsrow = ((size_t)page * p.Hkv + kvh) * kPage * (VQ4 ? D / 32 : ng);
  const size_t q4row = ((size_t)page * p.Hkv + kvh) * kPage * (D / 32);   // 4-bit K scales
  // a side of several 128-byte boxes a row comes in one 3-D copy (the map is 3-D)
  if constexpr (kStream) {
    const uint64_t pol = ptx::policy_evict_first();
    if constexpr (SP::KBOXES > 1)
      ptx::tma_load_3d_hint(stage + SP::K_OFF, tmk, 0, row, 0, full_bar, pol);
    else
      ptx::tma_load_2d_hint(stage + SP::K_OFF, tmk, 0, row, full_bar, pol);
    if constexpr (SP::VBOXES > 1)
      ptx::tma_load_3d_hint(stage + SP::V_OFF, tmv, 0, row, 0, full_bar, pol);
    else
      ptx::tma_load_2d_hint(stage + SP::V_OFF, tmv, 0, row, full_bar, pol);
    if (KI8) ptx::bulk_load_hint(stage + SP::KS_OFF, p.ks + srow, kPage * ng * 2, full_bar, pol);
    if (KQ4) ptx::bulk_load_hint(stage + SP::KS_OFF, p.ks + q4row, KSB, full_bar, pol);
    if (VI8) ptx::bulk_load_hint(stage + SP::VS_OFF, p.vs + srow, kPage * ng * 2, full_bar, pol);
    if (VQ4) ptx::bulk_load_hint(stage + SP::VS_OFF, p.vs + vsrow, VSB, full_bar, pol);
  } else {
    if constexpr (SP::KBOXES > 1)
      ptx::tma_load_3d(stage + SP::K_OFF, tmk, 0, row, 0, full_bar);
    else
      ptx::tma_load_2d(stage + SP::K_OFF, tmk, 0, row, full_bar);
    if constexpr (SP::VBOXES > 1)
      ptx::tma_load_3d(stage + SP::V_OFF, tmv, 0, row, 0, full_bar);
    else
      ptx::tma_load_2d(stage + SP::V_OFF, tmv, 0, row, full_bar);
    if (KI8) ptx::bulk_load(stage + SP::KS_OFF, p.ks + srow, kPage * ng * 2, full_bar);
    if (KQ4) ptx::bulk_load(stage + SP::KS_OFF, p.ks + q4row, KSB, full_bar);
    if (VI8) ptx::bulk_load(stage + SP::VS_OFF, p.vs + srow, kPage * ng * 2, full_bar);
    if (VQ4) ptx::bulk_load(stage + SP::VS_OFF, p.vs + vsrow, VSB, full_bar);
  }
}

}  // namespace mma
}  // namespace int8kv

// Quantization of one fp16 row by one warp (shared by the append kernel and the
// decode kernel's fused append).
//
// Method: absmax/127 per group of gs values (genie-ai-runtime v0.1.0-alpha.12
// "Path I series" I2; Strata pull request #2698 "What it does"):
//   s = fp16_rn(fp32(absmax) / 127.0f), code = clamp(rint_even(fp32(x) / fp32(s)), -127, 127),
//   code = 0 when s == 0, all divisions IEEE round-to-nearest.  Lane l holds
//   values [l*VPL, (l+1)*VPL) of the row.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

namespace int8kv {

template <int VPL>
struct Vec;
template <>
struct Vec<2> { using H = uint32_t; using B = uint16_t; };
template <>
struct Vec<4> { using H = uint2; using B = uint32_t; };
template <>
struct Vec<8> { using H = uint4; using B = uint2; };

template <int VPL>
__device__ __forceinline__ void load_halves(const uint16_t* src, float (&x)[VPL]) {
  typename Vec<VPL>::H raw = *reinterpret_cast<const typename Vec<VPL>::H*>(src);
  const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int i = 0; i < VPL / 2; ++i) {
    const float2 f = __half22float2(h2[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// Codes and scale of the lane's VPL values x; the scale is that of the lane's
// group (every lane of a group of lanes_per_group lanes gets it).
template <int VPL>
__device__ __forceinline__ void quantize_regs(const float (&x)[VPL], int lanes_per_group,
                                              typename Vec<VPL>::B& codes, uint16_t& scale) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) amax = fmaxf(amax, fabsf(x[i]));
  for (int off = 1; off < lanes_per_group; off <<= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const __half s16 = __float2half_rn(__fdiv_rn(amax, 127.0f));
  const float s = __half2float(s16);
  union { typename Vec<VPL>::B v; int8_t c[VPL]; } out;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    int c = 0;
    if (s != 0.f) {
      // The code is rint(fl(x / s)) with the IEEE quotient.  |x / s| < 128, so
      // __fdividef (at most 2 ulp off for these divisors) lands within 2e-5 of
      // fl(x / s); unless that is within 1e-4 of a half-integer, both round to
      // the same integer, and only then is the IEEE division needed.
      float qt = __fdividef(x[i], s);
      if (fabsf((qt - floorf(qt)) - 0.5f) < 1.0e-4f) qt = __fdiv_rn(x[i], s);
      c = __float2int_rn(qt);  // round half to even
      c = max(-127, min(127, c));
    }
    out.c[i] = (int8_t)c;
  }
  codes = out.v;
  scale = __half_as_ushort(s16);
}

template <int VPL>
__device__ __forceinline__ void quantize_row(const uint16_t* src, int8_t* dst_codes,
                                             uint16_t* dst_scales, int lane, int lanes_per_group) {
  float x[VPL];
  load_halves<VPL>(src + lane * VPL, x);
  typename Vec<VPL>::B codes;
  uint16_t scale;
  quantize_regs<VPL>(x, lanes_per_group, codes, scale);
  *reinterpret_cast<typename Vec<VPL>::B*>(dst_codes + lane * VPL) = codes;
  if ((lane % lanes_per_group) == 0) dst_scales[(lane * VPL) / (lanes_per_group * VPL)] = scale;
}

template <int VPL>
__device__ __forceinline__ void copy_row(const uint16_t* src, uint16_t* dst, int lane) {
  *reinterpret_cast<typename Vec<VPL>::H*>(dst + lane * VPL) =
      *reinterpret_cast<const typename Vec<VPL>::H*>(src + lane * VPL);
}

}  // namespace int8kv

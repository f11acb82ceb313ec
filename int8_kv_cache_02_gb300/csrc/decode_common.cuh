// Split combine shared by the decode kernels.
//
// genie-ai-runtime v1.3.0 "split-K decode attention": a reduce combines the
// per-split online-softmax partials per head.  With partials (m_s, l_s, o~_s)
// in base-2 exponent units:
//     M = max_s m_s,  w_s = 2^(m_s - M) / sum_t l_t 2^(m_t - M),  O = sum_s w_s o~_s
// Splits that saw no key carry (m = -inf, l = 0) and get weight 0; a head with
// no key at all gets O = 0.
#pragma once

#include "common.cuh"

namespace int8kv {

constexpr int kMaxSplits = 256;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Run by every thread of the last-arriving block of (b, kvh).  `scratch` is
// shared memory of at least 8 * n_splits floats.  Partials are read with
// L1-bypassing loads: other blocks wrote them.
__device__ __forceinline__ void combine_splits_block(const DecodeArgs& a, int b, int kvh,
                                                     float* scratch) {
  const int G = a.G, D = a.pool.D, S = a.n_splits;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int g = warp; g < G; g += nw) {
    const size_t h = (size_t)b * a.H + (size_t)kvh * G + g;
    const float2* ml = a.ws.part_ml + h * S;
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, __ldcg(ml + s).x);
    M = warp_max(M);
    float Ls = 0.f;
    if (M != -INFINITY)
      for (int s = lane; s < S; s += 32) {
        const float2 v = __ldcg(ml + s);
        if (v.y > 0.f) Ls = fmaf(v.y, exp2f(v.x - M), Ls);
      }
    Ls = warp_sum(Ls);
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    for (int s = lane; s < S; s += 32) {
      const float2 v = __ldcg(ml + s);
      scratch[g * S + s] = (v.y > 0.f && M != -INFINITY) ? exp2f(v.x - M) * inv : 0.f;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int g = e / D, d = e - g * D;
    const size_t h = (size_t)b * a.H + (size_t)kvh * G + g;
    const float* po = a.ws.part_o + h * S * D + d;
    float O = 0.f;
    for (int s = 0; s < S; ++s) {
      const float w = scratch[g * S + s];
      if (w != 0.f) O = fmaf(w, __ldcg(po + (size_t)s * D), O);
    }
    a.out[h * D + d] = O;
  }
}

cudaError_t launch_decode_simt(const DecodeArgs& a, bool k_int8, bool v_int8,
                               cudaStream_t stream);

}  // namespace int8kv

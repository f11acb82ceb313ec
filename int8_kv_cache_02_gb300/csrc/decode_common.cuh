// Declarations shared by the decode kernels: split limit, warp reductions and
// the launchers of the partial kernels and of the per-head combine.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace int8kv {

constexpr int kMaxSplits = 256;
constexpr int kMaxQueryWindow = 64;   // queries per sequence of one attn_decode_multi_int8 call

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

cudaError_t launch_decode_simt(const DecodeArgs& a, bool k_int8, bool v_int8,
                               cudaStream_t stream);
cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t stream);
bool decode_mma_supported(const PoolView& p, int G);
int decode_mma_resident_blocks(int D, bool k8, bool v8, int ng, bool v4, bool k4);
cudaError_t launch_decode_mma(const DecodeArgs& a, bool k8, bool v8, const CUtensorMap& tmk,
                              const CUtensorMap& tmv, int layer_page0, cudaStream_t stream);

}  // namespace int8kv

// Per-head combine of split-K decode partials (genie-ai-runtime v1.3.0,
// "split-K decode attention": a reduce kernel combines the per-split
// online-softmax partials per head).
//
// Partials are (m_s, l_s, o~_s) in base-2 exponent units:
//     M = max_s m_s,  w_s = 2^(m_s - M) / sum_t l_t 2^(m_t - M),  O = sum_s w_s o~_s
// Splits that saw no key carry (m = -inf, l = 0) and get weight 0; a head with
// no key at all gets O = 0.
//
// Grid (head_dim / 64, n_heads, batch), 64 threads: one output dim per thread,
// every split's row read coalesced.  Launched as a programmatic dependent of
// the partial kernel so its launch overlaps the partial kernel's tail; it waits
// on the grid dependency before touching the partials.

#include "common.cuh"
#include "decode_common.cuh"
#include "ptx.cuh"

namespace int8kv {
namespace {

__global__ void __launch_bounds__(64) decode_combine_kernel(const DecodeArgs a) {
  const int dchunk = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;
  const int D = a.pool.D, S = a.n_splits;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ float w[kMaxSplits];
  ptx::grid_dependency_wait();
  const size_t h = (size_t)b * a.H + hq;
  const float2* ml = a.ws.part_ml + h * S;
  if (warp == 0) {
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, ml[s].x);
    M = warp_max(M);
    float Ls = 0.f;
    if (M != -INFINITY)
      for (int s = lane; s < S; s += 32) {
        const float2 v = ml[s];
        if (v.y > 0.f) Ls = fmaf(v.y, exp2f(v.x - M), Ls);
      }
    Ls = warp_sum(Ls);
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    for (int s = lane; s < S; s += 32) {
      const float2 v = ml[s];
      w[s] = (v.y > 0.f && M != -INFINITY) ? exp2f(v.x - M) * inv : 0.f;
    }
  }
  __syncthreads();
  const int d = dchunk * 64 + threadIdx.x;
  const float* po = a.ws.part_o + h * S * D + d;
  float O = 0.f;
  for (int s = 0; s < S; ++s) {
    const float ws = w[s];
    if (ws != 0.f) O = fmaf(ws, po[(size_t)s * D], O);
  }
  a.out[h * D + d] = O;
}

}  // namespace

cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.pool.D / 64, a.H, a.B);
  cfg.blockDim = dim3(64);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel, a);
}

}  // namespace int8kv

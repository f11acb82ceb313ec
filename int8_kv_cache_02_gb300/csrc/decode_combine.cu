// Per-head combine of split-K decode partials (genie-ai-runtime v1.3.0,
// "split-K decode attention": a reduce kernel combines the per-split
// online-softmax partials per head).
//
// Partials are (m_s, l_s, o~_s) in base-2 exponent units:
//     M = max_s m_s,  w_s = 2^(m_s - M) / sum_t l_t 2^(m_t - M),  O = sum_s w_s o~_s
// Splits that saw no key carry (m = -inf, l = 0) and get weight 0; a head with
// no key at all gets O = 0.
//
// Grid (head_dim / 64, n_heads, batch); eight warps share the splits of one
// (head, 64-dim slice), each lane two adjacent dims, four independent loads in
// flight per lane; the eight warp sums meet in shared memory.  Launched as a programmatic dependent of
// the partial kernel so its launch overlaps the partial kernel's tail; it waits
// on the grid dependency before touching the partials.

#include "common.cuh"
#include "decode_common.cuh"
#include "ptx.cuh"

namespace int8kv {
namespace {

constexpr int kCombineWarps = 8;   // split range cut into 8 slices, one per warp

__global__ void __launch_bounds__(kCombineWarps * 32) decode_combine_kernel(const DecodeArgs a) {
  const int dchunk = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;
  const int D = a.pool.D, S = a.n_splits;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ float w[kMaxSplits];
  __shared__ float2 part[kCombineWarps][32];
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
  // warp `warp` sums splits warp, warp + 8, ...; each lane two adjacent dims
  const int d = dchunk * 64 + 2 * lane;
  const float* po = a.ws.part_o + h * S * D + d;
  float2 acc[4] = {};
  int s = warp, k = 0;
  for (; s + 3 * kCombineWarps < S; s += 4 * kCombineWarps) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float2 v = *reinterpret_cast<const float2*>(po + (size_t)(s + u * kCombineWarps) * D);
      const float ws = w[s + u * kCombineWarps];
      acc[u].x = fmaf(ws, v.x, acc[u].x);
      acc[u].y = fmaf(ws, v.y, acc[u].y);
    }
  }
  for (; s < S; s += kCombineWarps, k = (k + 1) & 3) {
    const float2 v = *reinterpret_cast<const float2*>(po + (size_t)s * D);
    acc[k].x = fmaf(w[s], v.x, acc[k].x);
    acc[k].y = fmaf(w[s], v.y, acc[k].y);
  }
  part[warp][lane] = make_float2(acc[0].x + acc[1].x + acc[2].x + acc[3].x,
                                 acc[0].y + acc[1].y + acc[2].y + acc[3].y);
  __syncthreads();
  if (warp == 0) {
    float2 o = part[0][lane];
#pragma unroll
    for (int q = 1; q < kCombineWarps; ++q) {
      o.x += part[q][lane].x;
      o.y += part[q][lane].y;
    }
    *reinterpret_cast<float2*>(a.out + h * D + d) = o;
  }
}

}  // namespace

cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.pool.D / 64, a.H, a.B);
  cfg.blockDim = dim3(kCombineWarps * 32);
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

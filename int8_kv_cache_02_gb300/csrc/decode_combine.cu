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
// (head, 64-dim slice), each lane two adjacent dims.  Every lane issues all its
// partial loads before the split weights are known (warp 0 computes those from
// the (m, l) pairs meanwhile), so the two round trips to L2 overlap; the eight
// warp sums meet in shared memory.  Launched as a programmatic dependent of
// the partial kernel so its launch overlaps the partial kernel's tail; it waits
// on the grid dependency before touching the partials.

#include "common.cuh"
#include "decode_common.cuh"
#include "ptx.cuh"

namespace int8kv {
namespace {

constexpr int kCombineWarps = 8;       // splits cut into 8 slices, one per warp
constexpr int kPerLane = kMaxSplits / kCombineWarps;   // splits a lane may hold (32)

__global__ void __launch_bounds__(kCombineWarps * 32) decode_combine_kernel(const DecodeArgs a) {
  const int dchunk = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;
  const int D = a.pool.D, S = a.n_splits;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ float w[kMaxSplits];
  __shared__ float2 part[kCombineWarps][32];
  // The next kernel of the stream may launch now: a decode kernel that follows
  // waits on this grid before it reads anything but its prefetch hints.
  ptx::grid_launch_dependents();
  ptx::grid_dependency_wait();
  const size_t h = (size_t)b * a.H + hq;
  // every lane first puts its partial rows in flight (they do not depend on the
  // weights): warp `warp` takes splits warp, warp + 8, ...; a lane two dims
  const int d = dchunk * 64 + 2 * lane;
  const float* po = a.ws.part_o + h * S * D + d;
  float2 x[kPerLane];
#pragma unroll
  for (int k = 0; k < kPerLane; ++k) {
    const int s = warp + k * kCombineWarps;
    x[k] = s < S ? *reinterpret_cast<const float2*>(po + (size_t)s * D) : make_float2(0.f, 0.f);
  }
  if (warp == 0) {   // split weights 2^(m_s - M) / L
    const float2* ml = a.ws.part_ml + h * S;
    float2 v[kMaxSplits / 32];
#pragma unroll
    for (int k = 0; k < kMaxSplits / 32; ++k) {
      const int s = lane + 32 * k;
      v[k] = s < S ? ml[s] : make_float2(-INFINITY, 0.f);
    }
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMaxSplits / 32; ++k) M = fmaxf(M, v[k].x);
    M = warp_max(M);
    float f[kMaxSplits / 32], Ls = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxSplits / 32; ++k) {
      f[k] = (M == -INFINITY || v[k].y == 0.f) ? 0.f : exp2f(v[k].x - M);
      Ls = fmaf(v[k].y, f[k], Ls);
    }
    Ls = warp_sum(Ls);
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
    for (int k = 0; k < kMaxSplits / 32; ++k) {
      const int s = lane + 32 * k;
      if (s < S) w[s] = f[k] * inv;
    }
  }
  __syncthreads();
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kPerLane; ++k) {
    const int s = warp + k * kCombineWarps;
    if (s < S) {
      acc.x = fmaf(w[s], x[k].x, acc.x);
      acc.y = fmaf(w[s], x[k].y, acc.y);
    }
  }
  part[warp][lane] = acc;
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

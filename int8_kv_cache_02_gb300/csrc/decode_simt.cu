// Split-K GQA decode attention over the int8 cache, CUDA-core version.
//
// Method: genie-ai-runtime v1.3.0 "split-K decode attention": the key range of
// each head is cut into n_splits pieces, each block computes an online-softmax
// partial (m, l, o~) and a reduce combines the partials per head.  Keys are
// dequantized on load with their own (position, kv head[, group]) scale
// (genie-ai-runtime v0.1.0-alpha.12 "Path I series" row I3).
//
// Grid (n_splits, Hkv, B); one block serves all G query heads of its kv head so
// every cached byte is read once.  Four warps take the block's keys round-robin;
// lane l owns dims [l*VPL, (l+1)*VPL) of every row, so a row is one coalesced
// warp access.  Scores are reduced with warp shuffles; softmax runs in base 2
// (scale folded with log2 e).  The warps' partials are merged in shared memory;
// with n_splits > 1 the block stores its partial and the combine kernel
// (decode_combine.cu) reduces the splits.
//
// This kernel is the general path (any G <= 8, head_dim 64/128/256, every
// store variant); the tensor-core kernel in decode_mma.cu serves the shapes it
// is specialised for.  The 4-bit stores (Strata pull request #2698, "Not in
// this PR": k8v4 and --kv q4_0 with the Hadamard rotation) hold rotated rows:
// with a rotated K store each query is rotated by the same normalised FWHT
// before its scores (q.k = Hq.Hk, H orthonormal); with a rotated V store the
// merged output rows are rotated back.

#include <cmath>

#include <cuda_fp16.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "q4_row.cuh"

namespace int8kv {
namespace {

constexpr int kWarps = 4;

template <int VPL>
__device__ __forceinline__ void load_row(const void* store, bool is_int8, const uint16_t* scales,
                                         size_t row, int D, int ng, int gs, int lane,
                                         float (&x)[VPL]) {
  if (is_int8) {
    const int8_t* src = (const int8_t*)store + row * D + lane * VPL;
    int8_t c[VPL];
    if constexpr (VPL == 8) {
      *reinterpret_cast<uint2*>(c) = __ldg(reinterpret_cast<const uint2*>(src));
    } else if constexpr (VPL == 4) {
      *reinterpret_cast<uint32_t*>(c) = __ldg(reinterpret_cast<const uint32_t*>(src));
    } else {
      *reinterpret_cast<uint16_t*>(c) = __ldg(reinterpret_cast<const uint16_t*>(src));
    }
    const float s = h2f(__ldg(scales + row * ng + (lane * VPL) / gs));
#pragma unroll
    for (int i = 0; i < VPL; ++i) x[i] = (float)c[i] * s;
  } else {
    const uint16_t* src = (const uint16_t*)store + row * D + lane * VPL;
#pragma unroll
    for (int i = 0; i < VPL; ++i) x[i] = h2f(__ldg(src + i));
  }
}

// A row of a 4-bit store: the lane's VPL values (code - 8) * d, in the rotated
// basis, d its block's fp16 scale.
template <int VPL>
__device__ __forceinline__ void load_row_q4(const void* store, const uint16_t* scales, size_t row,
                                            int D, int lane, float (&x)[VPL]) {
  const uint8_t* src = (const uint8_t*)store + row * (D / 2);
  const float d = h2f(__ldg(scales + row * (D / 32) + (lane * VPL) / 32));
#pragma unroll
  for (int p = 0; p < VPL / 2; ++p) {   // the lane's value pairs, one byte each
    const uint32_t b = __ldg(src + q4_byte_of(lane * VPL + 2 * p, D));
    x[2 * p] = (float)((int)(b & 15u) - 8) * d;
    x[2 * p + 1] = (float)((int)(b >> 4) - 8) * d;
  }
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) decode_simt_kernel(DecodeArgs a, bool k_int8,
                                                                   bool v_int8, float fwht_norm) {
  constexpr int VPL = D / 32;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int G = a.G;
  const PoolView& p = a.pool;

  __shared__ float s_m[kWarps][8], s_l[kWarps][8];
  __shared__ float s_o[kWarps][8][D];
  __shared__ float s_r[8][D], s_M[8], s_L[8];   // 4-bit V: merged rows before the rotation back

  float qr[8][VPL];
#pragma unroll
  for (int g = 0; g < 8; ++g)
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      qr[g][i] = g < G ? h2f(__ldg(a.q + ((size_t)b * a.H + kvh * G + g) * D + lane * VPL + i)) : 0.f;
  if (p.k4) {   // rotated keys: rotate the queries the same way
#pragma unroll
    for (int g = 0; g < 8; ++g)
      if (g < G) fwht_row<VPL>(qr[g], lane, fwht_norm);
  }

  const int L = clamp_length(__ldg(a.seq_lens + b), a.max_pages, p);
  const int lo = a.window > 0 ? max(0, L - a.window) : 0;
  int j0, j1;
  split_range(lo, L, split, a.n_splits, p.ps, &j0, &j1);

  float m[8], l[8], o[8][VPL];
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) o[g][i] = 0.f;
  }

  const int32_t* ptrow = a.page_table + (size_t)b * a.max_pages;
  for (int j = j0 + warp; j < j1; j += kWarps) {
    const int pg = lookup_page(ptrow, j / p.ps, a.max_pages, p);
    if (pg < 0) continue;
    const size_t row = row_index(p, pg, kvh, j % p.ps);
    float kf[VPL], vf[VPL];
    if (p.k4)
      load_row_q4<VPL>(p.k, p.ks, row, D, lane, kf);
    else
      load_row<VPL>(p.k, k_int8, p.ks, row, D, p.ng, p.gs, lane, kf);
    if (p.v4)
      load_row_q4<VPL>(p.v, p.vs, row, D, lane, vf);
    else
      load_row<VPL>(p.v, v_int8, p.vs, row, D, p.ng, p.gs, lane, vf);
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      if (g < G) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i) s = fmaf(qr[g][i], kf[i], s);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        const float z = s * a.scale_log2;
        const float mn = fmaxf(m[g], z);
        const float alpha = exp2f(m[g] - mn);
        const float pz = exp2f(z - mn);
        l[g] = l[g] * alpha + pz;
#pragma unroll
        for (int i = 0; i < VPL; ++i) o[g][i] = fmaf(o[g][i], alpha, pz * vf[i]);
        m[g] = mn;
      }
    }
  }

  // merge the warps' partials in shared memory
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    if (lane == 0) {
      s_m[warp][g] = m[g];
      s_l[warp][g] = l[g];
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) s_o[warp][g][lane * VPL + i] = o[g][i];
  }
  __syncthreads();

  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int g = e / D, d = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w][g]);
    float Ls = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = exp2f(s_m[w][g] - M);
        Ls = fmaf(s_l[w][g], f, Ls);
        O = fmaf(s_o[w][g][d], f, O);
      }
    }
    const size_t h = (size_t)b * a.H + kvh * G + g;
    if (p.v4) {   // the merged row is in the rotated basis: rotated back below
      if (d == 0) {
        s_M[g] = M;
        s_L[g] = Ls;
      }
      s_r[g][d] = O;
      continue;
    }
    if (a.n_splits == 1) {
      a.out[h * D + d] = Ls > 0.f ? O / Ls : 0.f;
    } else {
      a.ws.part_o[(h * a.n_splits + split) * D + d] = O;
      if (d == 0) a.ws.part_ml[h * a.n_splits + split] = make_float2(M, Ls);
    }
  }
  if (!p.v4) return;
  // 4-bit V: rotate each merged row back (the FWHT is its own inverse; the combine
  // of the splits is linear in their rows, so each split's row is rotated here)
  __syncthreads();
  for (int g = warp; g < G; g += kWarps) {
    float x[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) x[i] = s_r[g][lane * VPL + i];
    fwht_row<VPL>(x, lane, fwht_norm);
    const size_t h = (size_t)b * a.H + kvh * G + g;
    const float Ls = s_L[g];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int d = lane * VPL + i;
      if (a.n_splits == 1)
        a.out[h * D + d] = Ls > 0.f ? x[i] / Ls : 0.f;
      else
        a.ws.part_o[(h * a.n_splits + split) * D + d] = x[i];
    }
    if (a.n_splits > 1 && lane == 0) a.ws.part_ml[h * a.n_splits + split] = make_float2(s_M[g], Ls);
  }
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs& a, bool k_int8, bool v_int8,
                               cudaStream_t stream) {
  const dim3 grid(a.n_splits, a.pool.Hkv, a.B);
  const float norm = (float)(1.0 / std::sqrt((double)a.pool.D));   // FWHT scaling (4-bit stores)
  switch (a.pool.D) {
    case 64:
      decode_simt_kernel<64><<<grid, kWarps * 32, 0, stream>>>(a, k_int8, v_int8, norm);
      break;
    case 128:
      decode_simt_kernel<128><<<grid, kWarps * 32, 0, stream>>>(a, k_int8, v_int8, norm);
      break;
    case 256:
      decode_simt_kernel<256><<<grid, kWarps * 32, 0, stream>>>(a, k_int8, v_int8, norm);
      break;
    default:
      return cudaErrorNotSupported;
  }
  return cudaGetLastError();
}

}  // namespace int8kv

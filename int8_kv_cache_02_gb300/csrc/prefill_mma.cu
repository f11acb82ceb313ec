// Causal attention of a chunk of new queries over the int8 cache (prefill
// chunk), on the tensor cores (mma.sync m16n8k16, f16 operands, f32 accumulate).
//
// Method: Strata pull request #2698, "What it does": the prompt chunk reads the
// int8 K/V cache dequantizing on the fly; genie-ai-runtime v1.3.1: a fused
// query-tiled attention kernel for chunks.  Query i of the chunk sits at
// absolute position start + i and sees keys 0 .. start + i.  The chunk's own
// K/V are appended (quantized) before this runs, so every key comes from the
// int8 cache.
//
// Work split.  A block takes 128 query rows of one kv head -- (position, query
// head) pairs, 128 / G positions x the G heads that share the kv head -- and a
// balanced range of its keys (split-K; partials reduced by the combine
// kernel).  Eight warps own 16 rows each.
//
// Per page (64 keys): TMA brings the int8 rows (and scales) into a two-stage
// ring as in the decode kernel; all warps convert the page once to fp16 tiles
// in shared memory (exact: |code| <= 127), laid out in the same 128-byte
// swizzle, so that q.K^T and P.V fragments come from conflict-free ldmatrix.
// Scores: per 64-value K group, S_g = Q_g K_g^T on the tensor cores, then
// S += s_k(key, g) * S_g in f32.  Softmax: online, base 2, per row, with a lazy
// reference max (moved only when exceeded by more than 2^8).  P.V: for each V
// group the weights P'(row, key) = p * s_v(key, g) * 2^(6 - e_g) go in as an
// fp16 hi + lo pair against the exact fp16 codes (the decode kernel's range
// argument: 2^e_g bounds the group's V scales seen so far, P' < 2^14).

#include <climits>

#include <cuda.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "mma_common.cuh"
#include "ptx.cuh"

namespace int8kv {
namespace {

using mma::kBoxBytes;
using mma::kMaxPolls;
using mma::kPage;
using mma::pow2f;
using mma::exponent_of;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = kWarps * 16;   // query rows (position, head) per block
constexpr float kTau = 8.f;
constexpr int kPShift = 6;
constexpr int kNS = 2;               // stages of the page ring

template <int D, bool KI8, bool VI8>
struct PLayout {
  using SP = mma::StagedPage<D, KI8, VI8>;
  static constexpr int QBOX = kRows * 128;                 // one 64-dim box of the Q tile
  static constexpr int Q_OFF = 0;
  static constexpr int Q_BYTES = kRows * D * 2;             // fp16 [D/64][128 rows][128 B]
  static constexpr int ST_OFF = Q_OFF + Q_BYTES;
  static constexpr int KH_OFF = ST_OFF + kNS * SP::STAGE;   // converted K page (fp16), K int8 only
  static constexpr int KH_BYTES = KI8 ? kPage * D * 2 : 0;
  static constexpr int VH_OFF = KH_OFF + KH_BYTES;          // converted V page (fp16), V int8 only
  static constexpr int VH_BYTES = VI8 ? kPage * D * 2 : 0;
  static constexpr int SC_OFF = VH_OFF + VH_BYTES;          // scales [K|V][group][64 keys] fp16
  static constexpr int SC_BYTES = 2 * 4 * kPage * 2;
  static constexpr int BAR_OFF = SC_OFF + SC_BYTES;
  static constexpr int SMEM = 1024 + BAR_OFF + 64;
};

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// 16 int8 codes (one 16-byte chunk) -> 16 exact fp16 values in natural order.
__device__ __forceinline__ void codes_to_f16(const uint4 w, uint4& lo, uint4& hi) {
  const uint32_t in[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u,
                          w.w ^ 0x80808080u};
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    o[2 * k] = mma::sub1152(ptx::prmt(in[k], 0x64646464u, 0x4140));
    o[2 * k + 1] = mma::sub1152(ptx::prmt(in[k], 0x64646464u, 0x4342));
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Byte offset of 16-byte chunk c of row `row` in a 64-row x 128-byte swizzled box.
__device__ __forceinline__ int swz(int row, int c) { return row * 128 + ((c ^ (row & 7)) << 4); }

// Convert one staged page: int8 codes -> fp16 tiles (same swizzled box layout as
// a TMA-loaded fp16 store), scales -> [group][key] so a thread's two adjacent keys
// are one 32-bit load.
template <int D, bool KI8, bool VI8, int NG>
__device__ __forceinline__ void convert_page(const unsigned char* sb, unsigned char* smem) {
  using LY = PLayout<D, KI8, VI8>;
  using SP = typename LY::SP;
  constexpr int CPR = D / 16;   // 16-byte code chunks per row
#pragma unroll
  for (int side = 0; side < 2; ++side) {
    const bool is8 = side == 0 ? KI8 : VI8;
    if (!is8) continue;
    const unsigned char* src = sb + (side == 0 ? SP::K_OFF : SP::V_OFF);
    unsigned char* dst = smem + (side == 0 ? LY::KH_OFF : LY::VH_OFF);
    // Eight consecutive threads take one code chunk of eight consecutive rows:
    // rows r..r+7 put the chunk at eight different swizzled positions, so both
    // the 16-byte loads and the 16-byte fp16 stores are conflict free.
    for (int c = threadIdx.x; c < kPage * CPR; c += kThreads) {
      const int g8 = c >> 3;
      const int row = (g8 / CPR) * 8 + (c & 7), cc = g8 % CPR;
      const uint4 w = *reinterpret_cast<const uint4*>(src + (cc >> 3) * kBoxBytes + swz(row, cc & 7));
      uint4 lo, hi;
      codes_to_f16(w, lo, hi);
      unsigned char* box = dst + (cc >> 2) * kBoxBytes;     // 64 fp16 dims per box
      const int c16 = (cc & 3) * 2;
      *reinterpret_cast<uint4*>(box + swz(row, c16)) = lo;
      *reinterpret_cast<uint4*>(box + swz(row, c16 + 1)) = hi;
    }
  }
  uint16_t* sc = reinterpret_cast<uint16_t*>(smem + LY::SC_OFF);
  for (int i = threadIdx.x; i < kPage * NG; i += kThreads) {
    const int row = i / NG, g = i - row * NG;
    if (KI8) sc[g * kPage + row] = reinterpret_cast<const uint16_t*>(sb + SP::KS_OFF)[i];
    if (VI8) sc[4 * kPage + g * kPage + row] = reinterpret_cast<const uint16_t*>(sb + SP::VS_OFF)[i];
  }
}

template <int D, bool KI8, bool VI8, int NG>
__global__ void __launch_bounds__(kThreads, 1)
prefill_mma_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, int layer_page0) {
  using LY = PLayout<D, KI8, VI8>;
  using SP = typename LY::SP;
  constexpr int NT = D / 8;                 // 8-dim output n-tiles per row
  constexpr int NGK = KI8 ? NG : 1;         // K scale groups
  constexpr int NGV = VI8 ? NG : 1;         // V scale groups
  constexpr int KSG = D / 16 / NGK;         // 16-dim k-steps per K group
  constexpr int NTG = NT / NGV;             // output n-tiles per V group
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + LY::BAR_OFF);
  int* stage_page = reinterpret_cast<int*>(full + kNS);

  const int qt = blockIdx.x, kvh = blockIdx.y, split = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, r = lane >> 2, t = lane & 3;
  const PoolView& p = a.pool;
  const int G = a.G, ppb = kRows / G, pos0 = qt * ppb;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) ptx::mbar_init(&full[s], 1);
    ptx::fence_mbar_init();
  }
  const int last_pos = min(pos0 + ppb, a.n_new) - 1;
  const int hi_key = a.start + last_pos + 1;            // keys [0, hi_key) for this block
  int j0, j1;
  split_range(0, hi_key, split, a.n_splits, kPage, &j0, &j1);
  const int p_first = j0 / kPage;
  const int n_pg = j1 > j0 ? (j1 - 1) / kPage - p_first + 1 : 0;

  // q rows -> shared memory (rows past the chunk are zero)
  for (int c = threadIdx.x; c < kRows * (D / 8); c += kThreads) {
    const int R = c / (D / 8), ch = c - R * (D / 8);
    const int pos = pos0 + R / G;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (pos < a.n_new)
      v = ptx::ldg128(a.q + ((size_t)pos * a.H + (size_t)kvh * G + R % G) * D + ch * 8);
    *reinterpret_cast<uint4*>(smem + LY::Q_OFF + (ch >> 3) * LY::QBOX + swz(R, ch & 7)) = v;
  }
  __syncthreads();
  const int32_t* ptrow = a.page_table;
  auto page_row = [&](int page) { return ((layer_page0 + page) * p.Hkv + kvh) * kPage; };
  auto issue = [&](int i) {
    const int st = i % kNS;
    const int page = lookup_page(ptrow, p_first + i, a.max_pages, p);
    mma::issue_page<D, KI8, VI8>(smem + LY::ST_OFF + st * SP::STAGE, &full[st], &stage_page[st],
                                 page, page_row(page), p, kvh, &tmk, &tmv);
  };
  if (threadIdx.x == 0) {
    ptx::prefetch_tensormap(&tmk);
    ptx::prefetch_tensormap(&tmv);
    for (int i = 0; i < n_pg && i < kNS; ++i) issue(i);
  }

  // rows of this thread: R0 = warp*16 + r and R1 = R0 + 8
  const int R0 = warp * 16 + r, R1 = R0 + 8;
  const int posA = pos0 + R0 / G, posB = pos0 + R1 / G;
  const int limA = posA < a.n_new ? a.start + posA : -1;   // last key each row sees
  const int limB = posB < a.n_new ? a.start + posB : -1;
  const int lim_lo = min(limA, limB);

  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  int vexp[NGV];
  float cap[NGV], sh[NGV];
#pragma unroll
  for (int g = 0; g < NGV; ++g) {
    vexp[g] = INT_MIN;
    cap[g] = 0.f;
    sh[g] = 0.f;
  }

  for (int i = 0; i < n_pg; ++i) {
    const int st = i % kNS;
    // every thread waits (bounded); the block leaves together if any wait expired
    const bool expired = !ptx::mbar_wait(&full[st], (i / kNS) & 1, kMaxPolls);
    if (__syncthreads_or(expired)) {
      if (threadIdx.x == 0) flag_error(p.err, INT8KV_DEVERR_TIMEOUT);
      break;
    }
    const unsigned char* sb = smem + LY::ST_OFF + st * SP::STAGE;
    const int page = stage_page[st];
    if (page >= 0) convert_page<D, KI8, VI8, NG>(sb, smem);
    __syncthreads();
    if (KI8 && VI8 && threadIdx.x == 0 && i + kNS < n_pg) {   // stage fully read by the conversion
      ptx::fence_proxy_async();
      issue(i + kNS);
    }
    const int key0 = (p_first + i) * kPage;
    if (page >= 0) {
      const unsigned char* kt = KI8 ? smem + LY::KH_OFF : sb + SP::K_OFF;
      const unsigned char* vt = VI8 ? smem + LY::VH_OFF : sb + SP::V_OFF;
      const uint16_t* sck = reinterpret_cast<const uint16_t*>(smem + LY::SC_OFF);
      const uint16_t* scv = sck + 4 * kPage;
      const bool full_page = key0 >= j0 && key0 + kPage <= j1 && key0 + kPage - 1 <= lim_lo;

      // ---- scores s[j][*]: n-tile j = keys key0 + 8j + (2t, 2t+1), rows R0 (0,1) R1 (2,3)
      float s[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
      for (int g = 0; g < NGK; ++g) {
        float sg[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) sg[j][0] = sg[j][1] = sg[j][2] = sg[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KSG; ++kk) {
          const int ks = g * KSG + kk;        // 16-dim k-step
          const int q4 = lane >> 3, rr = lane & 7;
          uint32_t af[4];
          {
            const int R = warp * 16 + rr + 8 * (q4 & 1);
            const int ch = ks * 2 + (q4 >> 1);
            ptx::ldmatrix_x4(af, ptx::smem_u32(smem + LY::Q_OFF + (ch >> 3) * LY::QBOX +
                                               swz(R, ch & 7)));
          }
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int key = 16 * jj + rr + 8 * (q4 >> 1);
            const int ch = ks * 2 + (q4 & 1);
            uint32_t bf[4];
            ptx::ldmatrix_x4(bf, ptx::smem_u32(kt + (ch >> 3) * kBoxBytes + swz(key, ch & 7)));
            ptx::mma_f16(sg[2 * jj], af, bf[0], bf[1]);
            ptx::mma_f16(sg[2 * jj + 1], af, bf[2], bf[3]);
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float s0 = a.scale_log2, s1 = a.scale_log2;
          if constexpr (KI8) {
            const __half2 h = *reinterpret_cast<const __half2*>(sck + g * kPage + 8 * j + 2 * t);
            const float2 f = __half22float2(h);
            s0 *= f.x;
            s1 *= f.y;
          }
          s[j][0] = fmaf(sg[j][0], s0, s[j][0]);
          s[j][1] = fmaf(sg[j][1], s1, s[j][1]);
          s[j][2] = fmaf(sg[j][2], s0, s[j][2]);
          s[j][3] = fmaf(sg[j][3], s1, s[j][3]);
        }
      }
      if (!full_page) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = key0 + 8 * j + 2 * t + e;
            const bool in = key >= j0 && key < j1;
            if (!(in && key <= limA)) s[j][e] = -INFINITY;
            if (!(in && key <= limB)) s[j][2 + e] = -INFINITY;
          }
      }

      // ---- online softmax per row (quad lanes share a row), lazy reference max
      float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        mxA = fmaxf(mxA, fmaxf(s[j][0], s[j][1]));
        mxB = fmaxf(mxB, fmaxf(s[j][2], s[j][3]));
      }
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, off));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, off));
      }
      if (__any_sync(0xffffffffu, mxA > mA + kTau || mxB > mB + kTau)) {
        const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
        const float alA = nA == -INFINITY ? 1.f : ptx::ex2(mA - nA);
        const float alB = nB == -INFINITY ? 1.f : ptx::ex2(mB - nB);
        lA *= alA;
        lB *= alB;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          o[n][0] *= alA;
          o[n][1] *= alA;
          o[n][2] *= alB;
          o[n][3] *= alB;
        }
        mA = nA;
        mB = nB;
      }
      const float bA = mA == -INFINITY ? 0.f : mA, bB = mB == -INFINITY ? 0.f : mB;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        s[j][0] = ptx::ex2(s[j][0] - bA);
        s[j][1] = ptx::ex2(s[j][1] - bA);
        s[j][2] = ptx::ex2(s[j][2] - bB);
        s[j][3] = ptx::ex2(s[j][3] - bB);
        lA += s[j][0] + s[j][1];
        lB += s[j][2] + s[j][3];
      }

      // ---- P.V per V group
#pragma unroll
      for (int g = 0; g < NGV; ++g) {
        float w[8][2];   // per n-tile: weights of keys 2t, 2t+1
        if constexpr (VI8) {
          bool need = false;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const __half2 h = *reinterpret_cast<const __half2*>(scv + g * kPage + 8 * j + 2 * t);
            const float2 f = __half22float2(h);
            w[j][0] = f.x;
            w[j][1] = f.y;
            if (!full_page) {
              const int key = key0 + 8 * j + 2 * t;
              if (!(key >= j0 && key < j1)) w[j][0] = 0.f;
              if (!(key + 1 >= j0 && key + 1 < j1)) w[j][1] = 0.f;
            }
            need |= (w[j][0] > 0.f && w[j][0] >= cap[g]) || (w[j][1] > 0.f && w[j][1] >= cap[g]);
          }
          if (__any_sync(0xffffffffu, need)) {
            float mx = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fmaxf(w[j][0], w[j][1]));
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            if (mx > 0.f && mx >= cap[g]) {
              const int ne = exponent_of(mx) + 1;
              if (vexp[g] != INT_MIN) {
                const float f = pow2f(vexp[g] - ne);
#pragma unroll
                for (int n = g * NTG; n < (g + 1) * NTG; ++n) {
                  o[n][0] *= f;
                  o[n][1] *= f;
                  o[n][2] *= f;
                  o[n][3] *= f;
                }
              }
              vexp[g] = ne;
              cap[g] = pow2f(ne);
              sh[g] = pow2f(kPShift - ne);
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            w[j][0] *= sh[g];
            w[j][1] *= sh[g];
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            w[j][0] = w[j][1] = pow2f(kPShift);
            if (!full_page) {
              const int key = key0 + 8 * j + 2 * t;
              if (!(key >= j0 && key < j1)) w[j][0] = 0.f;
              if (!(key + 1 >= j0 && key + 1 < j1)) w[j][1] = 0.f;
            }
          }
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {   // 16 keys: n-tiles 2kk, 2kk+1 of the scores
          uint32_t ah[4], al[4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int j = 2 * kk + h;
            const float p0 = s[j][0] * w[j][0], p1 = s[j][1] * w[j][1];
            const float p2 = s[j][2] * w[j][0], p3 = s[j][3] * w[j][1];
            const uint32_t x01 = ptx::pack_f16x2(p0, p1), x23 = ptx::pack_f16x2(p2, p3);
            const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&x01));
            const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&x23));
            ah[2 * h] = x01;
            ah[2 * h + 1] = x23;
            al[2 * h] = ptx::pack_f16x2(p0 - f01.x, p1 - f01.y);
            al[2 * h + 1] = ptx::pack_f16x2(p2 - f23.x, p3 - f23.y);
          }
          // A fragment order: (row r, keys 2t..), (row r+8, keys 2t..), (row r, keys 8+2t..), (row r+8, ..)
          const uint32_t Ah[4] = {ah[0], ah[1], ah[2], ah[3]};
          const uint32_t Al[4] = {al[0], al[1], al[2], al[3]};
          const int q4 = lane >> 3, rr = lane & 7;
          const int key = 16 * kk + rr + 8 * (q4 & 1);
          uint32_t kmask_lo = 0xFFFFFFFFu, kmask_hi = 0xFFFFFFFFu;
          if constexpr (!VI8) {
            if (!full_page) {   // fp16 V rows outside [j0, j1) may hold any bits
              const int k0 = key0 + 16 * kk + 2 * t;
              kmask_lo = ((k0 >= j0 && k0 < j1) ? 0x0000FFFFu : 0u) |
                         ((k0 + 1 >= j0 && k0 + 1 < j1) ? 0xFFFF0000u : 0u);
              kmask_hi = ((k0 + 8 >= j0 && k0 + 8 < j1) ? 0x0000FFFFu : 0u) |
                         ((k0 + 9 >= j0 && k0 + 9 < j1) ? 0xFFFF0000u : 0u);
            }
          }
#pragma unroll
          for (int nn = 0; nn < NTG / 2; ++nn) {   // pairs of 8-dim n-tiles of this group
            const int n = g * NTG + 2 * nn;
            const int ch = n + (q4 >> 1);          // 8-dim chunk (fp16) of this lane's row
            uint32_t bf[4];
            ptx::ldmatrix_x4_trans(bf, ptx::smem_u32(vt + (ch >> 3) * kBoxBytes + swz(key, ch & 7)));
            if constexpr (!VI8) {
              bf[0] &= kmask_lo;
              bf[1] &= kmask_hi;
              bf[2] &= kmask_lo;
              bf[3] &= kmask_hi;
            }
            ptx::mma_f16(o[n], Ah, bf[0], bf[1]);
            ptx::mma_f16(o[n + 1], Ah, bf[2], bf[3]);
            ptx::mma_f16(o[n], Al, bf[0], bf[1]);
            ptx::mma_f16(o[n + 1], Al, bf[2], bf[3]);
          }
        }
      }
    }
    __syncthreads();   // the converted tiles (or the stage itself) are free again
    if (!(KI8 && VI8) && threadIdx.x == 0 && i + kNS < n_pg) {
      ptx::fence_proxy_async();
      issue(i + kNS);
    }
  }

  // ---- epilogue: rows R0 (position posA) and R1 (posB)
  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);
  const size_t hA = (size_t)posA * a.H + (size_t)kvh * G + R0 % G;
  const size_t hB = (size_t)posB * a.H + (size_t)kvh * G + R1 % G;
  const bool wA = posA < a.n_new, wB = posB < a.n_new;
  const int S = a.n_splits;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int g = n / NTG;
    float u = pow2f(-kPShift);
    if constexpr (VI8) u = vexp[g] == INT_MIN ? 0.f : pow2f(vexp[g] - kPShift);
    const int d = 8 * n + 2 * t;
    if (S == 1) {
      const float iA = lA > 0.f ? u / lA : 0.f, iB = lB > 0.f ? u / lB : 0.f;
      if (wA) *reinterpret_cast<float2*>(a.out + hA * D + d) = make_float2(o[n][0] * iA, o[n][1] * iA);
      if (wB) *reinterpret_cast<float2*>(a.out + hB * D + d) = make_float2(o[n][2] * iB, o[n][3] * iB);
    } else {
      if (wA)
        *reinterpret_cast<float2*>(a.ws.part_o + (hA * S + split) * D + d) =
            make_float2(o[n][0] * u, o[n][1] * u);
      if (wB)
        *reinterpret_cast<float2*>(a.ws.part_o + (hB * S + split) * D + d) =
            make_float2(o[n][2] * u, o[n][3] * u);
    }
  }
  if (S > 1 && t == 0) {
    if (wA) a.ws.part_ml[hA * S + split] = make_float2(mA, lA);
    if (wB) a.ws.part_ml[hB * S + split] = make_float2(mB, lB);
  }
}

template <int D, bool KI8, bool VI8, int NG>
cudaError_t launch_typed(const PrefillArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                         int layer_page0, cudaStream_t stream) {
  using LY = PLayout<D, KI8, VI8>;
  auto kern = prefill_mma_kernel<D, KI8, VI8, NG>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::SMEM);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = true;
  }
  const int ppb = kRows / a.G;
  const dim3 grid((a.n_new + ppb - 1) / ppb, a.pool.Hkv, a.n_splits);
  kern<<<grid, kThreads, LY::SMEM, stream>>>(a, tmk, tmv, layer_page0);
  return cudaGetLastError();
}

template <int D, bool KI8, bool VI8>
cudaError_t launch_ng(const PrefillArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                      int layer_page0, cudaStream_t stream) {
  switch (a.pool.ng) {
    case 1: return launch_typed<D, KI8, VI8, 1>(a, tmk, tmv, layer_page0, stream);
    case 2: return launch_typed<D, KI8, VI8, 2>(a, tmk, tmv, layer_page0, stream);
    case 4:
      if constexpr (D == 256) return launch_typed<D, KI8, VI8, 4>(a, tmk, tmv, layer_page0, stream);
      return cudaErrorNotSupported;
    default: return cudaErrorNotSupported;
  }
}

}  // namespace

bool prefill_supported(const int8kv_pool* pool, int G) {
  return pool->has_tmaps && pool->page_size == kPage && pool->group_size >= 64 &&
         (pool->head_dim == 128 || pool->head_dim == 256) && (G == 1 || G == 2 || G == 4 || G == 8);
}

cudaError_t launch_prefill(const int8kv_pool* pool, int layer, const PrefillArgs& a,
                           cudaStream_t stream) {
  cudaError_t e;
  const int lp0 = layer * pool->n_pages;
  const bool k8 = pool->k_int8, v8 = pool->v_int8;
  if (pool->head_dim == 256) {
    if (k8 && v8) e = launch_ng<256, true, true>(a, pool->tmap_k, pool->tmap_v, lp0, stream);
    else if (k8) e = launch_ng<256, true, false>(a, pool->tmap_k, pool->tmap_v, lp0, stream);
    else e = launch_ng<256, false, true>(a, pool->tmap_k, pool->tmap_v, lp0, stream);
  } else {
    if (k8 && v8) e = launch_ng<128, true, true>(a, pool->tmap_k, pool->tmap_v, lp0, stream);
    else if (k8) e = launch_ng<128, true, false>(a, pool->tmap_k, pool->tmap_v, lp0, stream);
    else e = launch_ng<128, false, true>(a, pool->tmap_k, pool->tmap_v, lp0, stream);
  }
  if (e != cudaSuccess || a.n_splits == 1) return e;
  DecodeArgs c{};
  c.pool = a.pool;
  c.out = a.out;
  c.ws = a.ws;
  c.B = a.n_new;
  c.H = a.H;
  c.G = a.G;
  c.n_splits = a.n_splits;
  return launch_decode_combine(c, stream);
}

}  // namespace int8kv

// Causal attention of a chunk of new queries over the int8 cache (prefill
// chunk) on the 5th-generation tensor cores: tcgen05.mma with operands in
// shared memory and tensor memory, accumulators in tensor memory.
//
// Method: Strata pull request #2698, "What it does" (the prompt chunk reads the
// int8 K/V cache dequantizing on the fly) and genie-ai-runtime v1.3.1 (a fused
// query-tiled attention kernel for chunks).  Query i of the chunk sits at
// absolute position start + i and sees keys 0 .. start + i; the chunk's own
// K/V are appended (quantized) before this runs.
//
// Work split.  A block takes 128 query rows of one kv head -- (position, head)
// pairs, 128 / G positions x the G heads sharing the kv head -- and a balanced
// range of its keys (split-K; the combine kernel reduces the partials).  Row R
// is thread R and tensor-memory lane R.
//
// Per page of 64 keys:
//   1. TMA brings the K/V rows and scales (a two-stage ring).  int8 rows are
//      converted once to fp16 tiles in shared memory (exact: |code| <= 127),
//      laid out as 128-byte-swizzled K-major boxes [D/64][64 keys][128 B].
//   2. Thread 0 issues S_g = Q_g K_g^T per 64-value K scale group g
//      (M = 128 rows, N = 64 keys, K = 16 per instruction) into tensor memory.
//   3. Four threads per row (warps w, w + 4, w + 8, w + 12 share tensor-memory
//      lanes) each read a quarter of the row's S_g (16 keys), form
//      s = scale * sum_g s_k * S_g, mask, and run the online softmax (lazy
//      reference max, base 2; the quarters' maxima meet in shared memory).
//      They write P' = p * s_v * 2^(6 - e_g) per V scale group as an fp16
//      hi + lo pair back into tensor memory, over the S columns they have read.
//   4. Thread 0 issues O += P'_hi V + P'_lo V with P' from tensor memory and V
//      from shared memory (MN-major: dims contiguous), N = 64 dims per
//      instruction.  O (128 rows x D fp32) lives in tensor memory throughout;
//      the rare rescales (reference max or V range moved) read and rewrite a
//      thread's own row.
// Completion of each MMA batch is signalled by tcgen05.commit on an mbarrier;
// every wait is bounded and sets a device error bit on expiry.

#include <climits>

#include <cuda.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "mma_common.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace int8kv {
namespace {

using mma::kBoxBytes;
using mma::kMaxPolls;
using mma::kPage;
using mma::pow2f;
using mma::exponent_of;

constexpr int kRows = 128;            // query rows per block = tensor-memory lanes
constexpr int kParts = 4;             // threads per row: each takes 16 of the 64 keys of a page
constexpr int kThreads = kParts * kRows;   // and D / kParts of the output columns
constexpr int kChunks = 4 / kParts;   // 16-key chunks per thread
constexpr int kNS = 2;                // stages of the page ring
constexpr float kTau = 8.f;           // lazy rescale threshold (log2 units)
constexpr int kPShift = 6;            // P' < 2^8 * 2^6 in fp16
constexpr int kPSplit = 5;            // weights formed as p * 2^5 (<= 2^13; the exponent's base
                                      // lowered by 5, the row sums dropping the 2^5 at the end)
                                      // and split into fp16 hi + lo, the P.V factors carrying
                                      // 2^-5: weights down to 2^-19 of the reference and V
                                      // scales down to 2^-15 of the group's range stay normal

template <int D, bool KI8, bool VI8, int NG>
struct TLayout {
  using SP = mma::StagedPage<D, KI8, VI8>;
  static constexpr int NGK = KI8 ? NG : 1;                  // K scale groups
  static constexpr int NGV = VI8 ? NG : 1;                  // V scale groups
  static constexpr int QBOX = kRows * 128;                  // one 64-dim box of the Q tile
  static constexpr int Q_OFF = 0;                           // fp16 [D/64][128 rows][128 B]
  static constexpr int ST_OFF = Q_OFF + kRows * D * 2;      // page ring
  static constexpr int KH_OFF = ST_OFF + kNS * SP::STAGE;   // converted K page (int8 K only)
  static constexpr int VH_OFF = KH_OFF + (KI8 ? kPage * D * 2 : 0);   // converted V page
  static constexpr int KSF_OFF = VH_OFF + (VI8 ? kPage * D * 2 : 0);   // fp32 K scales x scale [key][NG]
  static constexpr int VSF_OFF = KSF_OFF + kPage * 4 * 4;               // fp16 P.V factors [NG][key]
  static constexpr int BAR_OFF = VSF_OFF + kPage * 4 * 4;
  static constexpr int SMEM = 1024 + BAR_OFF + 128;
  // tensor memory: S_g / P'_g region, then O
  static constexpr int SREG = (NGK > NGV ? NGK : NGV) * 64;
  static constexpr int OB = SREG;
  static constexpr int TCOLS = SREG + D <= 256 ? 256 : 512;
  static_assert(SREG + D <= 512, "tensor memory holds S and O");
};

__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int b_mn) {
  return tc::idesc_f16(M, N, 0, b_mn);   // A K-major
}
using tc::sdesc;
using tc::mma_ss;
using tc::mma_ts;
using tc::mma_commit;
__device__ __forceinline__ void tc_fence_before() { tc::fence_before(); }
__device__ __forceinline__ void tc_fence_after() { tc::fence_after(); }
__device__ __forceinline__ void tmem_ld16(uint32_t ta, uint32_t (&v)[16]) { tc::ld16(ta, v); }
__device__ __forceinline__ void tmem_st16(uint32_t ta, const uint32_t (&v)[16]) { tc::st16(ta, v); }
__device__ __forceinline__ void tmem_wait_ld() { tc::wait_ld(); }
__device__ __forceinline__ void tmem_wait_st() { tc::wait_st(); }

// Multiply this lane's columns [c0, c0 + n) of tensor memory by f.
__device__ __forceinline__ void tmem_scale(uint32_t ta, int n, float f) {
  for (int c = 0; c < n; c += 16) {
    uint32_t v[16];
    tmem_ld16(ta + c, v);
    tmem_wait_ld();
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * f);
    tmem_st16(ta + c, v);
  }
  tmem_wait_st();
}

__device__ __forceinline__ int swz(int row, int c) { return row * 128 + ((c ^ (row & 7)) << 4); }

// 16 int8 codes -> 16 exact fp16 values, two per operation: bytes 0 and 2 of a
// word, then 1 and 3, so inside each group of four dims, positions 1 and 2 hold
// dims 2 and 1 (the Q tile is stored in the same order, and O's columns are
// read back through it).
__device__ __forceinline__ void codes_to_f16(const uint4 w, uint4& lo, uint4& hi) {
  using mma::lop_i8pair;
  using mma::sub1152;
  lo = make_uint4(sub1152(lop_i8pair(w.x)), sub1152(lop_i8pair(w.x >> 8)),
                  sub1152(lop_i8pair(w.y)), sub1152(lop_i8pair(w.y >> 8)));
  hi = make_uint4(sub1152(lop_i8pair(w.z)), sub1152(lop_i8pair(w.z >> 8)),
                  sub1152(lop_i8pair(w.w)), sub1152(lop_i8pair(w.w >> 8)));
}

// Dims of 8 consecutive fp16 values (one 16-byte chunk) in that order.
__device__ __forceinline__ uint4 pair_order(const uint4 x) {
  return make_uint4(ptx::prmt(x.x, x.y, 0x5410), ptx::prmt(x.x, x.y, 0x7632),
                    ptx::prmt(x.z, x.w, 0x5410), ptx::prmt(x.z, x.w, 0x7632));
}

// int8 rows of one side (K or V) of a staged page -> fp16 boxes [D/64][64][128 B].
// Eight consecutive threads take one code chunk of eight consecutive rows, so
// loads and stores hit eight different swizzled positions; every thread's
// loads are in flight before its first conversion.
template <int D>
__device__ __forceinline__ void convert_side(const unsigned char* src, unsigned char* dst) {
  constexpr int CPR = D / 16;                       // 16-byte code chunks per row
  constexpr int PER = kPage * CPR / kThreads;       // chunks per thread
  static_assert(PER * kThreads == kPage * CPR, "whole chunks per thread");
  uint4 w[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int c = threadIdx.x + k * kThreads, g8 = c >> 3;
    const int row = (g8 / CPR) * 8 + (c & 7), cc = g8 % CPR;
    w[k] = *reinterpret_cast<const uint4*>(src + (cc >> 3) * kBoxBytes + swz(row, cc & 7));
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int c = threadIdx.x + k * kThreads, g8 = c >> 3;
    const int row = (g8 / CPR) * 8 + (c & 7), cc = g8 % CPR;
    uint4 lo, hi;
    codes_to_f16(w[k], lo, hi);
    unsigned char* box = dst + (cc >> 2) * kBoxBytes;
    const int c16 = (cc & 3) * 2;
    *reinterpret_cast<uint4*>(box + swz(row, c16)) = lo;
    *reinterpret_cast<uint4*>(box + swz(row, c16 + 1)) = hi;
  }
}

// The same over threads [t0, kThreads) only (the first warp issues the score
// MMAs meanwhile): chunk c of thread t is t - t0 + k * (kThreads - t0).
template <int D, int T0>
__device__ __forceinline__ void convert_side_from(const unsigned char* src, unsigned char* dst) {
  constexpr int CPR = D / 16;
  constexpr int NT = kThreads - T0;
  constexpr int N = kPage * CPR;
  constexpr int PER = (N + NT - 1) / NT;
  const int me = (int)threadIdx.x - T0;
  if (me < 0) return;
  uint4 w[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int c = me + k * NT;
    if (c < N) {
      const int g8 = c >> 3, row = (g8 / CPR) * 8 + (c & 7), cc = g8 % CPR;
      w[k] = *reinterpret_cast<const uint4*>(src + (cc >> 3) * kBoxBytes + swz(row, cc & 7));
    }
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int c = me + k * NT;
    if (c < N) {
      const int g8 = c >> 3, row = (g8 / CPR) * 8 + (c & 7), cc = g8 % CPR;
      uint4 lo, hi;
      codes_to_f16(w[k], lo, hi);
      unsigned char* box = dst + (cc >> 2) * kBoxBytes;
      const int c16 = (cc & 3) * 2;
      *reinterpret_cast<uint4*>(box + swz(row, c16)) = lo;
      *reinterpret_cast<uint4*>(box + swz(row, c16 + 1)) = hi;
    }
  }
}

// The copies of one page as mma::issue_page makes them (the K side, the V side,
// then the K and V scales rows of an int8 side), for one copy at a time: copy c
// of kCopies, and the bytes the stage's barrier expects for all of them.
template <int D, bool KI8, bool VI8>
struct PageCopies {
  using SP = mma::StagedPage<D, KI8, VI8>;
  static constexpr int kCopies = 2 + (KI8 ? 1 : 0) + (VI8 ? 1 : 0);   // K, V (3-D when several boxes), scales
  static __device__ __forceinline__ uint32_t tx(int ng) {
    return SP::KBYTES + SP::VBYTES + (KI8 ? kPage * ng * 2 : 0) + (VI8 ? kPage * ng * 2 : 0);
  }
  static __device__ __forceinline__ void issue(int c, unsigned char* stage, uint64_t* full_bar,
                                               int page, int row, const PoolView& p, int kvh,
                                               const CUtensorMap* tmk, const CUtensorMap* tmv) {
    const size_t srow = ((size_t)page * p.Hkv + kvh) * kPage * p.ng;
    if (c == 0) {
      if constexpr (SP::KBOXES > 1)
        ptx::tma_load_3d(stage + SP::K_OFF, tmk, 0, row, 0, full_bar);
      else
        ptx::tma_load_2d(stage + SP::K_OFF, tmk, 0, row, full_bar);
    } else if (c == 1) {
      if constexpr (SP::VBOXES > 1)
        ptx::tma_load_3d(stage + SP::V_OFF, tmv, 0, row, 0, full_bar);
      else
        ptx::tma_load_2d(stage + SP::V_OFF, tmv, 0, row, full_bar);
    } else if (KI8 && c == 2) {
      ptx::bulk_load(stage + SP::KS_OFF, p.ks + srow, kPage * p.ng * 2, full_bar);
    } else if (VI8) {
      ptx::bulk_load(stage + SP::VS_OFF, p.vs + srow, kPage * p.ng * 2, full_bar);
    }
  }
};

// Zero the fp16 rows of a staged side whose keys fall outside [j0, j1) (they
// may hold any bits, and 0 * NaN would reach O).
template <int D>
__device__ __forceinline__ void zero_rows(unsigned char* side, int key0, int j0, int j1) {
  for (int c = threadIdx.x; c < kPage * (D / 8); c += kThreads) {
    const int row = c / (D / 8), ch = c % (D / 8);
    const int key = key0 + row;
    if (key < j0 || key >= j1)
      *reinterpret_cast<uint4*>(side + (ch >> 3) * kBoxBytes + row * 128 + ((ch & 7) << 4)) =
          make_uint4(0, 0, 0, 0);
  }
}

template <int D, bool KI8, bool VI8, int NG>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, int layer_page0) {
  using LY = TLayout<D, KI8, VI8, NG>;
  using SP = typename LY::SP;
  constexpr int NGK = LY::NGK, NGV = LY::NGV;
  constexpr int KSG = D / 16 / NGK;        // 16-dim k-steps per K group
  constexpr int BPG = D / 64 / NGV;        // 64-dim boxes per V group
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + LY::BAR_OFF);   // [kNS]
  uint64_t* mS = full + kNS;                                           // S batch done
  uint64_t* mO = mS + 1;                                               // P.V batch done
  int* stage_page = reinterpret_cast<int*>(mO + 1);                    // [kNS]
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(stage_page + kNS);
  __shared__ int s_fail;

  const int qt = blockIdx.x, kvh = blockIdx.y, split = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int R = tid & (kRows - 1), half = tid / kRows;   // row, and which part of it
  const PoolView& p = a.pool;
  const int G = a.G, ppb = kRows / G, pos0 = qt * ppb;

  if (tid == 0) {
    for (int s = 0; s < kNS; ++s) ptx::mbar_init(&full[s], 1);
    ptx::mbar_init(mS, 1);
    ptx::mbar_init(mO, 1);
    ptx::fence_mbar_init();
    s_fail = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     ptx::smem_u32(taddr_s)),
                 "r"((uint32_t)LY::TCOLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }

  const int last_pos = min(pos0 + ppb, a.n_new) - 1;
  const int hi_key = a.start + last_pos + 1;   // keys [0, hi_key) for this block
  int j0, j1;
  split_range(0, hi_key, split, a.n_splits, kPage, &j0, &j1);
  const int p_first = j0 / kPage;
  const int n_pg = j1 > j0 ? (j1 - 1) / kPage - p_first + 1 : 0;

  // q rows -> shared memory (rows past the chunk are zero)
  for (int c = tid; c < kRows * (D / 8); c += kThreads) {
    const int row = c / (D / 8), ch = c - row * (D / 8);
    const int pos = pos0 + row / G;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (pos < a.n_new) {
      v = ptx::ldg128(a.q + ((size_t)pos * a.H + (size_t)kvh * G + row % G) * D + ch * 8);
      if constexpr (KI8) v = pair_order(v);   // the order of the converted K tiles
    }
    *reinterpret_cast<uint4*>(smem + LY::Q_OFF + (ch >> 3) * LY::QBOX + swz(row, ch & 7)) = v;
  }
  ptx::fence_proxy_async();   // generic writes of the Q tile before the tensor-core reads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *taddr_s;
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;   // this warp's tensor-memory lanes

  const int32_t* ptrow = a.page_table;
  auto page_row = [&](int page) { return ((layer_page0 + page) * p.Hkv + kvh) * kPage; };
  auto issue_id = [&](int i, int page) {   // page: a checked id, or -1
    const int st = i % kNS;
    mma::issue_page<D, KI8, VI8>(smem + LY::ST_OFF + st * SP::STAGE, &full[st], &stage_page[st],
                                 page, page_row(page), p, kvh, &tmk, &tmv);
  };
  auto issue = [&](int i) { issue_id(i, lookup_page(ptrow, p_first + i, a.max_pages, p)); };
  if (tid == 0) {
    ptx::prefetch_tensormap(&tmk);
    ptx::prefetch_tensormap(&tmv);
    for (int i = 0; i < n_pg && i < kNS; ++i) issue(i);
  }

  const int pos = pos0 + R / G;
  const int lim = pos < a.n_new ? a.start + pos : -1;   // last key this row sees
  float m = -INFINITY, l = 0.f;
  int vexp[NGV];
  float cap[NGV], sh[NGV];
#pragma unroll
  for (int g = 0; g < NGV; ++g) {
    vexp[g] = INT_MIN;
    cap[g] = 0.f;
    sh[g] = 0.f;
  }
  constexpr uint32_t idS = idesc_f16(128, 64, 0), idO = idesc_f16(128, 64, 1);
  bool o_live = false;   // some P.V batch has written O
  int nS = 0, nO = 0;    // S and P.V batches committed so far (one mbarrier phase each)
  __shared__ float s_vmax[4];
  __shared__ float s_mx[kParts][kRows];   // the parts' score maxima (then sums) of each row

  constexpr int kRefill = 32;   // the thread that refills the ring (not in the issuing warp)
  for (int i = 0; i < n_pg; ++i) {
    const int st = i % kNS;
    // the id of the page the freed stage takes next: loaded now, checked at use,
    // so that the load's latency passes under the wait and the K conversion
    const int ri = i - 1 + kNS;
    const bool refill = tid == kRefill && i > 0 && ri < n_pg;
    const bool ri_in_row = p_first + ri < a.max_pages;
    int raw_next = -1;
    if (refill && ri_in_row) raw_next = ptx::ldg32(ptrow + p_first + ri);
    bool bad = !ptx::mbar_wait(&full[st], (i / kNS) & 1, kMaxPolls);
    unsigned char* sb = smem + LY::ST_OFF + st * SP::STAGE;
    const int page = stage_page[st];
    const int key0 = (p_first + i) * kPage;
    const bool edge = key0 < j0 || key0 + kPage > j1;
    // K side first: the K tile and table were last read by the previous page's
    // q.K and softmax, both done, so this overlaps the previous P.V batch
    if (!bad && page >= 0) {
      if constexpr (KI8) convert_side<D>(sb + SP::K_OFF, smem + LY::KH_OFF);
      if constexpr (!KI8) if (edge) zero_rows<D>(sb + SP::K_OFF, key0, j0, j1);
      if constexpr (KI8)   // K scales times the softmax scale
        if (tid < kPage * NG)
          reinterpret_cast<float*>(smem + LY::KSF_OFF)[tid] =
              __half2float(reinterpret_cast<const __half*>(sb + SP::KS_OFF)[tid]) * a.scale_log2;
      // Each group's largest V scale among the keys in [j0, j1) (warp 1 + g takes
      // group g) is formed here, in the wait for the previous P.V batch.
      if constexpr (VI8) {
        const int g = warp - 1;
        if (g >= 0 && g < NGV) {
          const uint16_t* vs = reinterpret_cast<const uint16_t*>(sb + SP::VS_OFF);
          const int lane = tid & 31;
          float mv = 0.f;
#pragma unroll
          for (int e = 0; e < 2; ++e) {   // keys 2 lane, 2 lane + 1
            const int k = 2 * lane + e;
            if (key0 + k >= j0 && key0 + k < j1)
              mv = fmaxf(mv, __half2float(__ushort_as_half(vs[k * NG + g])));
          }
          mv = warp_max(mv);
          if (lane == 0) s_vmax[g] = mv;
        }
      }
    }
    // the previous P.V batch is done: its V tile, P' columns and stage are free
    if (nO > 0 && !bad) bad = !ptx::mbar_wait(mO, (nO - 1) & 1, kMaxPolls);
    ptx::fence_proxy_async();   // the converted K tile, before the tensor-core reads
    tc_fence_before();
    if (__syncthreads_or(bad)) {
      if (tid == 0) s_fail = 1;
      break;
    }
    tc_fence_after();

    // ---- S_g = Q_g K_g^T into columns [64g, 64g + 64): issued now (the S
    // columns were freed with the P.V batch), so that it runs while the other
    // warps convert the V side.  Warp 0 (descriptors warp-uniform); one elected
    // lane issues.
    if (page >= 0 && warp == 0) {
      const uint64_t da0 = sdesc(ptx::smem_u32(smem + LY::Q_OFF), 16, 1024);
      const uint64_t db0 = sdesc(ptx::smem_u32(KI8 ? smem + LY::KH_OFF : sb + SP::K_OFF), 16, 1024);
      if (ptx::elect_one()) {
#pragma unroll
        for (int g = 0; g < NGK; ++g)
#pragma unroll
          for (int kk = 0; kk < KSG; ++kk) {
            const int ks = g * KSG + kk;   // 16-dim k-step: box ks/4, 32-byte step ks%4
            mma_ss(tbase + g * 64, da0 + (((ks >> 2) * LY::QBOX + (ks & 3) * 32) >> 4),
                   db0 + (((ks >> 2) * kBoxBytes + (ks & 3) * 32) >> 4), idS, kk > 0);
          }
        mma_commit(mS);
      }
      __syncwarp();
    }
    if (page >= 0) {
      if constexpr (VI8) convert_side_from<D, 32>(sb + SP::V_OFF, smem + LY::VH_OFF);
      if constexpr (!VI8) if (edge) zero_rows<D>(sb + SP::V_OFF, key0, j0, j1);
    }
    // The stage of page i - 1 (its last reader, the previous P.V batch, is done)
    // takes page ri, whose id was loaded at the top of the iteration and is
    // checked here as lookup_page checks it: thread 32 arms the stage's barrier
    // now, and after the barrier below one lane in each of the next warps issues
    // one of the page's copies (one thread issuing all of them held its warp for
    // ~700 clocks, and the block with it).
    const int rst = ri % kNS;
    if (refill) {
      if (!ri_in_row) flag_error(p.err, INT8KV_DEVERR_LENGTH);
      const int pg = ri_in_row ? check_page(raw_next, p) : -1;
      stage_page[rst] = pg;
      if (pg < 0)
        ptx::mbar_arrive(&full[rst]);
      else
        ptx::mbar_arrive_expect_tx(&full[rst], PageCopies<D, KI8, VI8>::tx(p.ng));
    }
    ptx::fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    {
      const int c = warp - 1;
      if (i > 0 && ri < n_pg && (tid & 31) == 0 && c >= 0 && c < PageCopies<D, KI8, VI8>::kCopies) {
        const int pg = stage_page[rst];
        if (pg >= 0)
          PageCopies<D, KI8, VI8>::issue(c, smem + LY::ST_OFF + rst * SP::STAGE, &full[rst], pg,
                                         page_row(pg), p, kvh, &tmk, &tmv);
      }
    }
    if (page < 0) continue;   // flagged by the lookup; every thread skips alike
    tc_fence_after();

    // V range per group: 2^e_g bounds every V scale of the group seen so far
    // (the same for every row: block-uniform branches).  O is stable here (the
    // last P.V batch is done; the S batch in flight writes other columns).
#pragma unroll
    for (int g = 0; g < NGV; ++g) {
      if constexpr (VI8) {
        const float mv = s_vmax[g];
        if (mv > 0.f && mv >= cap[g]) {
          const int ne = exponent_of(mv) + 1;
          // the group's columns that lie in this thread's part of O
          const int c_lo = max(g * (D / NGV), half * (D / kParts));
          const int c_hi = min((g + 1) * (D / NGV), (half + 1) * (D / kParts));
          if (vexp[g] != INT_MIN && o_live && c_hi > c_lo)
            tmem_scale(tbase + lane_off + LY::OB + c_lo, c_hi - c_lo, pow2f(vexp[g] - ne));
          vexp[g] = ne;
          cap[g] = pow2f(ne);
          sh[g] = pow2f(kPShift - kPSplit - ne);
        }
      } else {
        sh[g] = pow2f(kPShift - kPSplit);
      }
    }
    // the table of P.V factors, fp16 [group][key]: the V scale times the group's
    // range shift 2^(kPShift - kPSplit - e_g) (below 2^1: exact unless subnormal),
    // 0 for keys outside [j0, j1)
    if constexpr (VI8)
      if (tid < kPage * NG) {
        const int g = tid / kPage, k = tid % kPage;
        const float f = key0 + k >= j0 && key0 + k < j1
                            ? __half2float(reinterpret_cast<const __half*>(sb + SP::VS_OFF)[k * NG + g]) * sh[g]
                            : 0.f;
        reinterpret_cast<__half*>(smem + LY::VSF_OFF)[tid] = __float2half_rn(f);
      }
    const bool okS = ptx::mbar_wait(mS, nS & 1, kMaxPolls);
    ++nS;
    tc_fence_after();

    // ---- this part of the row: scores, softmax, P' per V group (chunks
    // c = kChunks * half ..)
    const bool full_page = !edge && key0 + kPage - 1 <= lim;
    const bool skip = !okS;
    // all of the part's scores first (the reference max must be settled before any P')
    float sv[kChunks][16];
    float mx = -INFINITY;
#pragma unroll
    for (int cc = 0; cc < kChunks; ++cc) {
      const int c = kChunks * half + cc;
      uint32_t v[NGK][16];
#pragma unroll
      for (int g = 0; g < NGK; ++g) tmem_ld16(tbase + lane_off + g * 64 + c * 16, v[g]);
      tmem_wait_ld();
      const float* ksf = reinterpret_cast<const float*>(smem + LY::KSF_OFF);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        float acc = 0.f;
        if constexpr (KI8) {
          float f[NG];
          if constexpr (NG == 4) {
            const float4 x = *reinterpret_cast<const float4*>(ksf + (c * 16 + k) * 4);
            f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
          } else if constexpr (NG == 2) {
            const float2 x = *reinterpret_cast<const float2*>(ksf + (c * 16 + k) * 2);
            f[0] = x.x; f[1] = x.y;
          } else {
            f[0] = ksf[c * 16 + k];
          }
#pragma unroll
          for (int g = 0; g < NG; ++g) acc = fmaf(__uint_as_float(v[g][k]), f[g], acc);
        } else {
          acc = __uint_as_float(v[0][k]) * a.scale_log2;
        }
        sv[cc][k] = acc;
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int key = key0 + c * 16 + k;
        if (!full_page && !(key >= j0 && key < j1 && key <= lim)) sv[cc][k] = -INFINITY;
        mx = fmaxf(mx, sv[cc][k]);
      }
    }
    s_mx[half][R] = mx;
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kParts; ++q) mx = fmaxf(mx, s_mx[q][R]);   // every part takes the same steps
    // move the reference max when exceeded by more than 2^kTau: O and l scale by
    // 2^(m_old - m_new); tensor-memory accesses are warp-wide, so the warp goes
    // together and unaffected rows scale by 1
    const bool need = !skip && mx > m + kTau;
    float al = 1.f;
    if (need) {
      const float mn = fmaxf(m, mx);
      al = m == -INFINITY ? 1.f : ptx::ex2(m - mn);
      l *= al;
      m = mn;
    }
    if (__any_sync(0xffffffffu, need && o_live && al != 1.f))
      tmem_scale(tbase + lane_off + LY::OB + half * (D / kParts), D / kParts, al);
    const float base = (m == -INFINITY ? 0.f : m) - kPSplit;   // p * 2^kPSplit below
#pragma unroll
    for (int cc = 0; cc < kChunks; ++cc)
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        sv[cc][k] = ptx::ex2(sv[cc][k] - base);   // now p * 2^kPSplit
        l += sv[cc][k];                           // this part's share of the row sum
      }
    // P'_g = p * factor(key, g) as fp16 hi | lo for chunk c, over the S columns of
    // chunk c (already read): p split once, each group's factor applied in half
    // precision
    uint32_t ph[kChunks][8], pl[kChunks][8];
#pragma unroll
    for (int cc = 0; cc < kChunks; ++cc)
#pragma unroll
      for (int k2 = 0; k2 < 8; ++k2)
        mma::split_pair(sv[cc][2 * k2], sv[cc][2 * k2 + 1], ph[cc][k2], pl[cc][k2]);
    const uint4* vsf = reinterpret_cast<const uint4*>(smem + LY::VSF_OFF);
#pragma unroll
    for (int g = 0; g < NGV; ++g)
#pragma unroll
      for (int cc = 0; cc < kChunks; ++cc) {
        const int c = kChunks * half + cc;
        uint32_t f[8];   // factor pairs of keys (16c + 2k2, 16c + 2k2 + 1)
        if constexpr (VI8) {
          const uint4 x0 = vsf[(g * kPage + c * 16) / 8], x1 = vsf[(g * kPage + c * 16) / 8 + 1];
          f[0] = x0.x; f[1] = x0.y; f[2] = x0.z; f[3] = x0.w;
          f[4] = x1.x; f[5] = x1.y; f[6] = x1.z; f[7] = x1.w;
        } else {
#pragma unroll
          for (int k2 = 0; k2 < 8; ++k2)
            f[k2] = (uint32_t)(kPShift - kPSplit + 15) * 0x04000400u;   // 2^(kPShift - kPSplit)
        }
        uint32_t v[16];
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2) mma::weight_pair(ph[cc][k2], pl[cc][k2], f[k2], v[k2], v[8 + k2]);
        tmem_st16(tbase + lane_off + g * 64 + c * 16, v);
      }
    tmem_wait_st();
    tc_fence_before();
    if (__syncthreads_or(skip)) {
      if (tid == 0) s_fail = 1;
      break;
    }
    tc_fence_after();

    // ---- O[:, box b] += P'_hi V_b + P'_lo V_b, chunk by chunk (16 keys each)
    if (warp == 0) {
      const uint64_t dv0 = sdesc(ptx::smem_u32(VI8 ? smem + LY::VH_OFF : sb + SP::V_OFF), 1024, 1024);
      if (ptx::elect_one()) {
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
          const int g = b / BPG;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint64_t dv = dv0 + ((b * kBoxBytes + c * 2048) >> 4);
            const uint32_t pa = tbase + g * 64 + c * 16;
            mma_ts(tbase + LY::OB + b * 64, pa, dv, idO, o_live || c > 0);
            mma_ts(tbase + LY::OB + b * 64, pa + 8, dv, idO, true);
          }
        }
        mma_commit(mO);
      }
      __syncwarp();
    }
    ++nO;
    o_live = true;
  }

  // ---- epilogue: the last P.V batch, then this row's O
  bool fail = s_fail != 0;
  if (!fail && nO > 0) fail = !ptx::mbar_wait(mO, (nO - 1) & 1, kMaxPolls);
  tc_fence_after();
  if (fail && tid == 0) flag_error(p.err, INT8KV_DEVERR_TIMEOUT);
  s_mx[half][R] = l;   // the row sum is the parts' sums
  __syncthreads();
  l = 0.f;
#pragma unroll
  for (int q = 0; q < kParts; ++q) l += s_mx[q][R];
  l *= 1.f / (1 << kPSplit);   // the row sum of p
  const bool wr = pos < a.n_new;
  const size_t h = (size_t)pos * a.H + (size_t)kvh * G + R % G;
  const int S = a.n_splits;
#pragma unroll 1
  for (int c = half * (D / kParts); c < (half + 1) * (D / kParts); c += 16) {
    uint32_t v[16];
    tmem_ld16(tbase + lane_off + LY::OB + c, v);
    tmem_wait_ld();
    const int g = c / (D / NGV);
    float u = pow2f(-kPShift);
    if constexpr (VI8) u = vexp[g] == INT_MIN ? 0.f : pow2f(vexp[g] - kPShift);
    if (!o_live) u = 0.f;
    const float f = S == 1 ? (l > 0.f ? u / l : 0.f) : u;
    float* dst = S == 1 ? a.out + h * D + c : a.ws.part_o + (h * S + split) * D + c;
    if (wr) {   // no P.V batch at all: O was never written, the row is 0
      // int8 V: columns 4j + 1 and 4j + 2 hold dims 4j + 2 and 4j + 1
      constexpr int X1 = VI8 ? 2 : 1, X2 = VI8 ? 1 : 2;
#pragma unroll
      for (int k = 0; k < 16; k += 4)
        *reinterpret_cast<float4*>(dst + k) =
            o_live ? make_float4(__uint_as_float(v[k]) * f, __uint_as_float(v[k + X1]) * f,
                                 __uint_as_float(v[k + X2]) * f, __uint_as_float(v[k + 3]) * f)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if (S > 1 && wr && half == 0) a.ws.part_ml[h * S + split] = make_float2(m, l);

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase),
                 "r"((uint32_t)LY::TCOLS)
                 : "memory");
  }
}

template <int D, bool KI8, bool VI8, int NG>
cudaError_t launch_typed(const PrefillArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                         int layer_page0, cudaStream_t stream) {
  using LY = TLayout<D, KI8, VI8, NG>;
  auto kern = prefill_tc_kernel<D, KI8, VI8, NG>;
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

static cudaError_t launch_prefill_tc(const int8kv_pool* pool, int layer, const PrefillArgs& a,
                                     cudaStream_t stream) {
  const int lp0 = layer * pool->n_pages;
  const bool k8 = pool->k_int8, v8 = pool->v_int8;
  if (pool->head_dim == 256) {
    if (k8 && v8) return launch_ng<256, true, true>(a, pool->tmap_k, pool->tmap_v, lp0, stream);
    if (k8) return launch_ng<256, true, false>(a, pool->tmap_k, pool->tmap_v, lp0, stream);
    return launch_ng<256, false, true>(a, pool->tmap_k, pool->tmap_v, lp0, stream);
  }
  if (k8 && v8) return launch_ng<128, true, true>(a, pool->tmap_k, pool->tmap_v, lp0, stream);
  if (k8) return launch_ng<128, true, false>(a, pool->tmap_k, pool->tmap_v, lp0, stream);
  return launch_ng<128, false, true>(a, pool->tmap_k, pool->tmap_v, lp0, stream);
}

bool prefill_supported(const int8kv_pool* pool, int G) {
  return pool->has_tmaps && !pool->v_q4 && !pool->k_q4 && pool->page_size == kPage && pool->group_size >= 64 &&
         (pool->head_dim == 128 || pool->head_dim == 256) && (G == 1 || G == 2 || G == 4 || G == 8);
}

cudaError_t launch_prefill(const int8kv_pool* pool, int layer, const PrefillArgs& a,
                           cudaStream_t stream) {
  const cudaError_t e = launch_prefill_tc(pool, layer, a, stream);
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

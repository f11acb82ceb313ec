// Split-K GQA decode attention over the int8 cache on the 5th-generation
// tensor cores (tcgen05.mma, accumulators in tensor memory), for long key
// ranges.
//
// Method: genie-ai-runtime v1.3.0 "split-K decode attention" (the key range of
// a head is cut into n_splits pieces; each block computes an online-softmax
// partial, a reduce combines them per head) over a cache dequantized on load
// (genie-ai-runtime v0.1.0-alpha.12 "Path I series" I3: every cached row has
// its own scale; Strata pull request #2698 "What it does": one scale per 64
// values).  The arithmetic is that of the mma.sync kernel (decode_mma.cu):
// exact fp16 codes and q, f32 products, K scales applied per (token, group)
// after each group's partial dot, P'= p * s_v fed as an fp16 hi + lo pair with
// a per-group power-of-two range, lazy reference max.
//
// Why a second decode kernel.  The mma.sync kernel holds O (G heads x D f32)
// in registers, so three blocks of four warps fit an SM, and at long contexts
// its ~1,000 instructions per 16-token tile are issued by too few warps to hide
// their latencies.  Here S and O live in tensor memory, one elected lane issues
// all the MMAs, and the CUDA cores are left with turning codes into fp16, the
// softmax and P', in separate warps working on different pages.
//
// Measured on GB300 (128K positions, k8v8): 41.9 us against 32.3 us for the
// mma.sync kernel, so the library does not pick it by itself.  K reaches the
// tensor core from tensor memory (the converters build mma-style fragments and
// store them with tcgen05.st.16x256b), V through an fp16 tile in shared memory.
// Per page the converters need ~2,000 clocks and the softmax ~1,500 (both chains
// of dependent latencies, one page at a time per role), against ~1,560 clocks of
// HBM time per page at the measured peak.
//
// Roles (448 threads, one block per SM at head_dim 256):
//   warps 0-3  softmax.  Warp w owns tokens 16w .. 16w + 15 of every page.
//   warps 4-11 converters.  int8 K rows of a staged page become the fp16 A
//              operand of q.K^T in tensor memory (Ka), V rows an fp16 tile Vc in
//              shared memory (128-byte-swizzled boxes [D/64][64 tokens][128 B]),
//              the scales fp32 tables; the page's largest V scale per group is
//              noted.
//              The staged page is released as soon as its codes are in
//              registers, so its stage refills while they are converted.
//   warp 12    producer of S: an elected lane issues the TMA copies of the
//              page ring (four stages) and q.K^T.
//   warp 13    producer of O: an elected lane issues P.V.
// Per page i (buffers b = i % 2 of Ka, Vc, the tables, P' and S):
//   converters K rows -> Ka[b] in tensor memory and the scale tables ("K ready"),
//              then V rows -> the fp16 tile Vc[b] in shared memory ("V ready").
//   producer   S_g[b] = sum over the group's 64-dim boxes of Ka q^T: M = 64
//              tokens, N = 16 (the G <= 8 heads, zero-padded), K = 16, A read
//              from tensor memory.
//   softmax    s = sum_g table_k * S_g (tensor memory, mma-fragment layout),
//              masks, per-head page maxima shared by the four warps, the lazy
//              rescale (O in tensor memory, read and rewritten per warp quarter),
//              p = 2^(s - m), and P'_g = p * s_v * 2^(6 - e_g) as fp16 hi | lo
//              into shared memory (no swizzle, MN-major: a token's 8 heads are
//              one 16-byte row).
//   producer   O_x += Vc_x^T P'_g(x) for every 64-dim box x: M = 64 dims,
//              N = 16 (8 heads' hi, 8 heads' lo), K = 16 tokens.
// Hand-offs are mbarriers: TMA completion, "converted", "S ready" and "O
// done" (tcgen05.commit), "P' written".  Every wait is bounded and sets a
// device error bit on expiry.
//
// Codes are turned into fp16 two at a time -- bytes 0 and 2 of a word, then 1
// and 3.  In Vc, positions 1 and 2 of every four dims swap, and the rows of O
// (dims) are read back through that order.  In Ka, K index 16e + 4u + x of a
// 64-dim box holds dim 16u + 4e + (0, 2, 1, 3)[x] (see KFrag); q is laid out in
// the same K order, so q.k is unchanged.

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

using mma::exponent_of;
using mma::kBoxBytes;
using mma::kMaxPolls;
using mma::kPage;
using mma::lop_i8pair;
using mma::pow2f;
using mma::sub1152;

constexpr int kSoftWarps = 4;
constexpr int kConvWarps = 8;
constexpr int kConv0 = kSoftWarps * 32;                  // first converter thread
constexpr int kProdK = kSoftWarps + kConvWarps;          // warp: copies and q.K
constexpr int kProdV = kProdK + 1;                       // warp: P.V
constexpr int kThreads = (kProdV + 1) * 32;
constexpr float kTau = 8.f;         // lazy rescale: the reference max moves when exceeded by > 2^8
constexpr int kPShift = 6;          // P' < 2^8 * 2^6 in fp16
constexpr int kPagesCached = 256;   // page ids of a block's range kept in shared memory

template <int D, int NG>
struct DLayout {
  using SP = mma::StagedPage<D, true, true>;
  static constexpr int NBOX = D / 64;                 // 64-dim boxes
  static constexpr int BPG = NBOX / NG;               // boxes per scale group
  static constexpr int CBYTES = kPage * D * 2;        // one converted V page
  static constexpr int PBG = 2048;                    // P' of one V group: [hi | lo][64][16 B]
  static constexpr int QBOX = 16 * 128;               // one 64-dim box of q: 16 rows x 128 B
  static constexpr int OTHER = 2 * CBYTES + 2 * NG * PBG + NBOX * QBOX + 4 * kPage * NG * 4;
  static constexpr int NS_FIT = (224 * 1024 - OTHER) / SP::STAGE;
  static constexpr int NS = NS_FIT > 4 ? 4 : NS_FIT;   // stages of the raw page ring
  static constexpr int RAW_OFF = 0;
  static constexpr int VC_OFF = RAW_OFF + NS * SP::STAGE;   // two Vc
  static constexpr int PB_OFF = VC_OFF + 2 * CBYTES;
  static constexpr int QB_OFF = PB_OFF + 2 * NG * PBG;
  static constexpr int KSF_OFF = QB_OFF + NBOX * QBOX;       // fp32 [2][64][NG]
  static constexpr int VSF_OFF = KSF_OFF + 2 * kPage * NG * 4;
  static constexpr int BAR_OFF = VSF_OFF + 2 * kPage * NG * 4;
  static constexpr int SMEM = 1024 + BAR_OFF + 256;
  // tensor memory: Ka[2] (the K tile of a page as the A operand: 64 token rows,
  // D/2 columns of dim pairs), S[2] (NG groups x 16 columns), O (NBOX boxes x 16)
  static constexpr int KA_COLS = D / 2;
  static constexpr int S_COL = 2 * KA_COLS;
  static constexpr int S_COLS = NG * 16;
  static constexpr int O_COL = S_COL + 2 * S_COLS;
  static constexpr int NEED = O_COL + NBOX * 16;
  static constexpr int TCOLS = NEED <= 64 ? 64 : NEED <= 128 ? 128 : NEED <= 256 ? 256 : 512;
  static_assert(NS >= 2, "at least two raw stages");
  static_assert(NEED <= 512, "tensor memory holds Ka, S and O");
  static_assert(QB_OFF % 1024 == 0 && VC_OFF % 1024 == 0, "swizzled tiles start on 1 KB");
  static_assert(SMEM <= 232448, "one block fits the shared memory of an SM");
};

__device__ __forceinline__ int swz(int row, int c) { return row * 128 + ((c ^ (row & 7)) << 4); }

// Dim held by tile position p (positions 1 and 2 of every four swap).
__device__ __forceinline__ int dim_of(int p) {
  return (p & ~3) | ((p & 1) << 1) | ((p >> 1) & 1);
}

// 16 int8 codes -> 16 exact fp16 values, positions (0, 2, 1, 3) per four codes.
__device__ __forceinline__ void codes_to_f16_pairs(const uint4 w, uint4& lo, uint4& hi) {
  lo = make_uint4(sub1152(lop_i8pair(w.x)), sub1152(lop_i8pair(w.x >> 8)),
                  sub1152(lop_i8pair(w.y)), sub1152(lop_i8pair(w.y >> 8)));
  hi = make_uint4(sub1152(lop_i8pair(w.z)), sub1152(lop_i8pair(w.z >> 8)),
                  sub1152(lop_i8pair(w.w)), sub1152(lop_i8pair(w.w >> 8)));
}

// int8 rows of one side of a staged page -> fp16 boxes [D/64][64][128 B], by the
// converter threads: first every thread's code chunks into registers (all loads
// in flight together), then the conversions and stores.  Eight consecutive
// threads take one code chunk of eight consecutive rows, so loads and stores
// hit eight different swizzled positions.
template <int D>
struct SideChunks {
  static constexpr int CPR = D / 16;                              // 16-byte code chunks per row
  static constexpr int PER = kPage * CPR / (kConvWarps * 32);     // chunks per thread
  uint4 w[PER];

  __device__ __forceinline__ static void where(int ct, int k, int& row, int& cc) {
    const int c = ct + k * kConvWarps * 32, g8 = c >> 3;
    row = (g8 / CPR) * 8 + (c & 7);
    cc = g8 % CPR;
  }
  __device__ __forceinline__ void load(const unsigned char* src, int ct) {
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      int row, cc;
      where(ct, k, row, cc);
      w[k] = *reinterpret_cast<const uint4*>(src + (cc >> 3) * kBoxBytes + swz(row, cc & 7));
    }
  }
  __device__ __forceinline__ void store(unsigned char* dst, int ct) const {
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      int row, cc;
      where(ct, k, row, cc);
      uint4 lo, hi;
      codes_to_f16_pairs(w[k], lo, hi);
      unsigned char* box = dst + (cc >> 2) * kBoxBytes;
      const int c16 = (cc & 3) * 2;
      *reinterpret_cast<uint4*>(box + swz(row, c16)) = lo;
      *reinterpret_cast<uint4*>(box + swz(row, c16 + 1)) = hi;
    }
  }
};

// K rows of a staged page -> the Ka tile in tensor memory: the A operand of
// q.K^T, 64 token rows in the M = 64 layout (row m in lane 32 (m / 16) + m % 16),
// column c holding K indices 2c and 2c + 1.  Converter warp (quarter qd, half h)
// takes tokens 16 qd .. 16 qd + 15 and the 64-dim boxes of its half; thread t
// holds tokens 16 qd + t/4 and + 8 and, per box, the 16-byte chunk u = t % 4
// (dims 16u .. 16u + 15) of both rows.  Word e of the chunk becomes columns 2u and
// 2u + 1 of the box's 8-column block e (tcgen05.st.16x256b, the mma.sync
// accumulator layout): K index 16e + 4u + x holds dim 16u + 4e + (0, 2, 1, 3)[x].
template <int D>
struct KFrag {
  static constexpr int BOXES = D / 64 / 2;   // boxes per half
  uint4 ra[BOXES], rb[BOXES];

  __device__ __forceinline__ void load(const unsigned char* src, int qd, int h, int lane) {
    const int rowA = 16 * qd + (lane >> 2), rowB = rowA + 8, u = lane & 3;
#pragma unroll
    for (int j = 0; j < BOXES; ++j) {
      const int cc = 4 * (h * BOXES + j) + u;   // 16-byte chunk of a 128-byte row box
      ra[j] = *reinterpret_cast<const uint4*>(src + (cc >> 3) * kBoxBytes + swz(rowA, cc & 7));
      rb[j] = *reinterpret_cast<const uint4*>(src + (cc >> 3) * kBoxBytes + swz(rowB, cc & 7));
    }
  }
  // ta: tensor-memory address of this warp's lanes at the Ka buffer's column 0
  __device__ __forceinline__ void store(uint32_t ta, int h) const {
#pragma unroll
    for (int j = 0; j < BOXES; ++j) {
      const uint32_t wa[4] = {ra[j].x, ra[j].y, ra[j].z, ra[j].w};
      const uint32_t wb[4] = {rb[j].x, rb[j].y, rb[j].z, rb[j].w};
      uint32_t v[16];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[4 * e + 0] = sub1152(lop_i8pair(wa[e]));
        v[4 * e + 1] = sub1152(lop_i8pair(wa[e] >> 8));
        v[4 * e + 2] = sub1152(lop_i8pair(wb[e]));
        v[4 * e + 3] = sub1152(lop_i8pair(wb[e] >> 8));
      }
      tc::st_frag_x4(ta + (h * BOXES + j) * 32, v);
    }
  }
};

template <int NG>
__device__ __forceinline__ void load_f32(const float* p, float (&x)[NG]) {
  if constexpr (NG == 4) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else if constexpr (NG == 2) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    x[0] = v.x; x[1] = v.y;
  } else {
    x[0] = p[0];
  }
}

__device__ __forceinline__ void sts32(unsigned char* p, uint32_t v) {
  *reinterpret_cast<uint32_t*>(p) = v;
}


template <int D, int NG>
__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmv, int layer_page0) {
  using LY = DLayout<D, NG>;
  using SP = typename LY::SP;
  constexpr int NBOX = LY::NBOX, NS = LY::NS, BPG = LY::BPG;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + LY::BAR_OFF);   // [NS] page landed
  uint64_t* convk = full + NS;    // [2] Ka tile and scale tables written
  uint64_t* convv = convk + 2;    // [2] Vc tile written
  uint64_t* sfull = convv + 2;    // [2] S ready
  uint64_t* pfull = sfull + 2;    // [2] P' written
  uint64_t* ofull = pfull + 2;    // [2] P.V done
  uint64_t* empty = ofull + 2;    // [NS] staged page read into registers
  int* stage_page = reinterpret_cast<int*>(empty + NS);  // [NS]
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(stage_page + NS);
  __shared__ int s_pages[kPagesCached];
  __shared__ int s_valid[2];                  // [buffer] the page exists
  __shared__ float s_vmax[2][2][NG];          // [buffer][converter warp][group] largest V scale
  __shared__ float s_px[2][kSoftWarps][8];    // [page parity][warp][head] score maxima
  __shared__ float s_sum[kSoftWarps][8];
  __shared__ float s_mref[8];

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PoolView& p = a.pool;
  const int G = a.G;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], kConvWarps);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&convk[s], kConvWarps);
      ptx::mbar_init(&convv[s], kConvWarps);
      ptx::mbar_init(&sfull[s], 1);
      ptx::mbar_init(&pfull[s], kSoftWarps);
      ptx::mbar_init(&ofull[s], 1);
    }
    ptx::fence_mbar_init();
  }
  if (warp == 0) tc::alloc(taddr_s, LY::TCOLS);
  // Launched as a programmatic dependent: no global memory is read before the
  // preceding kernel of the stream has completed.
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();

  const int L_raw = ptx::ldg32(a.seq_lens + b);
  const int32_t* ptrow = a.page_table + (size_t)b * a.max_pages;
  const bool row_cached = a.max_pages <= kPagesCached;
  if (row_cached)
    for (int i = tid; i < a.max_pages; i += kThreads) s_pages[i] = ptx::ldg32(ptrow + i);
  // q of the kv head's G heads -> 16 K-major rows (rows >= G zero), in the K order
  // of the Ka tile (see the converters): within a 64-dim box, K index 16e + 4u + x
  // holds dim 16u + 4e + (0, 2, 1, 3)[x]
  for (int c = tid; c < 16 * (D / 8); c += kThreads) {
    const int row = c / (D / 8), ch = c - row * (D / 8);   // 8 K indices 8ch .. 8ch + 7
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (row < G) {
      const uint16_t* qh = a.q + ((size_t)b * a.H + (size_t)kvh * G + row) * D + (ch >> 3) * 64;
#pragma unroll
      for (int k2 = 0; k2 < 4; ++k2) {
        uint16_t hv[2];
#pragma unroll
        for (int z = 0; z < 2; ++z) {
          const int kk = (ch & 7) * 8 + 2 * k2 + z;   // K index within the box
          const int e = kk >> 4, u = (kk >> 2) & 3, x = kk & 3;
          hv[z] = __ldg(qh + 16 * u + 4 * e + ((x == 1) ? 2 : (x == 2) ? 1 : x));
        }
        w[k2] = (uint32_t)hv[0] | ((uint32_t)hv[1] << 16);
      }
    }
    *reinterpret_cast<uint4*>(smem + LY::QB_OFF + (ch >> 3) * LY::QBOX + swz(row, ch & 7)) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
  const int L = clamp_length(L_raw, a.max_pages, p);
  const int lo_pos = a.window > 0 ? max(0, L - a.window) : 0;
  int j0, j1;
  split_range(lo_pos, L, split, a.n_splits, kPage, &j0, &j1);
  const int p_first = j0 / kPage;
  const int n_pg = j1 > j0 ? (j1 - 1) / kPage - p_first + 1 : 0;
  ptx::fence_proxy_async();   // the q tile (generic stores) is read by the tensor core
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *taddr_s;
  auto page_of = [&](int i) {   // page i of the block's range
    return row_cached ? check_page(s_pages[p_first + i], p)
                      : lookup_page(ptrow, p_first + i, a.max_pages, p);
  };

  if (warp == kProdK || warp == kProdV) {
    // ----------------------------------------------------------- producers
    // Each warp runs its loop whole (waits and descriptors stay warp-uniform);
    // one elected lane issues each copy and MMA batch.  Warp kProdK: the page
    // ring and S = Ka q^T; warp kProdV: O += Vc^T P'.  Their MMAs use disjoint
    // operands, and each commit tracks its own warp's MMAs.
    constexpr uint32_t idS = tc::idesc_f16(64, 16, 0, 0);   // A = Ka (tensor memory), B = q
    constexpr uint32_t idO = tc::idesc_f16(64, 16, 1, 1);   // A = Vc^T (MN-major), B = P'
    bool ok = true;
    if (warp == kProdK) {
      if (lane == 0) {
        ptx::prefetch_tensormap(&tmk);
        ptx::prefetch_tensormap(&tmv);
      }
      auto issue = [&](int i) {
        const int st = i % NS, page = page_of(i);
        mma::issue_page<D, true, true, true>(smem + LY::RAW_OFF + st * SP::STAGE, &full[st],
                                             &stage_page[st], page,
                                             ((layer_page0 + page) * p.Hkv + kvh) * kPage, p,
                                             kvh, &tmk, &tmv);
      };
      if (ptx::elect_one())
        for (int i = 0; i < NS && i < n_pg; ++i) issue(i);
      __syncwarp();
      const uint64_t dq = tc::sdesc(ptx::smem_u32(smem + LY::QB_OFF), 16, 1024);
      for (int i = 0; i < n_pg; ++i) {
        const int bb = i & 1;
        if (i + NS < n_pg) {   // page i's codes are in registers: its stage takes page i + NS
          ok = ok && ptx::mbar_wait(&empty[i % NS], (i / NS) & 1, kMaxPolls);
          if (ptx::elect_one()) issue(i + NS);
          __syncwarp();
        }
        ok = ok && ptx::mbar_wait(&convk[bb], (i >> 1) & 1, kMaxPolls);
        tc::fence_after();
        if (ptx::elect_one()) {
#pragma unroll
          for (int x = 0; x < NBOX; ++x)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc::mma_ts(tbase + LY::S_COL + bb * LY::S_COLS + (x / BPG) * 16,
                         tbase + bb * LY::KA_COLS + x * 32 + ks * 8,
                         dq + ((x * LY::QBOX + 32 * ks) >> 4), idS, (x % BPG) != 0 || ks != 0);
          tc::mma_commit(&sfull[bb]);
        }
        __syncwarp();
      }
    } else {
      const uint64_t dv = tc::sdesc(ptx::smem_u32(smem + LY::VC_OFF), 1024, 1024);
      const uint64_t dp = tc::sdesc(ptx::smem_u32(smem + LY::PB_OFF), 128, 1024, tc::kSwizzleNone);
      for (int i = 0; i < n_pg; ++i) {
        const int bb = i & 1;
        ok = ok && ptx::mbar_wait(&convv[bb], (i >> 1) & 1, kMaxPolls);
        ok = ok && ptx::mbar_wait(&pfull[bb], (i >> 1) & 1, kMaxPolls);
        tc::fence_after();
        if (ptx::elect_one()) {
#pragma unroll
          for (int x = 0; x < NBOX; ++x)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc::mma_ss(tbase + LY::O_COL + x * 16,
                         dv + ((bb * LY::CBYTES + x * kBoxBytes + 2048 * ks) >> 4),
                         dp + (((bb * NG + x / BPG) * LY::PBG + 256 * ks) >> 4), idO,
                         i != 0 || ks != 0);
          tc::mma_commit(&ofull[bb]);
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) flag_error(p.err, INT8KV_DEVERR_TIMEOUT);
  } else if (warp >= kSoftWarps) {
    // ----------------------------------------------------------- converters
    const int ct = tid - kConv0;
    bool ok = true;
    for (int i = 0; i < n_pg; ++i) {
      const int st = i % NS, bb = i & 1;
      ok = ok && ptx::mbar_wait(&full[st], (i / NS) & 1, kMaxPolls);
      const unsigned char* sb = smem + LY::RAW_OFF + st * SP::STAGE;
      KFrag<D> kf;
      SideChunks<D> vw;
      kf.load(sb + SP::K_OFF, warp & 3, (warp - kSoftWarps) >> 2, lane);
      vw.load(sb + SP::V_OFF, ct);
      const bool page_ok = stage_page[st] >= 0;
      float kx[NG], vx[NG];   // token ct's scales (warps 4 and 5)
      if (ct < kPage) {
        const uint16_t* ks = reinterpret_cast<const uint16_t*>(sb + SP::KS_OFF) + ct * NG;
        const uint16_t* vs = reinterpret_cast<const uint16_t*>(sb + SP::VS_OFF) + ct * NG;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          kx[g] = h2f(ks[g]) * a.scale_log2;
          vx[g] = h2f(vs[g]);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[st]);   // every read of the stage is done
      // ---- K side (all that q.K^T and the softmax of page i need): the tables and
      // s_valid[b] were read last by the softmax of page i - 2, Ka[b] by its q.K
      if (i >= 2) {
        ok = ok && ptx::mbar_wait(&pfull[bb], ((i - 2) >> 1) & 1, kMaxPolls);
        ok = ok && ptx::mbar_wait(&sfull[bb], ((i - 2) >> 1) & 1, kMaxPolls);
      }
      tc::fence_after();
      if (ct < kPage) {
        const int pos = (p_first + i) * kPage + ct;
        const bool valid = page_ok && pos >= j0 && pos < j1;
        float* ksf = reinterpret_cast<float*>(smem + LY::KSF_OFF) + (bb * kPage + ct) * NG;
        float* vsf = reinterpret_cast<float*>(smem + LY::VSF_OFF) + (bb * kPage + ct) * NG;
        if constexpr (NG == 4) {
          *reinterpret_cast<float4*>(ksf) = make_float4(kx[0], kx[1], kx[2], kx[3]);
          *reinterpret_cast<float4*>(vsf) = make_float4(vx[0], vx[1], vx[2], vx[3]);
        } else {
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            ksf[g] = kx[g];
            vsf[g] = vx[g];
          }
        }
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const float mx = warp_max(valid ? vx[g] : 0.f);
          if (lane == 0) s_vmax[bb][ct >> 5][g] = mx;
        }
      }
      if (ct == 0) s_valid[bb] = page_ok ? 1 : 0;
      kf.store(tbase + ((uint32_t)((warp & 3) * 32) << 16) + bb * LY::KA_COLS,
               (warp - kSoftWarps) >> 2);
      tc::wait_st();
      tc::fence_before();   // the Ka stores precede the MMA that reads them
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&convk[bb]);
      // ---- V side (only the P.V of page i needs it): Vc[b] was read last by the
      // P.V of page i - 2
      if (i >= 2) ok = ok && ptx::mbar_wait(&ofull[bb], ((i - 2) >> 1) & 1, kMaxPolls);
      vw.store(smem + LY::VC_OFF + bb * LY::CBYTES, ct);
      ptx::fence_proxy_async();   // the V tile (generic stores) is read by the tensor core
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&convv[bb]);
    }
    if (!ok) flag_error(p.err, INT8KV_DEVERR_TIMEOUT);
  } else {
    // -------------------------------------------------------------- softmax
    const int r = lane >> 2, c = lane & 3;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;   // this warp's tensor-memory lanes
    const float* ksf_all = reinterpret_cast<const float*>(smem + LY::KSF_OFF);
    const float* vsf_all = reinterpret_cast<const float*>(smem + LY::VSF_OFF);
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // heads 2c, 2c + 1
    int vexp[NG];             // per V group: 2^vexp > every V scale seen (block-wide)
    float cap[NG], sh[NG];    // 2^vexp and 2^(kPShift - vexp), 0 before the first scale
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      vexp[g] = INT_MIN;
      cap[g] = 0.f;
      sh[g] = 0.f;
    }
    bool ok = true;
    for (int i = 0; i < n_pg; ++i) {
      const int bb = i & 1;
      ok = ok && ptx::mbar_wait(&convk[bb], (i >> 1) & 1, kMaxPolls);
      ok = ok && ptx::mbar_wait(&sfull[bb], (i >> 1) & 1, kMaxPolls);
      tc::fence_after();
      float sg[NG][4];
#pragma unroll
      for (int g = 0; g < NG; ++g)
        tc::ld_frag(tbase + lane_off + LY::S_COL + bb * LY::S_COLS + g * 16, sg[g]);
      tc::wait_ld();
      const int t0 = warp * 16 + r, t1 = t0 + 8;             // tokens of the page
      const int pos0 = (p_first + i) * kPage + t0, pos1 = pos0 + 8;
      const bool page_ok = s_valid[bb] != 0;
      const bool v0 = page_ok && pos0 >= j0 && pos0 < j1;
      const bool v1 = page_ok && pos1 >= j0 && pos1 < j1;
      float ka[NG], kb[NG];
      load_f32<NG>(ksf_all + (bb * kPage + t0) * NG, ka);
      load_f32<NG>(ksf_all + (bb * kPage + t1) * NG, kb);
      float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        s[0] = fmaf(sg[g][0], ka[g], s[0]);
        s[1] = fmaf(sg[g][1], ka[g], s[1]);
        s[2] = fmaf(sg[g][2], kb[g], s[2]);
        s[3] = fmaf(sg[g][3], kb[g], s[3]);
      }
      if (!v0) s[0] = s[1] = -INFINITY;
      if (!v1) s[2] = s[3] = -INFINITY;
      // ---- per-head page maxima of the four warps; the same decision in all
      float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      if (r == 0) {
        s_px[bb][warp][2 * c] = mx0;
        s_px[bb][warp][2 * c + 1] = mx1;
      }
      ptx::named_barrier_sync(1, kSoftWarps * 32);
      float M0 = s_px[bb][0][2 * c], M1 = s_px[bb][0][2 * c + 1];
#pragma unroll
      for (int w = 1; w < kSoftWarps; ++w) {
        M0 = fmaxf(M0, s_px[bb][w][2 * c]);
        M1 = fmaxf(M1, s_px[bb][w][2 * c + 1]);
      }
      float vm[NG];
      bool need_v = false;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        vm[g] = fmaxf(s_vmax[bb][0][g], s_vmax[bb][1][g]);
        need_v |= vm[g] > 0.f && vm[g] >= cap[g];
      }
      const bool need_m = M0 > m0 + kTau || M1 > m1 + kTau;
      if (__any_sync(0xffffffffu, need_m) || need_v) {
        // move the reference max (O and l scale by 2^(m_old - m_new)) and raise
        // the V ranges (O of the group's boxes scales by 2^(e_old - e_new))
        float al0 = 1.f, al1 = 1.f;
        if (M0 > m0 + kTau) {
          const float mn = fmaxf(m0, M0);
          al0 = mn == -INFINITY ? 1.f : ptx::ex2(m0 - mn);
          m0 = mn;
        }
        if (M1 > m1 + kTau) {
          const float mn = fmaxf(m1, M1);
          al1 = mn == -INFINITY ? 1.f : ptx::ex2(m1 - mn);
          m1 = mn;
        }
        l0 *= al0;
        l1 *= al1;
        float be[NG];
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          be[g] = 1.f;
          if (vm[g] > 0.f && vm[g] >= cap[g]) {
            const int ne = exponent_of(vm[g]) + 1;
            if (vexp[g] != INT_MIN) be[g] = pow2f(vexp[g] - ne);
            vexp[g] = ne;
            cap[g] = pow2f(ne);
            sh[g] = pow2f(kPShift - ne);
          }
        }
        if (i >= 1) {   // O holds pages 0 .. i-1 once the last of their P.V is done
          ok = ok && ptx::mbar_wait(&ofull[(i - 1) & 1], ((i - 1) >> 1) & 1, kMaxPolls);
          tc::fence_after();
          float alh[8];   // head h's factor sits in lane h / 2 (r = 0, c = h / 2)
#pragma unroll
          for (int h = 0; h < 8; ++h) alh[h] = __shfl_sync(0xffffffffu, (h & 1) ? al1 : al0, h >> 1);
#pragma unroll
          for (int x = 0; x < NBOX; ++x) {
            uint32_t v[16];
            tc::ld16(tbase + lane_off + LY::O_COL + x * 16, v);
            tc::wait_ld();
            const float bx = be[x / BPG];
#pragma unroll
            for (int n = 0; n < 16; ++n) v[n] = __float_as_uint(__uint_as_float(v[n]) * (alh[n & 7] * bx));
            tc::st16(tbase + lane_off + LY::O_COL + x * 16, v);
          }
          tc::wait_st();
        }
      }
      const float base0 = m0 == -INFINITY ? 0.f : m0, base1 = m1 == -INFINITY ? 0.f : m1;
      float pr[4];
      pr[0] = ptx::ex2(s[0] - base0);
      pr[1] = ptx::ex2(s[1] - base1);
      pr[2] = ptx::ex2(s[2] - base0);
      pr[3] = ptx::ex2(s[3] - base1);
      l0 += pr[0] + pr[2];
      l1 += pr[1] + pr[3];
      // ---- P'_g as fp16 hi | lo rows of P'[b] (read last by the P.V of page i - 2)
      if (i >= 2) ok = ok && ptx::mbar_wait(&ofull[bb], ((i - 2) >> 1) & 1, kMaxPolls);
      float va[NG], vb[NG];
      load_f32<NG>(vsf_all + (bb * kPage + t0) * NG, va);
      load_f32<NG>(vsf_all + (bb * kPage + t1) * NG, vb);
      unsigned char* pbb = smem + LY::PB_OFF + bb * NG * LY::PBG + 4 * c;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const float wa = v0 ? va[g] * sh[g] : 0.f, wb = v1 ? vb[g] * sh[g] : 0.f;
        const float p0 = pr[0] * wa, p1 = pr[1] * wa, p2 = pr[2] * wb, p3 = pr[3] * wb;
        const uint32_t h01 = ptx::pack_f16x2(p0, p1), h23 = ptx::pack_f16x2(p2, p3);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
        unsigned char* pg = pbb + g * LY::PBG;
        sts32(pg + t0 * 16, h01);
        sts32(pg + t1 * 16, h23);
        sts32(pg + 1024 + t0 * 16, ptx::pack_f16x2(p0 - f01.x, p1 - f01.y));
        sts32(pg + 1024 + t1 * 16, ptx::pack_f16x2(p2 - f23.x, p3 - f23.y));
      }
      ptx::fence_proxy_async();   // P' (generic stores) is read by the tensor core
      tc::fence_before();         // and the S columns read above may be overwritten
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&pfull[bb]);
    }

    // ---- epilogue: the last P.V, then this block's partial (or the output)
    if (n_pg > 0) ok = ok && ptx::mbar_wait(&ofull[(n_pg - 1) & 1], ((n_pg - 1) >> 1) & 1, kMaxPolls);
    tc::fence_after();
    if (!ok) flag_error(p.err, INT8KV_DEVERR_TIMEOUT);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    if (r == 0) {
      s_sum[warp][2 * c] = l0;
      s_sum[warp][2 * c + 1] = l1;
      if (warp == 0) {
        s_mref[2 * c] = m0;
        s_mref[2 * c + 1] = m1;
      }
    }
    ptx::named_barrier_sync(1, kSoftWarps * 32);
    float Lh[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) Lh[h] = s_sum[0][h] + s_sum[1][h] + s_sum[2][h] + s_sum[3][h];
    const int S = a.n_splits;
    const size_t hb = (size_t)b * a.H + (size_t)kvh * G;
#pragma unroll
    for (int x = 0; x < NBOX; ++x) {
      uint32_t v[16];
      if (n_pg > 0) {
        tc::ld16(tbase + lane_off + LY::O_COL + x * 16, v);
        tc::wait_ld();
      }
      if (lane < 16) {
        const int d = x * 64 + dim_of(warp * 16 + lane);
        const int g = x / BPG;
        const float u = (n_pg == 0 || vexp[g] == INT_MIN) ? 0.f : pow2f(vexp[g] - kPShift);
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          if (h >= G) break;
          const float o = u == 0.f ? 0.f : (__uint_as_float(v[h]) + __uint_as_float(v[8 + h])) * u;
          if (S == 1)
            a.out[(hb + h) * D + d] = Lh[h] > 0.f ? o / Lh[h] : 0.f;
          else
            a.ws.part_o[((hb + h) * S + split) * D + d] = o;
        }
      }
    }
    if (S > 1 && warp == 0 && lane < G)
      a.ws.part_ml[(hb + lane) * S + split] =
          make_float2(s_mref[lane], s_sum[0][lane] + s_sum[1][lane] + s_sum[2][lane] + s_sum[3][lane]);
  }

  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::dealloc(tbase, LY::TCOLS);
  }
}

template <int D, int NG>
cudaError_t launch_typed(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                         int layer_page0, cudaStream_t stream) {
  using LY = DLayout<D, NG>;
  auto kern = decode_tc_kernel<D, NG>;
  static bool configured[64] = {};   // per device: the attribute belongs to the device's function
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::SMEM);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_splits, a.pool.Hkv, a.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = LY::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, tmk, tmv, layer_page0);
}

template <int D, int NG>
int resident_typed() {
  using LY = DLayout<D, NG>;
  auto kern = decode_tc_kernel<D, NG>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::SMEM) !=
      cudaSuccess)
    return 0;
  int per_sm = 0, dev = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, LY::SMEM) !=
          cudaSuccess ||
      cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return per_sm * sms;
}

}  // namespace

bool decode_tc_supported(const PoolView& p, bool k8, bool v8, int G) {
  return k8 && v8 && G <= 8 && p.ps == kPage && (p.D == 128 || p.D == 256) && p.gs >= 64 &&
         p.gs % 64 == 0;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                             int layer_page0, cudaStream_t stream) {
  if (a.pool.D == 256) {
    switch (a.pool.ng) {
      case 1: return launch_typed<256, 1>(a, tmk, tmv, layer_page0, stream);
      case 2: return launch_typed<256, 2>(a, tmk, tmv, layer_page0, stream);
      case 4: return launch_typed<256, 4>(a, tmk, tmv, layer_page0, stream);
      default: return cudaErrorNotSupported;
    }
  }
  if (a.pool.D == 128) {
    switch (a.pool.ng) {
      case 1: return launch_typed<128, 1>(a, tmk, tmv, layer_page0, stream);
      case 2: return launch_typed<128, 2>(a, tmk, tmv, layer_page0, stream);
      default: return cudaErrorNotSupported;
    }
  }
  return cudaErrorNotSupported;
}

// Blocks of the tensor-memory decode kernel the current device keeps resident
// at once for this shape; 0 if unknown.
int decode_tc_resident_blocks(int D, int ng) {
  if (D == 256) {
    if (ng == 1) return resident_typed<256, 1>();
    if (ng == 2) return resident_typed<256, 2>();
    if (ng == 4) return resident_typed<256, 4>();
  }
  if (D == 128) {
    if (ng == 1) return resident_typed<128, 1>();
    if (ng == 2) return resident_typed<128, 2>();
  }
  return 0;
}

}  // namespace int8kv

// Split-K GQA decode attention over the int8 cache on the tensor cores
// (mma.sync m16n8k16, f16 operands, f32 accumulation), pages staged by TMA.
//
// Method: genie-ai-runtime v1.3.0 "split-K decode attention" (the key range of
// a head is cut into n_splits pieces; each block computes an online-softmax
// partial, a reduce combines them per head) over a cache dequantized on load
// (genie-ai-runtime v0.1.0-alpha.12 "Path I series" I3: every cached row has
// its own scale; Strata pull request #2698 "What it does": one scale per 64
// values, k8v8 / one-store variants).
//
// Why tensor cores in a bandwidth-bound kernel: one block serves the G <= 8
// query heads of its kv head, so every cached byte feeds 2*G multiply-adds
// (G for q.k, G for p.v).  At G = 8 and head_dim 256 that is ~7.8 FMA per byte,
// more than the CUDA cores can retire at HBM speed (152 SMs x 128 FMA/clk is
// ~5 TB/s worth at 1.9 GHz before any conversion work).  Both products are
// genuine dense contractions over the G heads (q.K^T: [16 tok x D] x [D x 8
// heads]; P.V: [D x 16 tok] x [16 tok x 8 heads]), so they go to mma.sync.
//
// Exactness.  int8 codes (|c| <= 127) and fp16 q are exact in fp16 and their
// products are exact in the f32 accumulator; the K scales (and softmax scale)
// are applied per (token, 64-value group) in f32 after each 64-wide partial
// dot.  On the P.V side the weight of token j for output dims of V group g is
// P'_jg = p_j * s_v(j, g) (exp-weights times the V scale); it is fed to the
// tensor core as an fp16 hi + lo pair (two MMAs), which keeps ~21 bits.  To keep
// P' away from fp16's subnormal range whatever the magnitude of V, each warp
// tracks a power of two 2^e_g > every V scale of group g it has seen and
// feeds p_j * s_v(j, g) * 2^(6 - e_g) < 2^8 * 2^6 = 2^14 (the lazy max bounds p by
// 2^8); when e_g grows, the group's accumulators
// are rescaled by the exact power-of-two ratio (the same move the online
// softmax makes with its running max).
//
// Data movement.  A block owns a contiguous run of pages of one (sequence, kv
// head).  One producer lane streams each page (K codes, V codes: 64 rows x
// 128 B boxes with the 128-byte swizzle; scales: one bulk copy each) into a
// ring of stages, completion counted on mbarriers; four consumer warps take
// one 16-token tile of every page.  The swizzle plus the row/slot permutations
// below make every shared-memory fragment load bank-conflict free.
//
// Layout of the work inside a 16-token tile (r = lane/4, t = lane%4):
//  q.K^T : A = K rows.  MMA row r <-> token RHO(r), row r+8 <-> 8+RHO(r).
//          K int8: thread loads 16 code bytes per 64-dim group; k-step i uses
//          bytes 4i..4i+3, slots (2t, 2t+1, 2t+8, 2t+9) <-> bytes (0, 2, 1, 3),
//          and q's B fragment follows the same permutation.  K fp16: ldmatrix.
//  P.V   : A = V^T, B = P'^T.  Slots (2t, 2t+1) <-> tokens (RHO(2t), RHO(2t+1)),
//          (2t+8, 2t+9) <-> 8 + the same; the q.K^T accumulator fragment, cast
//          to f16x2, becomes this B fragment with one movmatrix transpose.
//          V int8: M-tile m of group g holds dims 64g + 8r + 2m (row r) and
//          +1 (row r+8).  V fp16: ldmatrix.trans, dims d0 + r and d0 + 8 + r.
// RHO = (0,4,2,6,5,1,7,3) makes both the q.K^T and P.V loads conflict free and
// lines the transposed fragment up with the P.V slots.
//
// Query windows (WIN, attn_decode_multi_int8; Strata pull request #2698, "What
// it does": the verify windows of speculative decoding go through the decode
// kernels): the 8 columns are (query, head) pairs instead of heads, query i of
// a window of q_len at position L - q_len + i; a tile after the window's first
// position masks each column's keys beyond its query.

#include <climits>
#include <type_traits>

#include <cooperative_groups.h>
#include <cuda.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "mma_common.cuh"
#include "q4_row.cuh"
#include "quant_row.cuh"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace int8kv {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kMaxCluster = 8;             // splits reduced together through DSMEM
constexpr int kThreads = kConsumerWarps * 32;
constexpr float kTau = 8.f;                // lazy rescale: the running max moves when exceeded by > 2^8
constexpr int kPShift = 6;                 // P' fed to the MMA as P' * 2^(6 - e) < 2^8 * 2^6 = 2^14

// With several V groups a tile splits its softmax weights into fp16 hi + lo once
// and scales them per group in half precision (mma::weight_pair).  The weights are
// split as p * 2^5 (at most 2^13 under the lazy max; an exact scaling) and the
// group factors carry 2^-5 (below 2^1), so that weights down to 2^-19 of the
// reference and V scales down to 2^-15 of the group's range stay normal in fp16.
template <int D, bool VI8, int NG, bool VQ4>
__host__ __device__ constexpr int weight_shift() {
  return (VQ4 ? D / 32 : (VI8 ? NG : 1)) > 1 ? 5 : 0;
}
constexpr int kPagesCached = 256;          // page ids of a block's range kept in shared memory
constexpr float kCap0 = 1.17549435e-38f;   // smallest normal float: below every nonzero fp16 scale
using mma::kPage;
using mma::kBoxBytes;
using mma::kMaxPolls;
using mma::lop_i8pair;
using mma::sub1152;
using mma::pow2f;
using mma::exponent_of;

__device__ __forceinline__ int rho(int r) { return (0x37156240u >> (4 * r)) & 0xF; }

// The block's column group (grid y = kv head + Hkv * column group), read from
// the special register at each use so that it holds no register across the
// page loop.
__device__ __forceinline__ int column_group(int Hkv) {
  int y;
  asm volatile("mov.u32 %0, %%ctaid.y;" : "=r"(y));
  return y / Hkv;
}

template <int D, bool KI8, bool VI8, bool VQ4, bool KQ4 = false>
struct Layout : mma::StagedPage<D, KI8, VI8, VQ4, KQ4> {
  using SP = mma::StagedPage<D, KI8, VI8, VQ4, KQ4>;
  // 4-bit K: the rotated queries' score fragments, fp16 hi + lo pairs, 16 bytes
  // per (k-step, column, lane quarter)
  static constexpr int QFB = KQ4 ? D * 32 : 0;
  // stage budget: three blocks per SM at head_dim 256, four at 128 (whose
  // accumulators fit in the 128 registers that leaves a thread)
  static constexpr int NS_FIT = ((D == 128 ? 52 : 70) * 1024 - QFB) / SP::STAGE;
  static constexpr int NS = NS_FIT < 2 ? 2 : (NS_FIT > 4 ? 4 : NS_FIT);
  // epilogue buffers (reuse the stages): warp partials [warp][head 8][DP], block
  // partial [8][D].  Row pitch DP and dim placement make the warps' fragment
  // stores conflict free: with int8 V a lane holds dims 8r + 2m (+1) of heads
  // 2t, 2t+1, placed at d + d/32 in rows of pitch = 1 (mod 16); with fp16 V,
  // dims r (+8) of the same heads in rows of pitch D + 4 (= 4 mod 16).
  static constexpr int DP = (VI8 || VQ4) ? ((D + D / 32) / 16 + 1) * 16 + 1 : D + 4;
  static constexpr int MERGE = kConsumerWarps * 8 * DP * 4 + 8 * D * 4;
  static constexpr int BARS = NS * SP::STAGE;
  static constexpr int QF_OFF = (BARS + 2 * NS * 8 + NS * 4 + 64 + 127) / 128 * 128;
  static constexpr int SMEM = 1024 + QF_OFF + QFB;   // stages, barriers, page ids, q fragments
  static_assert(MERGE <= NS * SP::STAGE, "merge buffer must fit in the stages");
  // Request pages 1 .. NS-1 only once page 0 has landed (see the kernel).  Only
  // where the tile arithmetic paces the kernel (int8 K and V at head_dim 256):
  // there the smaller first burst lets every block start computing sooner; the
  // byte-bound variants lose more from the shallower start than they gain.
  static constexpr bool DEFER = D == 256 && (KI8 || KQ4) && (VI8 || VQ4);
};

// Codes at byte k of W0 and W1 -> exact f16x2 (lo = W0's, hi = W1's).
__device__ __forceinline__ uint32_t v_pair(uint32_t w0, uint32_t w1, int k) {
  const uint32_t sel = (uint32_t)k | ((uint32_t)k << 4) | ((uint32_t)(4 + k) << 8) |
                       ((uint32_t)(4 + k) << 12);
  return sub1152(lop_i8pair(ptx::prmt(w0, w1, sel)));
}

// 4-bit store: x holds byte b of two keys' chunk words (bytes 0 and 2, and their
// copies in bytes 1 and 3, as v_pair arranges them).  The low nibbles become
// the f16x2 pair (q0 - 8, q1 - 8) with 0x6400 | q = 1024 + q and one subtraction
// of 1032; the high nibbles with 0x6400 | 16 q = 1024 + 16 q, times 1/16, minus
// 72.  All exact in fp16.
__device__ __forceinline__ uint32_t q4_lo(uint32_t x) {
  const uint32_t h = (x & 0x000F000Fu) | 0x64006400u;
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h),
                            __half2half2(__ushort_as_half(0x6408)));
  return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t q4_hi(uint32_t x) {
  const uint32_t h = (x & 0x00F000F0u) | 0x64006400u;
  const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&h),
                            __half2half2(__ushort_as_half(0x2C00)),
                            __half2half2(__ushort_as_half(0xD480)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

template <int D, bool KI8, bool VI8, bool VQ4, bool KQ4 = false>
__device__ __forceinline__ void issue_page(unsigned char* smem, uint64_t* full, int* stage_page,
                                           int st, int page, int row, const PoolView& p, int kvh,
                                           const CUtensorMap* tmk, const CUtensorMap* tmv,
                                           bool expire) {
  if (expire) {   // diagnostic: arm the stage for bytes no copy brings, issue nothing
    stage_page[st] = page;
    ptx::mbar_arrive_expect_tx(&full[st], 16);
    return;
  }
  mma::issue_page<D, KI8, VI8, true, VQ4, KQ4>(smem + st * Layout<D, KI8, VI8, VQ4, KQ4>::STAGE,
                                               &full[st], &stage_page[st], page, row, p, kvh, tmk,
                                               tmv);
}

template <int NG>
__device__ __forceinline__ void load_row_scales(const unsigned char* base, int row, float (&x)[NG]) {
  const unsigned char* p = base + row * NG * 2;
  if constexpr (NG == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  } else if constexpr (NG == 2) {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v));
    x[0] = a.x; x[1] = a.y;
  } else {
    x[0] = __half2float(*reinterpret_cast<const __half*>(p));
  }
}

// The new token's K or V row as one lane of a warp holds it (values
// [lane*VPL, (lane+1)*VPL)): its int8 codes and its group's scale, or, for an
// fp16 store, the values themselves.
template <int D, bool I8>
struct NewRow {
  static constexpr int VPL = D / 32;
  typename Vec<VPL>::H raw;
  typename Vec<VPL>::B codes;
  uint16_t scale;

  // The lane's values (one vector load), then, for an int8 store, their codes
  // and their group's scale.
  __device__ __forceinline__ void fetch(const uint16_t* src, int lane) {
    raw = *reinterpret_cast<const typename Vec<VPL>::H*>(src + lane * VPL);
  }
  __device__ __forceinline__ void quantize(int lanes_per_group) {
    if constexpr (I8) {
      float x[VPL];
      const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
      for (int i = 0; i < VPL / 2; ++i) {
        const float2 f = __half22float2(h2[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
      }
      quantize_regs<VPL>(x, lanes_per_group, codes, scale);
    }
  }
  // Over row `slot` of a staged page: boxes of 64 rows x 128 B with the
  // 128-byte swizzle, scales rows of ng fp16.
  __device__ __forceinline__ void stage(unsigned char* boxes, unsigned char* scales, int slot,
                                        int lane, int lanes_per_group, int ng) const {
    constexpr int EB = I8 ? 1 : 2;   // bytes per value
    const int byte0 = lane * VPL * EB, box = byte0 >> 7, inb = byte0 & 127;
    unsigned char* dst =
        boxes + box * kBoxBytes + slot * 128 + (((inb >> 4) ^ (slot & 7)) << 4) + (inb & 15);
    if constexpr (I8) {
      *reinterpret_cast<typename Vec<VPL>::B*>(dst) = codes;
      if (lane % lanes_per_group == 0)
        reinterpret_cast<uint16_t*>(scales)[slot * ng + lane / lanes_per_group] = scale;
    } else {
      *reinterpret_cast<typename Vec<VPL>::H*>(dst) = raw;
    }
  }
  // Into pool row `row` (values row * D on, scales row * ng on).
  __device__ __forceinline__ void store(void* values, uint16_t* scales, size_t row, int lane,
                                        int lanes_per_group, int ng) const {
    if constexpr (I8) {
      *reinterpret_cast<typename Vec<VPL>::B*>((int8_t*)values + row * D + lane * VPL) = codes;
      if (lane % lanes_per_group == 0) scales[row * ng + lane / lanes_per_group] = scale;
    } else {
      *reinterpret_cast<typename Vec<VPL>::H*>((uint16_t*)values + row * D + lane * VPL) = raw;
    }
  }
};

// The new token's V row for the 4-bit store (head_dim 256, 8 values a lane):
// rotated and quantized by the warp as the append kernel does it, then written
// over its staged row and to the pool in the chunked nibble order.
struct NewRowQ4 {
  static constexpr int D = 256, VPL = 8;
  uint4 raw;
  uint32_t packed;
  uint16_t scale;
  __device__ __forceinline__ void fetch(const uint16_t* src, int lane) {
    raw = *reinterpret_cast<const uint4*>(src + lane * VPL);
  }
  __device__ __forceinline__ void quantize(int) {
    float x[VPL];
    const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
    for (int i = 0; i < VPL / 2; ++i) {
      const float2 f = __half22float2(h2[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
    fwht_row<VPL>(x, threadIdx.x & 31, 0.0625f);
    packed = q4_0_regs<VPL>(x, threadIdx.x & 31, scale);
  }
  __device__ __forceinline__ void stage(unsigned char* boxes, unsigned char* scales, int slot,
                                        int lane, int, int) const {
#pragma unroll
    for (int q = 0; q < VPL / 2; ++q) {
      const int byte = q4_byte_of(lane * VPL + 2 * q, D);
      boxes[slot * 128 + ((((byte >> 4) ^ (slot & 7))) << 4) + (byte & 15)] = (uint8_t)(packed >> (8 * q));
    }
    if (lane % 4 == 0) reinterpret_cast<uint16_t*>(scales)[slot * (D / 32) + lane / 4] = scale;
  }
  __device__ __forceinline__ void store(void* values, uint16_t* scales, size_t row, int lane, int,
                                        int) const {
#pragma unroll
    for (int q = 0; q < VPL / 2; ++q)
      ((uint8_t*)values)[row * (D / 2) + q4_byte_of(lane * VPL + 2 * q, D)] = (uint8_t)(packed >> (8 * q));
    if (lane % 4 == 0) scales[row * (D / 32) + lane / 4] = scale;
  }
};

// One 16-token tile of one page for one warp: scores for the G heads, online
// softmax (lazy: the reference max moves only when a score exceeds it by more
// than 2^kTau), and the P.V accumulation.  FULL: every token of the tile is in
// [j0, j1), so no masking.
template <int D, bool KI8, bool VI8, int NG, bool FULL, bool VQ4, bool KQ4>
__device__ __forceinline__ void decode_tile(const unsigned char* sb, int warp, int lane, int tile0,
                                            int j0, int j1, const uint32_t (&qf)[D / 16][2],
                                            const uint4* qfrag, float scale_log2,
                                            float (&o)[D / 16][4], float& m0, float& m1, float& l0,
                                            float& l1, float (&cap)[NG], float (&sh)[NG],
                                            int (&vexp)[NG], int lim0, int lim1) {
  using LY = Layout<D, KI8, VI8, VQ4, KQ4>;
  constexpr int MACROS = D / 64, MTILES = D / 16;
  constexpr int NGV = VQ4 ? D / 32 : (VI8 ? NG : 1);   // V scale groups (4-bit store: of 32)
  constexpr int MPG = VQ4 ? 0 : MACROS / NGV;   // 64-dim macros per V scale group
  const int r = lane >> 2, t = lane & 3;
  const int rowA = rho(r), rowB = rowA + 8;
  const int trA = warp * 16 + rowA, trB = warp * 16 + rowB;   // rows within the page
  const int tokS0 = rho(2 * t), tokS1 = rho(2 * t + 1);       // P.V slot tokens
  bool vA = true, vB = true;
  if constexpr (!FULL) {
    vA = tile0 + rowA >= j0 && tile0 + rowA < j1;
    vB = tile0 + rowB >= j0 && tile0 + rowB < j1;
  }

  // ---- scores: s[0..1] token A heads (2t, 2t+1); s[2..3] token B
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (KQ4) {
    // 4-bit K (rotated rows, Q4_0 blocks of 32 values, signed fp16 scales): the
    // lane loads chunks t and t + 4 of its two rows, values 32g + 4t + j and
    // 32g + 16 + 4t + j of every block g.  Block g is two k-steps (chunk t, then
    // t + 4); in each, k-slots (2t, 2t + 1) take the low nibbles of bytes 2g and
    // 2g + 1 (values 4t + 0, 4t + 2 of the chunk's group) and slots (2t + 8,
    // 2t + 9) their high nibbles (4t + 1, 4t + 3); the rotated query fragments
    // follow the same order, as fp16 hi + lo pairs (two MMAs per k-step).
    const int sa_ = rowA, sb_ = rowB & 7;
    // word w of chunk (t + 4h) of each row, loaded where it is used (four words
    // a chunk; holding the chunks whole would cost 16 registers)
    const uint32_t* kA0 = reinterpret_cast<const uint32_t*>(sb + LY::K_OFF + trA * 128 + ((t ^ sa_) << 4));
    const uint32_t* kA1 = reinterpret_cast<const uint32_t*>(sb + LY::K_OFF + trA * 128 + (((t + 4) ^ sa_) << 4));
    const uint32_t* kB0 = reinterpret_cast<const uint32_t*>(sb + LY::K_OFF + trB * 128 + ((t ^ sb_) << 4));
    const uint32_t* kB1 = reinterpret_cast<const uint32_t*>(sb + LY::K_OFF + trB * 128 + (((t + 4) ^ sb_) << 4));
    const uint32_t* dA = reinterpret_cast<const uint32_t*>(sb + LY::KS_OFF + trA * 16);
    const uint32_t* dB = reinterpret_cast<const uint32_t*>(sb + LY::KS_OFF + trB * 16);
    const uint4* qv = qfrag + r * 4 + t;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int wi = g >> 1;
        const uint32_t wa = (h ? kA1 : kA0)[wi], wb = (h ? kB1 : kB0)[wi];
        const uint32_t sel = (g & 1) ? 0x4342u : 0x4140u;   // bytes 2g, 2g + 1 -> bytes 0, 2
        const uint32_t xa = ptx::prmt(wa, 0u, sel), xb = ptx::prmt(wb, 0u, sel);
        uint32_t af[4];
        af[0] = q4_lo(xa);
        af[1] = q4_lo(xb);
        af[2] = q4_hi(xa);
        af[3] = q4_hi(xb);
        const uint4 qq = qv[(g * 2 + h) * 32];
        ptx::mma_f16(acc, af, qq.x, qq.y);
        ptx::mma_f16(acc, af, qq.z, qq.w);
      }
      const uint32_t pa = dA[g >> 1], pb = dB[g >> 1];
      const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&pa));
      const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&pb));
      const float sa = (g & 1) ? fa.y : fa.x, sbb = (g & 1) ? fb.y : fb.x;
      s[0] = fmaf(acc[0], sa, s[0]);
      s[1] = fmaf(acc[1], sa, s[1]);
      s[2] = fmaf(acc[2], sbb, s[2]);
      s[3] = fmaf(acc[3], sbb, s[3]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) s[k] *= scale_log2;   // the softmax scale, once
  } else if constexpr (KI8) {
    float ka[NG], kb[NG];
    load_row_scales<NG>(sb + LY::KS_OFF, trA, ka);
    load_row_scales<NG>(sb + LY::KS_OFF, trB, kb);
    const int xa0 = trA * 128 + ((t ^ rowA) << 4), xa1 = trA * 128 + (((4 + t) ^ rowA) << 4);
    const int xb0 = trB * 128 + ((t ^ (rowB & 7)) << 4);
    const int xb1 = trB * 128 + (((4 + t) ^ (rowB & 7)) << 4);
#pragma unroll
    for (int mc = 0; mc < MACROS; ++mc) {
      const unsigned char* kb0 = sb + LY::K_OFF + (mc >> 1) * kBoxBytes;
      const uint4 wa = *reinterpret_cast<const uint4*>(kb0 + ((mc & 1) ? xa1 : xa0));
      const uint4 wb = *reinterpret_cast<const uint4*>(kb0 + ((mc & 1) ? xb1 : xb0));
      const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w};
      const uint32_t wB[4] = {wb.x, wb.y, wb.z, wb.w};
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        uint32_t af[4];
        af[0] = sub1152(lop_i8pair(wA[ii]));
        af[1] = sub1152(lop_i8pair(wB[ii]));
        af[2] = sub1152(lop_i8pair(wA[ii] >> 8));
        af[3] = sub1152(lop_i8pair(wB[ii] >> 8));
        ptx::mma_f16(acc, af, qf[mc * 4 + ii][0], qf[mc * 4 + ii][1]);
      }
      // the softmax scale: with a group per macro, once on the sums below;
      // otherwise folded into each group's scale (fewer multiplies either way)
      const int grp = mc / (MACROS / NG);
      const float sa = NG == MACROS ? ka[grp] : ka[grp] * scale_log2;
      const float sbb = NG == MACROS ? kb[grp] : kb[grp] * scale_log2;
      s[0] = fmaf(acc[0], sa, s[0]);
      s[1] = fmaf(acc[1], sa, s[1]);
      s[2] = fmaf(acc[2], sbb, s[2]);
      s[3] = fmaf(acc[3], sbb, s[3]);
    }
    if constexpr (NG == MACROS)
#pragma unroll
      for (int k = 0; k < 4; ++k) s[k] *= scale_log2;
  } else {
    const int q4 = lane >> 3, rr = lane & 7;
    const int tok = warp * 16 + rho(rr) + 8 * (q4 & 1);
#pragma unroll
    for (int mc = 0; mc < MACROS; ++mc) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const int c = ii * 2 + (q4 >> 1);   // 8-half chunk within the 64-dim box row
        uint32_t af[4];
        ptx::ldmatrix_x4(af, ptx::smem_u32(sb + LY::K_OFF + mc * kBoxBytes + tok * 128 +
                                           ((c ^ (tok & 7)) << 4)));
        ptx::mma_f16(acc, af, qf[mc * 4 + ii][0], qf[mc * 4 + ii][1]);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) s[k] += acc[k];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) s[k] *= scale_log2;
  }
  if constexpr (!FULL) {   // outside [j0, j1), or after the column's query position
    const int pA = tile0 + rowA, pB = tile0 + rowB;
    if (!vA || pA > lim0) s[0] = -INFINITY;
    if (!vA || pA > lim1) s[1] = -INFINITY;
    if (!vB || pB > lim0) s[2] = -INFINITY;
    if (!vB || pB > lim1) s[3] = -INFINITY;
  }

  // ---- online softmax (base 2) per head column, lazy reference max: a lane's
  // own scores decide whether the tile moves it; the column maxima are formed
  // only then (rarely)
  float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
  if (__any_sync(0xffffffffu, mx0 > m0 + kTau || mx1 > m1 + kTau)) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = mn0 == -INFINITY ? 1.f : ptx::ex2(m0 - mn0);
    const float al1 = mn1 == -INFINITY ? 1.f : ptx::ex2(m1 - mn1);
    l0 *= al0;
    l1 *= al1;
#pragma unroll
    for (int j = 0; j < MTILES; ++j) {
      o[j][0] *= al0;
      o[j][1] *= al1;
      o[j][2] *= al0;
      o[j][3] *= al1;
    }
    m0 = mn0;
    m1 = mn1;
  }
  constexpr int KPS = weight_shift<D, VI8, NG, VQ4>();
  const float base0 = m0 == -INFINITY ? 0.f : m0, base1 = m1 == -INFINITY ? 0.f : m1;
  float pr[4];
  pr[0] = ptx::ex2(s[0] - base0);
  pr[1] = ptx::ex2(s[1] - base1);
  pr[2] = ptx::ex2(s[2] - base0);
  pr[3] = ptx::ex2(s[3] - base1);
  l0 += pr[0] + pr[2];
  l1 += pr[1] + pr[3];

  // ---- token weights per V group: s_v * 2^(kPShift - e_g) (times 2^-5 where the
  // weights are split first, see weight_shift), the range 2^e_g raised (and the
  // group's accumulators rescaled) when a larger V scale shows up
  float wa[NGV], wb[NGV];
  if constexpr (VI8) {
    float va[NG], vb[NG];
    load_row_scales<NG>(sb + LY::VS_OFF, trA, va);
    load_row_scales<NG>(sb + LY::VS_OFF, trB, vb);
    bool need = false;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      if constexpr (!FULL) {
        va[g] = vA ? va[g] : 0.f;
        vb[g] = vB ? vb[g] : 0.f;
      }
      need |= fmaxf(va[g], vb[g]) >= cap[g];   // cap > 0: a zero scale never moves it
    }
    if (__any_sync(0xffffffffu, need)) {
      // the scales depend on the lane's rows only (lanes 4r .. 4r + 3 agree):
      // the three upper xor levels give the warp's maximum, the groups' chains
      // interleaved
      float mx[NG];
#pragma unroll
      for (int g = 0; g < NG; ++g) mx[g] = fmaxf(va[g], vb[g]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)
#pragma unroll
        for (int g = 0; g < NG; ++g) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xffffffffu, mx[g], off));
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        if (mx[g] >= cap[g]) {
          const int ne = exponent_of(mx[g]) + 1;
          if (vexp[g] != INT_MIN) {
            const float f = pow2f(vexp[g] - ne);
#pragma unroll
            for (int j = g * MPG * 4; j < (g + 1) * MPG * 4; ++j) {
              o[j][0] *= f;
              o[j][1] *= f;
              o[j][2] *= f;
              o[j][3] *= f;
            }
          }
          vexp[g] = ne;
          cap[g] = pow2f(ne);
          sh[g] = pow2f(kPShift - KPS - ne);
        }
      }
    }
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      wa[g] = va[g] * sh[g];
      wb[g] = vb[g] * sh[g];
    }
  } else if constexpr (VQ4) {
    // 4-bit store: D/32 signed scales per key (d = m * -1/8).  One range 2^e per
    // warp bounds |d| of every block (index 0 of the range arrays): the rotation
    // makes the blocks' scales of a key alike, and a block far below the range
    // only loses bits of weights that are already negligible.
    float va[NGV], vb[NGV];
    {
      const uint4 xa = *reinterpret_cast<const uint4*>(sb + LY::VS_OFF + trA * (NGV * 2));
      const uint4 xb = *reinterpret_cast<const uint4*>(sb + LY::VS_OFF + trB * (NGV * 2));
      const uint32_t wa32[4] = {xa.x, xa.y, xa.z, xa.w}, wb32[4] = {xb.x, xb.y, xb.z, xb.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&wa32[i]));
        const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&wb32[i]));
        va[2 * i] = fa.x;
        va[2 * i + 1] = fa.y;
        vb[2 * i] = fb.x;
        vb[2 * i + 1] = fb.y;
      }
    }
    float mx = 0.f;
#pragma unroll
    for (int g = 0; g < NGV; ++g) {
      if constexpr (!FULL) {
        va[g] = vA ? va[g] : 0.f;
        vb[g] = vB ? vb[g] : 0.f;
      }
      mx = fmaxf(mx, fmaxf(fabsf(va[g]), fabsf(vb[g])));
    }
    if (__any_sync(0xffffffffu, mx >= cap[0])) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      if (mx >= cap[0]) {   // warp-uniform
        const int ne = exponent_of(mx) + 1;
        if (vexp[0] != INT_MIN) {
          const float f = pow2f(vexp[0] - ne);
#pragma unroll
          for (int j = 0; j < MTILES; ++j) {
            o[j][0] *= f;
            o[j][1] *= f;
            o[j][2] *= f;
            o[j][3] *= f;
          }
        }
        vexp[0] = ne;
        cap[0] = pow2f(ne);
        sh[0] = pow2f(kPShift - KPS - ne);
      }
    }
#pragma unroll
    for (int g = 0; g < NGV; ++g) {
      wa[g] = va[g] * sh[0];
      wb[g] = vb[g] * sh[0];
    }
  } else {
    wa[0] = (FULL || vA) ? pow2f(kPShift) : 0.f;
    wb[0] = (FULL || vB) ? pow2f(kPShift) : 0.f;
  }

  if constexpr (VQ4) {
    // ---- P.V for the 4-bit store: each key's chunk r (16 bytes: values
    // 32g + 4r .. 32g + 4r + 3 of every block g) is one load; M-tile (g, h) takes
    // rows r <-> value 32g + 4r + 2h (low nibble of byte 2g + h), r + 8 <-> the
    // next value (high nibble)
    const int tk[4] = {warp * 16 + tokS0, warp * 16 + tokS1, warp * 16 + 8 + tokS0,
                       warp * 16 + 8 + tokS1};
    uint4 qv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      qv[j] = *reinterpret_cast<const uint4*>(sb + LY::V_OFF + tk[j] * 128 + ((r ^ (tk[j] & 7)) << 4));
    uint32_t pha, pla, phb, plb;   // p * 2^5 of tokens A and B (heads 2t, 2t + 1), fp16 hi + lo
    mma::split_pair(pr[0] * (1 << KPS), pr[1] * (1 << KPS), pha, pla);
    mma::split_pair(pr[2] * (1 << KPS), pr[3] * (1 << KPS), phb, plb);
#pragma unroll
    for (int g = 0; g < NGV; ++g) {
      uint32_t h01, e01, h23, e23;
      mma::weight_pair(pha, pla, ptx::pack_f16x2(wa[g], wa[g]), h01, e01);
      mma::weight_pair(phb, plb, ptx::pack_f16x2(wb[g], wb[g]), h23, e23);
      const uint32_t bh0 = ptx::movmatrix_trans(h01), bh1 = ptx::movmatrix_trans(h23);
      const uint32_t bl0 = ptx::movmatrix_trans(e01), bl1 = ptx::movmatrix_trans(e23);
      const int wi = g >> 1;   // the word of the chunk that holds block g's bytes
      const uint32_t w0 = wi == 0 ? qv[0].x : wi == 1 ? qv[0].y : wi == 2 ? qv[0].z : qv[0].w;
      const uint32_t w1 = wi == 0 ? qv[1].x : wi == 1 ? qv[1].y : wi == 2 ? qv[1].z : qv[1].w;
      const uint32_t w2 = wi == 0 ? qv[2].x : wi == 1 ? qv[2].y : wi == 2 ? qv[2].z : qv[2].w;
      const uint32_t w3 = wi == 0 ? qv[3].x : wi == 1 ? qv[3].y : wi == 2 ? qv[3].z : qv[3].w;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int bsel = 2 * (g & 1) + hh;   // byte 2g + hh of the chunk, within word wi
        const uint32_t sel = (uint32_t)bsel | ((uint32_t)bsel << 4) | ((uint32_t)(4 + bsel) << 8) |
                             ((uint32_t)(4 + bsel) << 12);
        const uint32_t x01 = ptx::prmt(w0, w1, sel), x23 = ptx::prmt(w2, w3, sel);
        uint32_t af[4];
        af[0] = q4_lo(x01);
        af[1] = q4_hi(x01);
        af[2] = q4_lo(x23);
        af[3] = q4_hi(x23);
        ptx::mma_f16(o[2 * g + hh], af, bh0, bh1);
        ptx::mma_f16(o[2 * g + hh], af, bl0, bl1);
      }
    }
    return;
  }

  // ---- P.V per V group: P' = p * w as an f16 hi + lo pair, transposed into the
  // B fragment.  Several groups: p * 2^5 is split once and each group's factor
  // w * 2^-5 (an fp16 scale times a power of two, below 2^1: exact in fp16 unless
  // subnormal) applied in half precision; one group: P' formed in fp32 and split.
  uint32_t pha = 0, pla = 0, phb = 0, plb = 0;   // p of tokens A and B (heads 2t, 2t + 1)
  if constexpr (NGV > 1) {   // split as p * 2^5
    mma::split_pair(pr[0] * (1 << KPS), pr[1] * (1 << KPS), pha, pla);
    mma::split_pair(pr[2] * (1 << KPS), pr[3] * (1 << KPS), phb, plb);
  }
#pragma unroll
  for (int g = 0; g < NGV; ++g) {
    uint32_t h01, e01, h23, e23;
    if constexpr (NGV > 1) {
      mma::weight_pair(pha, pla, ptx::pack_f16x2(wa[g], wa[g]), h01, e01);
      mma::weight_pair(phb, plb, ptx::pack_f16x2(wb[g], wb[g]), h23, e23);
    } else {
      mma::weight_pair_f32(pr[0], pr[1], wa[0], h01, e01);
      mma::weight_pair_f32(pr[2], pr[3], wb[0], h23, e23);
    }
    const uint32_t bh0 = ptx::movmatrix_trans(h01), bh1 = ptx::movmatrix_trans(h23);
    const uint32_t bl0 = ptx::movmatrix_trans(e01), bl1 = ptx::movmatrix_trans(e23);
#pragma unroll
    for (int mm = 0; mm < MPG; ++mm) {
      const int mc = g * MPG + mm;
      if constexpr (VI8) {
        const unsigned char* vb0 = sb + LY::V_OFF + (mc >> 1) * kBoxBytes;
        const int c16 = (mc & 1) * 4 + (r >> 1), h8 = (r & 1) << 3;
        const int tk[4] = {warp * 16 + tokS0, warp * 16 + tokS1, warp * 16 + 8 + tokS0,
                           warp * 16 + 8 + tokS1};
        uint2 w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          w[j] = *reinterpret_cast<const uint2*>(vb0 + tk[j] * 128 + (((c16 ^ (tk[j] & 7)) << 4) | h8));
        uint32_t af[4][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          const int kbyte = 2 * (mt & 1);
          const uint32_t x0 = (mt >> 1) ? w[0].y : w[0].x, x1 = (mt >> 1) ? w[1].y : w[1].x;
          const uint32_t x2 = (mt >> 1) ? w[2].y : w[2].x, x3 = (mt >> 1) ? w[3].y : w[3].x;
          af[mt][0] = v_pair(x0, x1, kbyte);
          af[mt][1] = v_pair(x0, x1, kbyte + 1);
          af[mt][2] = v_pair(x2, x3, kbyte);
          af[mt][3] = v_pair(x2, x3, kbyte + 1);
        }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) ptx::mma_f16(o[mc * 4 + mt], af[mt], bh0, bh1);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) ptx::mma_f16(o[mc * 4 + mt], af[mt], bl0, bl1);
      } else {
        const int q4 = lane >> 3, rr = lane & 7;
        const int tok = warp * 16 + rho(rr) + 8 * (q4 >> 1);
        uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
        if constexpr (!FULL) {
          // rows outside [j0, j1) may hold any bits: zero them (P' is 0 there)
          const bool ok0 = tile0 + tokS0 >= j0 && tile0 + tokS0 < j1;
          const bool ok1 = tile0 + tokS1 >= j0 && tile0 + tokS1 < j1;
          const bool ok2 = tile0 + 8 + tokS0 >= j0 && tile0 + 8 + tokS0 < j1;
          const bool ok3 = tile0 + 8 + tokS1 >= j0 && tile0 + 8 + tokS1 < j1;
          mlo = (ok0 ? 0x0000FFFFu : 0u) | (ok1 ? 0xFFFF0000u : 0u);
          mhi = (ok2 ? 0x0000FFFFu : 0u) | (ok3 ? 0xFFFF0000u : 0u);
        }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          const int c = mt * 2 + (q4 & 1);
          uint32_t af[4];
          ptx::ldmatrix_x4_trans(af, ptx::smem_u32(sb + LY::V_OFF + mc * kBoxBytes + tok * 128 +
                                                   ((c ^ (tok & 7)) << 4)));
          if constexpr (!FULL) {
            af[0] &= mlo;
            af[1] &= mlo;
            af[2] &= mhi;
            af[3] &= mhi;
          }
          ptx::mma_f16(o[mc * 4 + mt], af, bh0, bh1);
          ptx::mma_f16(o[mc * 4 + mt], af, bl0, bl1);
        }
      }
    }
  }
}

// WIN: a window of q_len queries per sequence (attn_decode_multi_int8); without
// it the kernel serves one query per sequence and none of the window's column
// arithmetic is compiled in.
template <int D, bool KI8, bool VI8, int NG, bool WIN, bool VQ4, bool KQ4 = false>
__global__ void __launch_bounds__(kThreads, D == 128 ? 4 : 3)
decode_mma_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, int layer_page0) {
  static_assert(!KQ4 || (D == 256 && VQ4 && !KI8 && !VI8 && NG == 1),
                "4-bit K: head_dim 256, with the 4-bit V store");
  using LY = Layout<D, KI8, VI8, VQ4, KQ4>;
  constexpr int KSTEPS = D / 16;     // 16-dim k-steps of q.K^T
  constexpr int MACROS = D / 64;     // 64-dim groups
  constexpr int MTILES = D / 16;     // 16-dim M-tiles of P.V
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = (uint64_t*)(smem + LY::BARS);
  int* stage_page = (int*)(full + 2 * LY::NS);
  __shared__ float s_m[kConsumerWarps][8], s_l[kConsumerWarps][8];
  __shared__ float s_f[kConsumerWarps][8], s_inv[8];
  __shared__ float s_cm[8][8], s_cl[8][8], s_cL[8];
  __shared__ int s_rel[4];                // per stage: release tickets (the last warp refills)
  __shared__ int s_q0[kConsumerWarps];   // WIN: L - q_len, the first query's position
  // page ids: the sequence's whole page-table row when it has at most
  // kPagesCached entries, else the entries of the block's first pages
  __shared__ int s_pages[kPagesCached];

  const PoolView& p = a.pool;
  const int split = blockIdx.x, kvh = blockIdx.y % p.Hkv, b = blockIdx.z;
  const uint32_t max_polls = a.expire_polls ? a.expire_polls : kMaxPolls;   // bounded waits
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.G;
  // B operand column c <-> (query, head) pair colg * 8 + c of the kv head's
  // q_len * G (colg: the block's column group); with one query (decode) column
  // c is head c.  Live columns: c < ncol().
  auto ncol = [&]() { return WIN ? min(8, a.q_len * G - column_group(p.Hkv) * 8) : G; };
  auto col_row = [&](int c) -> size_t {   // the column's row of q and out: [B][q_len][H]
    if constexpr (!WIN) return (size_t)b * a.H + (size_t)kvh * G + c;
    const int f = column_group(p.Hkv) * 8 + c;
    return ((size_t)b * a.q_len + f / G) * a.H + (size_t)kvh * G + f % G;
  };
  constexpr int gs = D / NG;   // width of a scale group (>= 64)

  if (threadIdx.x == 0) {
    ptx::prefetch_tensormap(&tmk);   // kernel parameters: safe before the grid dependency
    ptx::prefetch_tensormap(&tmv);
    for (int s = 0; s < LY::NS; ++s) {
      ptx::mbar_init(&full[s], 1);
      s_rel[s] = 0;
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();
  // Launched as a programmatic dependent: nothing read before the preceding
  // kernel of the stream has completed is used, except as a prefetch hint.
  // Thread 0 reads the length and the first page id of its range through L2
  // (never L1, so no stale line outlives the wait) and has L2 fetch that page,
  // which overlaps its HBM latency with the end of the preceding kernel.  A
  // length or page id that kernel still changes only makes the prefetch
  // useless: the id is checked against the pool before use, and L2 is coherent
  // with the writes that follow.
  const int lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);   // launch order
  if (threadIdx.x == 0 && lin < a.pf_blocks) {
    int Ls = ptx::ldcg32(a.seq_lens + b);
    Ls = Ls < 0 ? 0 : min(Ls, a.max_pages * kPage);
    const int lo = a.window > 0 ? max(0, Ls - a.window) : 0;
    int s0 = lo, s1 = lo;
    split_range(lo, Ls, split, a.n_splits, kPage, &s0, &s1);
    const int pg = s1 > s0 ? ptx::ldcg32(a.page_table + (size_t)b * a.max_pages + s0 / kPage) : -1;
    if (pg >= 0 && pg < p.n_pages) {
      const size_t r0 = ((size_t)pg * p.Hkv + kvh) * kPage;   // first row of the page-head
      constexpr int KROW = KQ4 ? D / 2 : (KI8 ? D : 2 * D);   // bytes of a K row
      constexpr int VROW = VQ4 ? D / 2 : (VI8 ? D : 2 * D);   // bytes of a V row
      ptx::bulk_prefetch_l2((const char*)p.k + r0 * KROW, KROW * kPage);
      ptx::bulk_prefetch_l2((const char*)p.v + r0 * VROW, VROW * kPage);
      if (KI8) ptx::bulk_prefetch_l2(p.ks + r0 * NG, kPage * NG * 2);
      if (KQ4) ptx::bulk_prefetch_l2(p.ks + r0 * (D / 32), kPage * (D / 32) * 2);
      if (VI8) ptx::bulk_prefetch_l2(p.vs + r0 * NG, kPage * NG * 2);
      if (VQ4) ptx::bulk_prefetch_l2(p.vs + r0 * (D / 32), kPage * (D / 32) * 2);
    }
  }
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();

  const int L_raw = ptx::ldg32(a.seq_lens + b);
  // A short page-table row is read whole, along with the length (the block's
  // pages are not known before it).
  const int32_t* ptrow = a.page_table + (size_t)b * a.max_pages;
  const bool row_cached = a.max_pages <= kPagesCached;
  if (row_cached) {
    constexpr int PER = kPagesCached / kThreads;
    int e[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = threadIdx.x + k * kThreads;
      e[k] = i < a.max_pages ? ptx::ldg32(ptrow + i) : 0;
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) s_pages[threadIdx.x + k * kThreads] = e[k];
  }
  // q of head r (B operand columns = heads): requested now, arranged in the
  // slot order of the K loads once the pages are on their way
  const int r = lane >> 2, t = lane & 3;
  constexpr int QV = D / 64 * 2;   // 16-byte pieces of q a lane holds
  uint4 qraw[QV];
  {
    const bool live = r < ncol();
    const uint16_t* qh = a.q + col_row(live ? r : 0) * D;
#pragma unroll
    for (int v = 0; v < QV; ++v) {
      // int8 K: dims 64mc + 16t + 8h (v = 2mc + h); fp16 K: dims 16ks + 2t (+8), see below
      if constexpr (KI8)
        qraw[v] = live ? ptx::ldg128(qh + (v >> 1) * 64 + 16 * t + 8 * (v & 1)) : make_uint4(0, 0, 0, 0);
    }
    if constexpr (!KI8 && !KQ4) {
      const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qh);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t* w = reinterpret_cast<uint32_t*>(&qraw[ks >> 1]) + 2 * (ks & 1);
        w[0] = live ? __ldg(q32 + (ks * 16 + 2 * t) / 2) : 0u;
        w[1] = live ? __ldg(q32 + (ks * 16 + 8 + 2 * t) / 2) : 0u;
      }
    }
  }
  const int L = clamp_length(L_raw, a.max_pages, p);
  const int lo_pos = a.window > 0 ? max(0, L - a.window) : 0;
  // Query i of a window sits at L - q_len + i and sees keys up to it.  The
  // first query's position is kept in shared memory (one copy per warp, read
  // only by the warp), so that the page loop holds no register for it.
  if constexpr (WIN) {
    if (lane == 0) s_q0[warp] = L - a.q_len;
    __syncwarp();
  }
  int j0, j1;
  split_range(lo_pos, L, split, a.n_splits, kPage, &j0, &j1);
  const int p_first = j0 / kPage;
  const int n_pg = j1 > j0 ? (j1 - 1) / kPage - p_first + 1 : 0;

  // Fused append: when the block's range holds the new token (position L-1),
  // it is the range's last row.  The warp whose tile holds it writes the new K
  // row, its neighbour the new V row (loads issued here, the rest once the
  // pages are requested).  No other block reads the row.
  const bool appends = a.k_new != nullptr && L == L_raw && L > 0 && L - 1 >= j0 && L - 1 < j1;
  const int app_slot = (L - 1) & (kPage - 1);
  const bool app_k = appends && warp == app_slot / 16;
  const bool app_v = appends && warp == ((app_slot / 16) ^ 1);
  std::conditional_t<KQ4, NewRowQ4, NewRow<D, KI8>> nk;
  std::conditional_t<VQ4, NewRowQ4, NewRow<D, VI8>> nv;
  if (app_k) nk.fetch(a.k_new + ((size_t)b * p.Hkv + kvh) * D, lane);
  if (app_v) nv.fetch(a.v_new + ((size_t)b * p.Hkv + kvh) * D, lane);

  // Thread 0 requests the block's first NS pages; with LY::DEFER, the first
  // page alone, and pages 1 .. NS-1 once it has landed: every block of the
  // grid starts at once, so a first burst of NS pages per block makes every
  // block's first page land late.  (A block that appends requests all NS at
  // once: its append warps may wait on any of them before the page loop.)
  // Afterwards the last warp to release a stage refills it with page i + NS.
  // When the row is not held whole, the ids of the block's first pages go to
  // shared memory meanwhile; no barrier is needed before the refills read
  // them: every warp writes its share before it first releases a stage (a
  // release the refilling warp acquires), and the consumers learn of a
  // stage's page through its mbarrier.
  auto page_row = [&](int page) { return ((layer_page0 + page) * p.Hkv + kvh) * kPage; };
  if (row_cached) __syncthreads();
  auto page_direct = [&](int i) {   // page i of the block's range, from the row or from memory
    return row_cached ? check_page(s_pages[p_first + i], p)
                      : lookup_page(ptrow, p_first + i, a.max_pages, p);
  };
  if (threadIdx.x == 0) {
    int first[LY::NS];
#pragma unroll
    for (int i = 0; i < LY::NS; ++i)   // independent loads, in flight together
      first[i] = i < n_pg ? page_direct(i) : -1;
#pragma unroll
    for (int i = 0; i < LY::NS; ++i)
      if (i < n_pg) {
        if (i == 0 || appends || !LY::DEFER)
          issue_page<D, KI8, VI8, VQ4, KQ4>(smem, full, stage_page, i, first[i], page_row(first[i]), p, kvh,
                                  &tmk, &tmv, a.expire_polls != 0);
        else
          stage_page[i] = first[i];   // kept for the request after page 0 lands; no consumer
                                      // reads it before that request's mbarrier completes
      }
  }
  if (!row_cached)
    for (int i = threadIdx.x; i < n_pg && i < kPagesCached; i += kThreads)
      s_pages[i] = lookup_page(ptrow, p_first + i, a.max_pages, p);
  auto page_of = [&](int i) {
    if (row_cached) return check_page(s_pages[p_first + i], p);
    return i < kPagesCached ? s_pages[i] : lookup_page(ptrow, p_first + i, a.max_pages, p);
  };
  uint32_t qf[KSTEPS][2];
  const uint4* qfrag = reinterpret_cast<const uint4*>(smem + LY::QF_OFF);
  if constexpr (KQ4) {
    // Rotated queries for the 4-bit K store: warp w rotates columns w and w + 4
    // (a lane 8 consecutive dims; the same fp32 FWHT as the store), splits each
    // value into an fp16 hi + lo pair and stores them in the tile's k-slot order:
    // dims 8 lane + 4u + j are values 32g + 16h + 4t + j with g = lane / 4,
    // h = (lane / 2) & 1, t = 2 (lane & 1) + u; the piece of (g, h, column c,
    // t) holds the pairs (j0, j2), (j1, j3) of hi, then of lo.
    uint4* qw = reinterpret_cast<uint4*>(smem + LY::QF_OFF);
    for (int c = warp; c < 8; c += kConsumerWarps) {
      float x[8];
      if (c < ncol()) {
        const uint4 raw = ptx::ldg128(a.q + col_row(c) * D + lane * 8);
        const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(h2[i]);
          x[2 * i] = f.x;
          x[2 * i + 1] = f.y;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = 0.f;
      }
      fwht_row<8>(x, lane, 0.0625f);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        uint16_t hi[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __half h = __float2half_rn(x[4 * u + j]);
          hi[j] = __half_as_ushort(h);
          lo[j] = __half_as_ushort(__float2half_rn(x[4 * u + j] - __half2float(h)));
        }
        const int g = lane >> 2, h = (lane >> 1) & 1, tt = 2 * (lane & 1) + u;
        qw[((g * 2 + h) * 8 + c) * 4 + tt] =
            make_uint4(hi[0] | ((uint32_t)hi[2] << 16), hi[1] | ((uint32_t)hi[3] << 16),
                       lo[0] | ((uint32_t)lo[2] << 16), lo[1] | ((uint32_t)lo[3] << 16));
      }
    }
    __syncthreads();
  } else if constexpr (KI8) {
#pragma unroll
    for (int mc = 0; mc < MACROS; ++mc) {
      // dims 64mc + 16t .. +16: k-step i takes (4i, 4i+2) and (4i+1, 4i+3)
      const uint4 x = qraw[2 * mc], y = qraw[2 * mc + 1];
      const uint32_t w[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        qf[mc * 4 + i][0] = ptx::prmt(w[2 * i], w[2 * i + 1], 0x5410);
        qf[mc * 4 + i][1] = ptx::prmt(w[2 * i], w[2 * i + 1], 0x7632);
      }
    }
  } else {
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      const uint32_t* w = reinterpret_cast<const uint32_t*>(&qraw[ks >> 1]) + 2 * (ks & 1);
      qf[ks][0] = w[0];
      qf[ks][1] = w[1];
    }
  }
  if (app_k || app_v) {
    // If the last page was issued above, the new row is written over its
    // staged row once it has landed (the copy brought the row's old contents)
    // and then to the pool; otherwise it goes to the pool now, ahead of that
    // page's copy (a refill, issued only after both warps released a stage).
    constexpr int LPG = (D / NG) / (D / 32);   // lanes per scale group
    if (app_k)
      nk.quantize(LPG);
    else
      nv.quantize(LPG);
    const int last = n_pg - 1;
    int page = -1;
    if (last < LY::NS) {
      if (ptx::mbar_wait(&full[last], 0, max_polls)) {
        page = stage_page[last];
        if (page >= 0) {
          unsigned char* sw = smem + last * LY::STAGE;
          if (app_k)
            nk.stage(sw + LY::K_OFF, sw + LY::KS_OFF, app_slot, lane, LPG, NG);
          else
            nv.stage(sw + LY::V_OFF, sw + LY::VS_OFF, app_slot, lane, LPG, NG);
        }
      }   // a timeout is flagged by the loop's own wait on this stage
    } else {
      page = page_direct(last);
    }
    if (page >= 0) {
      const size_t row = row_index(p, page, kvh, app_slot);
      if (app_k)
        nk.store((void*)p.k, (uint16_t*)p.ks, row, lane, LPG, NG);
      else
        nv.store((void*)p.v, (uint16_t*)p.vs, row, lane, LPG, NG);
      if (last >= LY::NS) ptx::fence_proxy_async_global();   // visible to that copy
    }
    ptx::named_barrier_sync(1, 64);   // both rows in place before either warp reads them
  }

  // ---------------------------------------------------------------- consumers
  float o[MTILES][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  int vexp[NG];      // per V group: 2^vexp > every V scale this warp has seen
  float cap[NG], sh[NG];   // 2^vexp and 2^(kPShift - weight_shift - vexp); kCap0 and 0 before
                           // the first scale
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    vexp[g] = INT_MIN;
    cap[g] = kCap0;
    sh[g] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < MTILES; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  {
    for (int i = 0; i < n_pg; ++i) {
      const int st = i % LY::NS;
      if (!ptx::mbar_wait(&full[st], (i / LY::NS) & 1, max_polls)) {
        flag_error(p.err, INT8KV_DEVERR_TIMEOUT);
        break;
      }
      if (LY::DEFER && i == 0 && !appends && threadIdx.x == 0) {   // the rest of the first NS pages
#pragma unroll
        for (int k = 1; k < LY::NS; ++k)
          if (k < n_pg) {
            const int pg = stage_page[k];
            issue_page<D, KI8, VI8, VQ4, KQ4>(smem, full, stage_page, k, pg, page_row(pg), p, kvh, &tmk,
                                    &tmv, a.expire_polls != 0);
          }
      }
      const int page = stage_page[st];
      const int tile0 = (p_first + i) * kPage + warp * 16;   // position of the tile's token 0
      if (page >= 0 && tile0 < j1 && tile0 + 16 > j0) {
        const unsigned char* sb = smem + st * LY::STAGE;
        // a tile that ends by the first query's position needs no per-column test
        if (tile0 >= j0 && tile0 + 16 <= j1 && (!WIN || tile0 + 16 <= s_q0[warp] + 1)) {
          decode_tile<D, KI8, VI8, NG, true, VQ4, KQ4>(sb, warp, lane, tile0, j0, j1, qf, qfrag,
              a.scale_log2, o,
                                             m0, m1, l0, l1, cap, sh, vexp, 0, 0);
        } else if constexpr (!WIN) {
          decode_tile<D, KI8, VI8, NG, false, VQ4, KQ4>(sb, warp, lane, tile0, j0, j1, qf, qfrag,
              a.scale_log2, o,
                                              m0, m1, l0, l1, cap, sh, vexp, INT_MAX, INT_MAX);
        } else {
          // causal limits of the lane's columns 2t, 2t + 1 (a dead column: L - 1)
          const int q0 = s_q0[warp], c0 = 2 * (lane & 3), nc = ncol();
          auto lim = [&](int c) {
            return c < nc ? q0 + (column_group(p.Hkv) * 8 + c) / G : q0 + a.q_len - 1;
          };
          decode_tile<D, KI8, VI8, NG, false, VQ4, KQ4>(sb, warp, lane, tile0, j0, j1, qf, qfrag,
              a.scale_log2, o,
                                              m0, m1, l0, l1, cap, sh, vexp, lim(c0), lim(c0 + 1));
        }
      }
      __syncwarp();   // every lane of this warp is done reading stage st
      if (lane == 0) {
        // Tickets only grow: the last warp of every round of four refills.  The
        // stage's reads have all returned (their values are consumed) before the
        // release, so the copy that overwrites it needs no proxy fence.
        if ((ptx::atom_add_acq_rel_shared(&s_rel[st], 1) & (kConsumerWarps - 1)) ==
            kConsumerWarps - 1) {
          if (i + LY::NS < n_pg) {
            const int page = page_of(i + LY::NS);
            issue_page<D, KI8, VI8, VQ4, KQ4>(smem, full, stage_page, st, page, page_row(page), p, kvh,
                                    &tmk, &tmv, a.expire_polls != 0);
          }
        }
      }
      __syncwarp();
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 4);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 8);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 16);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 4);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 8);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 16);
  }
  __syncthreads();   // every stage consumed: the stage memory becomes the merge buffer

  constexpr int DP = LY::DP;
  auto pos = [](int d) { return (VI8 || VQ4) ? d + (d >> 5) : d; };   // place of dim d in a row
  float* s_o = reinterpret_cast<float*>(smem);                // [warp][head 8][DP]
  if (r == 0) {
    s_m[warp][2 * t] = m0;
    s_m[warp][2 * t + 1] = m1;
    s_l[warp][2 * t] = l0;
    s_l[warp][2 * t + 1] = l1;
  }
#pragma unroll
  for (int j = 0; j < MTILES; ++j) {
    const int mc = j >> 2, mt = j & 3;
    int dx, dy;
    float u;
    if constexpr (VI8) {
      dx = mc * 64 + 8 * r + 2 * mt;
      dy = dx + 1;
      const int g = (mc * 64) / gs;
      u = vexp[g] == INT_MIN ? 0.f : pow2f(vexp[g] - kPShift);
    } else if constexpr (VQ4) {   // M-tile (g, h) = j: rows r, r + 8 <-> values 32g + 4r + 2h, + 1
      dx = 32 * (j >> 1) + 4 * r + 2 * (j & 1);
      dy = dx + 1;
      u = vexp[0] == INT_MIN ? 0.f : pow2f(vexp[0] - kPShift);
    } else {
      dx = mc * 64 + mt * 16 + r;
      dy = dx + 8;
      u = pow2f(-kPShift);
    }
    float* h0 = s_o + ((size_t)warp * 8 + 2 * t) * DP;
    float* h1 = h0 + DP;
    h0[pos(dx)] = o[j][0] * u;
    h1[pos(dx)] = o[j][1] * u;
    h0[pos(dy)] = o[j][2] * u;
    h1[pos(dy)] = o[j][3] * u;
  }
  __syncthreads();
  // Per-head merge weights of the four warps: f_w = 2^(m_w - M), M the block
  // max, L = sum_w l_w f_w.
  auto merge_weights = [&](int g, float (&f)[kConsumerWarps], float& M, float& Ls) {
    M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, s_m[w][g]);
    Ls = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      f[w] = M == -INFINITY ? 0.f : ptx::ex2(s_m[w][g] - M);
      Ls = fmaf(s_l[w][g], f[w], Ls);
    }
  };

  // ---- this block's partial (M, L, O~) of its split
  if (!VQ4 && a.n_splits > kMaxCluster) {
    // many splits: the partial goes to the workspace and the combine kernel
    // (launched next, as a programmatic dependent) reduces the splits.
    // Thread: 4 consecutive dims (one 16-byte store) of heads g0, g0 + stride,
    // ..., each head's weights formed by the thread itself.
    constexpr int TPH = D / 4;                    // threads per head row
    constexpr int HSTEP = kThreads / TPH;         // heads handled in parallel
    const int d = (threadIdx.x % TPH) * 4;
    const int nc = ncol();
    for (int g = threadIdx.x / TPH; g < nc; g += HSTEP) {   // g: the column
      float f[kConsumerWarps], M, Ls;
      merge_weights(g, f, M, Ls);
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float* row = s_o + ((size_t)w * 8 + g) * DP;
        float4 x;
        if constexpr (VI8)
          x = make_float4(row[pos(d)], row[pos(d) + 1], row[pos(d) + 2], row[pos(d) + 3]);
        else
          x = *reinterpret_cast<const float4*>(row + d);
        O.x = fmaf(x.x, f[w], O.x);
        O.y = fmaf(x.y, f[w], O.y);
        O.z = fmaf(x.z, f[w], O.z);
        O.w = fmaf(x.w, f[w], O.w);
      }
      const size_t h = col_row(g);
      *reinterpret_cast<float4*>(a.ws.part_o + (h * a.n_splits + split) * D + d) = O;
      if (d == 0) a.ws.part_ml[h * a.n_splits + split] = make_float2(M, Ls);
    }
    return;
  }
  if (threadIdx.x < 8) {
    const int g = threadIdx.x;
    float f[kConsumerWarps], M, Ls;
    merge_weights(g, f, M, Ls);
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) s_f[w][g] = f[w];
    s_inv[g] = Ls;
    s_m[0][g] = M;   // warp 0's entry is no longer needed: keep the block max there
  }
  __syncthreads();
  float* cta_o = s_o + kConsumerWarps * 8 * DP;   // [8][D]
  const int nc = ncol();
  for (int e = threadIdx.x; e < nc * D; e += kThreads) {
    const int g = e / D, d = e - g * D;
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w)
      O = fmaf(s_o[((size_t)w * 8 + g) * DP + pos(d)], s_f[w][g], O);
    cta_o[g * D + d] = O;
  }
  if constexpr (VQ4) {
    // The 4-bit store's rows were rotated: rotate each column's merged row back
    // (the FWHT is its own inverse, and the combine is linear in the rows).
    // Warp w takes columns w, w + 4; a lane 8 consecutive dims.
    __syncthreads();
    for (int g = warp; g < nc; g += kConsumerWarps) {
      float x[8];
      float4* row = reinterpret_cast<float4*>(cta_o + g * D + lane * 8);
      const float4 x0 = row[0], x1 = row[1];
      x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
      x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
      fwht_row<8>(x, lane, 0.0625f);
      row[0] = make_float4(x[0], x[1], x[2], x[3]);
      row[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
    __syncthreads();
    if (a.n_splits > kMaxCluster) {   // the partial goes to the workspace; the combine follows
      for (int e = threadIdx.x; e < nc * (D / 4); e += kThreads) {
        const int g = e / (D / 4), d = (e - g * (D / 4)) * 4;
        const size_t h = col_row(g);
        *reinterpret_cast<float4*>(a.ws.part_o + (h * a.n_splits + split) * D + d) =
            *reinterpret_cast<const float4*>(cta_o + g * D + d);
        if (d == 0) a.ws.part_ml[h * a.n_splits + split] = make_float2(s_m[0][g], s_inv[g]);
      }
      return;
    }
  }

  // ---- up to 8 splits form one cluster: block `rank` combines dims
  // [rank*D/CS, (rank+1)*D/CS) over the cluster's splits, reading their partials
  // from distributed shared memory, and writes the output
  cg::cluster_group cluster = cg::this_cluster();
  const int CS = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
  cluster.sync();
  if (threadIdx.x < CS * 8) {
    const int j = threadIdx.x >> 3, g = threadIdx.x & 7;
    s_cm[j][g] = *cluster.map_shared_rank(&s_m[0][g], j);
    s_cl[j][g] = *cluster.map_shared_rank(&s_inv[g], j);
  }
  __syncthreads();
  if (threadIdx.x < 8) {
    const int g = threadIdx.x;
    float M = -INFINITY;
    for (int j = 0; j < CS; ++j) M = fmaxf(M, s_cm[j][g]);
    float Ls = 0.f;
    for (int j = 0; j < CS; ++j) {
      const float f = (M == -INFINITY || s_cl[j][g] == 0.f) ? 0.f : ptx::ex2(s_cm[j][g] - M);
      s_cm[j][g] = f;   // now the weight of block j
      Ls = fmaf(s_cl[j][g], f, Ls);
    }
    s_cL[g] = Ls;
  }
  __syncthreads();
  const int slice = (D + CS - 1) / CS, d0 = rank * slice;   // CS need not divide D
  for (int e = threadIdx.x; e < nc * slice; e += kThreads) {
    const int g = e / slice, d = d0 + (e - g * slice);
    if (d >= D) continue;
    float v[kMaxCluster];
#pragma unroll
    for (int j = 0; j < kMaxCluster; ++j)   // all remote loads in flight at once
      v[j] = j < CS ? *cluster.map_shared_rank(&cta_o[g * D + d], j) : 0.f;
    float O = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxCluster; ++j)
      if (j < CS) O = fmaf(s_cm[j][g], v[j], O);
    const size_t h = col_row(g);
    const float Ls = s_cL[g];
    a.out[h * D + d] = Ls > 0.f ? O / Ls : 0.f;
  }
  cluster.sync();   // no block leaves while others read its shared memory
}

template <int D, bool KI8, bool VI8, int NG, bool WIN, bool VQ4, bool KQ4 = false>
cudaError_t launch_typed(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                         int layer_page0, cudaStream_t stream) {
  using LY = Layout<D, KI8, VI8, VQ4, KQ4>;
  auto kern = decode_mma_kernel<D, KI8, VI8, NG, WIN, VQ4, KQ4>;
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
  cfg.gridDim = dim3(a.n_splits, a.pool.Hkv * a.n_cg, a.B);   // y: kv head + Hkv * column group
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = LY::SMEM;
  cfg.stream = stream;
  // up to 8 splits: one cluster combines them in the kernel; more: no cluster,
  // the combine kernel follows
  const int cs = a.n_splits <= kMaxCluster ? a.n_splits : 1;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cs;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a, tmk, tmv, layer_page0);
}

}  // namespace

bool decode_mma_supported(const PoolView& p, int G) {
  // group_size only shapes an int8 store (q4_0 has none)
  const bool groups_ok = (p.k4 && p.v4) || (p.gs >= 64 && p.gs % 64 == 0);
  return G <= 8 && p.ps == kPage && (p.D == 128 || p.D == 256) && groups_ok &&
         (!p.v4 || p.D == 256) &&   // the 4-bit V store: head_dim 256 (one 128-byte box a row)
         (!p.k4 || p.v4);           // a 4-bit K store comes with a 4-bit V store (q4_0)
}

template <int D, bool KI8, bool VI8, bool WIN, bool VQ4>
cudaError_t launch_ng(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                      int layer_page0, cudaStream_t stream) {
  switch (a.pool.ng) {
    case 1: return launch_typed<D, KI8, VI8, 1, WIN, VQ4>(a, tmk, tmv, layer_page0, stream);
    case 2: return launch_typed<D, KI8, VI8, 2, WIN, VQ4>(a, tmk, tmv, layer_page0, stream);
    case 4:
      if constexpr (D == 256)
        return launch_typed<D, KI8, VI8, 4, WIN, VQ4>(a, tmk, tmv, layer_page0, stream);
      return cudaErrorNotSupported;
    default: return cudaErrorNotSupported;
  }
}

template <int D, bool KI8, bool VI8, bool VQ4>
cudaError_t launch_win(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                       int layer_page0, cudaStream_t stream) {
  return a.q_len > 1 ? launch_ng<D, KI8, VI8, true, VQ4>(a, tmk, tmv, layer_page0, stream)
                     : launch_ng<D, KI8, VI8, false, VQ4>(a, tmk, tmv, layer_page0, stream);
}

cudaError_t launch_decode_mma(const DecodeArgs& a, bool k8, bool v8, const CUtensorMap& tmk,
                              const CUtensorMap& tmv, int layer_page0, cudaStream_t stream) {
  if (a.pool.k4) {   // q4_0: head_dim 256 only
    if (a.pool.D != 256 || !a.pool.v4) return cudaErrorNotSupported;
    return a.q_len > 1
               ? launch_typed<256, false, false, 1, true, true, true>(a, tmk, tmv, layer_page0, stream)
               : launch_typed<256, false, false, 1, false, true, true>(a, tmk, tmv, layer_page0, stream);
  }
  if (a.pool.D == 256) {
    if (a.pool.v4) return launch_win<256, true, false, true>(a, tmk, tmv, layer_page0, stream);
    if (k8 && v8) return launch_win<256, true, true, false>(a, tmk, tmv, layer_page0, stream);
    if (k8) return launch_win<256, true, false, false>(a, tmk, tmv, layer_page0, stream);
    return launch_win<256, false, true, false>(a, tmk, tmv, layer_page0, stream);
  }
  if (a.pool.v4) return cudaErrorNotSupported;
  if (k8 && v8) return launch_win<128, true, true, false>(a, tmk, tmv, layer_page0, stream);
  if (k8) return launch_win<128, true, false, false>(a, tmk, tmv, layer_page0, stream);
  return launch_win<128, false, true, false>(a, tmk, tmv, layer_page0, stream);
}

template <int D, bool KI8, bool VI8, int NG, bool VQ4, bool KQ4 = false>
int resident_typed() {
  using LY = Layout<D, KI8, VI8, VQ4, KQ4>;
  auto kern = decode_mma_kernel<D, KI8, VI8, NG, false, VQ4, KQ4>;
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

template <int D, bool KI8, bool VI8, bool VQ4 = false>
int resident_ng(int ng) {
  if (ng == 1) return resident_typed<D, KI8, VI8, 1, VQ4>();
  if (ng == 2) return resident_typed<D, KI8, VI8, 2, VQ4>();
  if constexpr (D == 256)
    if (ng == 4) return resident_typed<D, KI8, VI8, 4, VQ4>();
  return 0;
}

// Blocks of the tensor-core kernel for this shape that the current device keeps
// resident at once; 0 if unknown.
int decode_mma_resident_blocks(int D, bool k8, bool v8, int ng, bool v4, bool k4) {
  if (k4) return D == 256 && v4 ? resident_typed<256, false, false, 1, true, true>() : 0;
  if (D == 256) {
    if (v4) return resident_ng<256, true, false, true>(ng);
    if (k8 && v8) return resident_ng<256, true, true>(ng);
    if (k8) return resident_ng<256, true, false>(ng);
    return resident_ng<256, false, true>(ng);
  }
  if (D == 128) {
    if (k8 && v8) return resident_ng<128, true, true>(ng);
    if (k8) return resident_ng<128, true, false>(ng);
    return resident_ng<128, false, true>(ng);
  }
  return 0;
}

}  // namespace int8kv

// Internal definitions shared by the C-ABI host code and the kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "int8kv.h"

// Host-side pool descriptor (opaque in the public header).
struct int8kv_pool {
  int n_layers, n_kv_heads, head_dim, group_size, n_groups, page_size, n_pages, variant;
  bool k_int8, v_int8;
  bool k_q4, v_q4;   // K / V rotated (FWHT) and stored as Q4_0 (4-bit codes, fp16 per 32)
  void* k_store;
  void* v_store;
  uint16_t* k_scales;
  uint16_t* v_scales;
  int32_t* dev_error;
  int device;        // CUDA device the pool was created on
  int num_sms;       // its SM count (split heuristic)
  bool has_tmaps;    // TMA descriptors below are valid (shapes the tensor-core decode serves)
  int decode_kernel; // INT8KV_DECODE_*: the kernel its decode calls use (AUTO = the library's choice)
  int resident[4];   // per INT8KV_DECODE_* kernel: blocks resident at once (0 = not yet queried)
  uint32_t expire_polls;   // diagnostic wait expiry of the decode calls (0: off)
  CUtensorMap tmap_k;              // K store as [rows][head_dim], 64-row x 128-byte swizzled boxes
  CUtensorMap tmap_v;              // V store, same
};

namespace int8kv {

// The pool as the kernels see it, for one layer (pointers already offset).
struct PoolView {
  const void* k;            // K store of the layer: int8 or fp16 [n_pages][Hkv][ps][D]
  const void* v;            // V store of the layer
  const uint16_t* ks;       // K scales of the layer (fp16) [n_pages][Hkv][ps][ng], or null
  const uint16_t* vs;       // V scales of the layer, or null
  int32_t* err;             // device error word, or null
  int n_pages, Hkv, D, gs, ng, ps;
  bool k4;                  // K store: Q4_0 codes [..][D/2] bytes, scales [..][D/32] (ks)
  bool v4;                  // V store: the same (vs)
};

inline PoolView layer_view(const int8kv_pool* p, int layer) {
  PoolView v;
  const size_t rows = (size_t)p->n_pages * p->n_kv_heads * p->page_size;
  const size_t kb = p->k_int8 ? 1 : 2, vb = p->v_int8 ? 1 : 2;
  // bytes of one row and fp16 scales of one row, per store
  const size_t krow = p->k_q4 ? p->head_dim / 2 : p->head_dim * kb;
  const size_t ksrow = p->k_q4 ? p->head_dim / 32 : p->n_groups;
  const size_t vrow = p->v_q4 ? p->head_dim / 2 : p->head_dim * vb;
  const size_t vsrow = p->v_q4 ? p->head_dim / 32 : p->n_groups;
  v.k = (const char*)p->k_store + (size_t)layer * rows * krow;
  v.v = (const char*)p->v_store + (size_t)layer * rows * vrow;
  v.ks = p->k_scales ? p->k_scales + (size_t)layer * rows * ksrow : nullptr;
  v.vs = p->v_scales ? p->v_scales + (size_t)layer * rows * vsrow : nullptr;
  v.err = p->dev_error;
  v.n_pages = p->n_pages;
  v.Hkv = p->n_kv_heads;
  v.D = p->head_dim;
  v.gs = p->group_size;
  v.ng = p->n_groups;
  v.ps = p->page_size;
  v.k4 = p->k_q4;
  v.v4 = p->v_q4;
  return v;
}

// Workspace of the split-K decode: partial (m, l) and unnormalised o per
// (sequence, query head, split); every call overwrites what it reads.
struct DecodeWorkspace {
  float* part_o;      // [B][H][n_splits][D]
  float2* part_ml;    // [B][H][n_splits]
};

size_t decode_workspace_layout(int B, int H, int Hkv, int D, int n_splits,
                               DecodeWorkspace* ws, void* base);

struct DecodeArgs {
  PoolView pool;
  const uint16_t* q;        // [B][H][D] fp16
  const int32_t* seq_lens;  // [B]
  const int32_t* page_table;// [B][max_pages]
  float* out;               // [B][H][D]
  const uint16_t* k_new;    // [B][Hkv][D] fp16 token appended at seq_lens[b]-1, or null
  const uint16_t* v_new;
  DecodeWorkspace ws;
  int B, H, G, max_pages, window, n_splits;
  float scale_log2;         // softmax_scale * log2(e)
  // Queries per sequence (1: decode; > 1: a verify window, query i at position
  // seq_lens[b] - q_len + i, q and out [B][q_len][H][D]) and the blocks per
  // (sequence, kv head) that share its q_len * G (query, head) columns, eight
  // each (grid y = kv head + Hkv * column group).  Only the warp-level
  // tensor-core kernel serves q_len > 1.
  int q_len = 1, n_cg = 1;
  // Diagnostic (kv_pool_test_expire_waits): nonzero makes the warp-level kernel
  // issue no page copies, arm each stage for bytes that never arrive, and give
  // up each wait after this many polls.
  uint32_t expire_polls = 0;
  // Blocks (in launch order) that prefetch their first page to L2 before the
  // grid dependency: the first wave only (later blocks start after it has
  // resolved, and the prefetch would only lengthen their prologue).
  int pf_blocks = 0;
};


struct PrefillArgs {
  PoolView pool;
  const uint16_t* q;          // [n_new][H][D] fp16
  const int32_t* page_table;  // [max_pages] of the sequence
  float* out;                 // [n_new][H][D]
  DecodeWorkspace ws;         // partials [n_new][H][n_splits][D] when n_splits > 1
  int n_new, H, G, start, max_pages, n_splits;
  float scale_log2;           // softmax_scale * log2(e)
};

// Token i of sequence b goes to position seq_pos[b] + pos_offset + i.
cudaError_t launch_quant_append(const PoolView& pool, const uint16_t* k_new, const uint16_t* v_new,
                                int n_seqs, int n_new, const int32_t* seq_pos,
                                const int32_t* page_table, int max_pages, bool k_int8,
                                bool v_int8, cudaStream_t stream, int pos_offset = 0);

// Split count for units (sequence, kv head, column group) of at most max_ctx
// positions: the shortest chain of waves x pages per block, at most max_splits.
int decode_splits_heuristic(const int8kv_pool* pool, long long units, int max_ctx,
                            int max_splits);

// The split count a decode call with n_splits = 0 runs with: the heuristic for
// the longest context the page table holds (or the window plus one page), over
// batch x column groups x kv heads units; with max_workspace > 0, the largest
// count whose workspace fits in it competes only with smaller ones.
int decode_auto_splits(const int8kv_pool* pool, int batch, int q_len, int G, int max_pages,
                       int window, size_t max_workspace);

// The decode kernel (INT8KV_DECODE_WARP_MMA or _SIMT) that serves a
// call with G query heads per kv head on this pool.
int decode_kernel_for(const int8kv_pool* pool, int G);

// Partial kernel (the one decode_kernel_for picks) and, with n_splits > 1 where
// that kernel does not combine itself, the combine.  cudaErrorNotSupported when
// no kernel fits.
cudaError_t launch_decode(const int8kv_pool* pool, int layer, const DecodeArgs& a,
                          cudaStream_t stream);

// Prefill-chunk kernel (and, with n_splits > 1, the combine).  cudaErrorNotSupported
// when no kernel fits the shape.
cudaError_t launch_prefill(const int8kv_pool* pool, int layer, const PrefillArgs& a,
                           cudaStream_t stream);
bool prefill_supported(const int8kv_pool* pool, int G);

}  // namespace int8kv

// Host side of the C ABI declared in include/int8kv.h: argument validation,
// pool descriptors, workspace layout, split heuristic and kernel dispatch.
// Nothing here allocates device memory or synchronises (except
// kv_pool_read_device_error, which is documented to).

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <new>

#include <cuda_runtime.h>

#include "decode_common.cuh"
#include "internal.h"

using namespace int8kv;

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

bool valid_head_dim(int d) { return d == 64 || d == 128 || d == 256; }

bool valid_page_size(int ps) { return ps == 16 || ps == 32 || ps == 64 || ps == 128; }

// group_size: a power of two in [16, head_dim] dividing head_dim, and at least
// head_dim / 32 (a lane of the quantizer never straddles two groups).
bool valid_group(int d, int gs) {
  if (gs < 16 || gs > d || (gs & (gs - 1)) != 0 || d % gs != 0) return false;
  return gs >= d / 32;
}

// Stores of a variant: K int8, V int8, K 4-bit, V 4-bit; the rest are fp16.
bool variant_stores(int variant, bool* k8, bool* v8, bool* k4, bool* v4) {
  *k4 = *v4 = false;
  switch (variant) {
    case INT8KV_K8V8: *k8 = true; *v8 = true; return true;
    case INT8KV_K8V16: *k8 = true; *v8 = false; return true;
    case INT8KV_K16V8: *k8 = false; *v8 = true; return true;
    case INT8KV_K8V4: *k8 = true; *v8 = false; *v4 = true; return true;
    case INT8KV_Q4_0: *k8 = false; *v8 = false; *k4 = true; *v4 = true; return true;
    default: return false;
  }
}

bool variant_int8(int variant, bool* k8, bool* v8) {
  bool k4, v4;
  return variant_stores(variant, k8, v8, &k4, &v4);
}

int shape_status(int n_layers, int n_kv_heads, int head_dim, int group_size, int page_size,
                 int n_pages, int variant) {
  bool k8, v8;
  if (!variant_int8(variant, &k8, &v8)) return INT8KV_ERR_INVALID_ARG;
  if (n_layers <= 0 || n_kv_heads <= 0 || n_pages <= 0) return INT8KV_ERR_INVALID_ARG;
  if (!valid_head_dim(head_dim)) return INT8KV_ERR_UNSUPPORTED;
  if (!valid_page_size(page_size)) return INT8KV_ERR_UNSUPPORTED;
  if (!valid_group(head_dim, group_size)) return INT8KV_ERR_GROUP;
  return INT8KV_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_tiled_fn() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiled)f;
  }
  return fn;
}

// 2-D view [rows][head_dim] of a whole store (all layers), 64-row x 128-byte
// boxes with the 128-byte swizzle.
// A store as rows of head_dim elements, copied in boxes of 64 rows x 128 bytes
// (128-byte swizzle).  Rows of one box: a 2-D map [rows][128 B].  Rows of
// several boxes: a 3-D map (x in the box, row, box) with strides (row bytes,
// 128 B), so that one copy of the box {128 B, 64 rows, all boxes} brings a
// page's rows as consecutive 64-row boxes.
bool make_store_map(CUtensorMap* map, void* base, bool is_int8, int head_dim, size_t rows) {
  EncodeTiled enc = encode_tiled_fn();
  if (!enc) return false;
  const size_t esz = is_int8 ? 1 : 2;
  const size_t row_bytes = (size_t)head_dim * esz;
  const cuuint32_t nbox = (cuuint32_t)(row_bytes / 128);
  const CUtensorMapDataType ty = is_int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  if (nbox <= 1) {
    cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)(128 / esz), 64};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, ty, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  cuuint64_t dims[3] = {(cuuint64_t)(128 / esz), (cuuint64_t)rows, (cuuint64_t)nbox};
  cuuint64_t strides[2] = {(cuuint64_t)row_bytes, 128};
  cuuint32_t box[3] = {(cuuint32_t)(128 / esz), 64, nbox};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, ty, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace int8kv {

size_t decode_workspace_layout(int B, int H, int Hkv, int D, int n_splits, DecodeWorkspace* ws,
                               void* base) {
  (void)Hkv;
  if (n_splits <= 1) {
    if (ws) *ws = DecodeWorkspace{nullptr, nullptr};
    return 0;
  }
  const size_t o_bytes = round_up((size_t)B * H * n_splits * D * sizeof(float), 256);
  const size_t ml_bytes = round_up((size_t)B * H * n_splits * sizeof(float2), 256);
  if (ws) {
    char* p = (char*)base;
    ws->part_o = (float*)p;
    ws->part_ml = (float2*)(p + o_bytes);
  }
  return o_bytes + ml_bytes;
}

// Blocks of the pool's decode kernel resident at once on its device (queried
// once per pool and kernel).  The CUDA-core kernel is taken as three per SM.
static void query_residency(const int8kv_pool* pool, int kind) {
  int8kv_pool* mp = const_cast<int8kv_pool*>(pool);
  if (pool->resident[kind] != 0) return;
  int n = 0;
  if (kind == INT8KV_DECODE_WARP_MMA) {
    int prev = -1;
    if (cudaGetDevice(&prev) == cudaSuccess && prev != pool->device) cudaSetDevice(pool->device);
    n = decode_mma_resident_blocks(pool->head_dim, pool->k_int8, pool->v_int8, pool->n_groups,
                                   pool->v_q4, pool->k_q4);
    if (prev >= 0 && prev != pool->device) cudaSetDevice(prev);
  }
  mp->resident[kind] = n > 0 ? n : 3 * pool->num_sms;
}

int decode_splits_heuristic(const int8kv_pool* pool, long long units, int max_ctx, int max_splits) {
  const int kind = decode_kernel_for(pool, 1);
  query_residency(pool, kind);
  // units x splits blocks run in ceil(blocks / resident) waves, each as long as
  // a block's ceil(pages / splits) pages plus about one page of prologue and
  // epilogue; more than one split adds the combine (about two pages).  Take the
  // split count with the shortest chain (the smallest on a tie).
  const int ps = pool->page_size;
  const int pages = max_ctx > 0 ? (max_ctx + ps - 1) / ps : 1;
  int top = pages < kMaxSplits ? pages : kMaxSplits;
  if (max_splits < top) top = max_splits;
  const long long resident = pool->resident[kind];
  long long best = -1;
  int n = 1;
  for (int s = 1; s <= top; ++s) {
    const long long waves = (units * s + resident - 1) / resident;
    const long long cost = waves * ((pages + s - 1) / s + 1) + (s > 1 ? 2 : 0);
    if (best < 0 || cost < best) {
      best = cost;
      n = s;
    }
  }
  return n;
}

int decode_auto_splits(const int8kv_pool* pool, int batch, int q_len, int G, int max_pages,
                       int window, size_t max_workspace) {
  const int n_cg = (q_len * G + 7) / 8;   // blocks per (sequence, kv head) sharing the columns
  int ctx = max_pages * pool->page_size;
  if (window > 0 && window + pool->page_size < ctx) ctx = window + pool->page_size;
  int top = kMaxSplits;
  if (max_workspace > 0)
    while (top > 1 && decode_workspace_layout(batch * q_len, G * pool->n_kv_heads,
                                              pool->n_kv_heads, pool->head_dim, top, nullptr,
                                              nullptr) > max_workspace)
      --top;
  return decode_splits_heuristic(pool, (long long)batch * n_cg * pool->n_kv_heads, ctx, top);
}

}  // namespace int8kv

extern "C" {

const char* int8kv_status_string(int status) {
  switch (status) {
    case INT8KV_OK: return "ok";
    case INT8KV_ERR_INVALID_ARG: return "invalid argument";
    case INT8KV_ERR_NULL_PTR: return "required pointer is NULL";
    case INT8KV_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case INT8KV_ERR_GROUP: return "group_size does not fit head_dim";
    case INT8KV_ERR_CAPACITY: return "request exceeds pool or workspace capacity";
    case INT8KV_ERR_UNSUPPORTED: return "shape not supported by the kernels";
    case INT8KV_ERR_CUDA: return "CUDA runtime error";
    case INT8KV_ERR_WORKSPACE: return "workspace missing or too small";
    case INT8KV_ERR_FORMAT: return "pool image of another format version, variant or shape";
    default: return "unknown status";
  }
}

int int8kv_pool_region_bytes(int n_layers, int n_kv_heads, int head_dim, int group_size,
                             int page_size, int n_pages, int variant, int region,
                             size_t* out_bytes) {
  if (!out_bytes) return INT8KV_ERR_NULL_PTR;
  const int st = shape_status(n_layers, n_kv_heads, head_dim, group_size, page_size, n_pages,
                              variant);
  if (st != INT8KV_OK) return st;
  bool k8, v8, k4, v4;
  variant_stores(variant, &k8, &v8, &k4, &v4);
  const size_t rows = (size_t)n_layers * n_pages * n_kv_heads * page_size;
  switch (region) {
    case INT8KV_REGION_K_STORE:
      *out_bytes = k4 ? rows * head_dim / 2 : rows * head_dim * (k8 ? 1 : 2);
      break;
    case INT8KV_REGION_V_STORE:
      *out_bytes = v4 ? rows * head_dim / 2 : rows * head_dim * (v8 ? 1 : 2);
      break;
    case INT8KV_REGION_K_SCALES:
      *out_bytes = k4 ? rows * (head_dim / 32) * 2 : (k8 ? rows * (head_dim / group_size) * 2 : 0);
      break;
    case INT8KV_REGION_V_SCALES:
      *out_bytes = v4 ? rows * (head_dim / 32) * 2 : (v8 ? rows * (head_dim / group_size) * 2 : 0);
      break;
    default: return INT8KV_ERR_INVALID_ARG;
  }
  return INT8KV_OK;
}

int kv_pool_create(int8kv_pool** out, int n_layers, int n_kv_heads, int head_dim,
                   int group_size, int page_size, int n_pages, int variant, void* k_store,
                   void* v_store, void* k_scales, void* v_scales, int32_t* dev_error) {
  if (!out) return INT8KV_ERR_NULL_PTR;
  *out = nullptr;
  const int st = shape_status(n_layers, n_kv_heads, head_dim, group_size, page_size, n_pages,
                              variant);
  if (st != INT8KV_OK) return st;
  bool k8, v8, k4, v4;
  variant_stores(variant, &k8, &v8, &k4, &v4);
  if (!k_store || !v_store) return INT8KV_ERR_NULL_PTR;
  if (((k8 || k4) && !k_scales) || ((v8 || v4) && !v_scales)) return INT8KV_ERR_NULL_PTR;
  if ((!k8 && !k4 && k_scales) || (!v8 && !v4 && v_scales)) return INT8KV_ERR_INVALID_ARG;
  if (!aligned16(k_store) || !aligned16(v_store) || !aligned16(k_scales) ||
      !aligned16(v_scales))
    return INT8KV_ERR_ALIGNMENT;
  if (((uintptr_t)dev_error & 3u) != 0) return INT8KV_ERR_ALIGNMENT;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return INT8KV_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return INT8KV_ERR_CUDA;
  int8kv_pool* p = new (std::nothrow) int8kv_pool;
  if (!p) return INT8KV_ERR_CAPACITY;
  p->n_layers = n_layers;
  p->n_kv_heads = n_kv_heads;
  p->head_dim = head_dim;
  p->group_size = group_size;
  p->n_groups = head_dim / group_size;
  p->page_size = page_size;
  p->n_pages = n_pages;
  p->variant = variant;
  p->k_int8 = k8;
  p->v_int8 = v8;
  p->k_q4 = k4;
  p->v_q4 = v4;
  p->k_store = k_store;
  p->v_store = v_store;
  p->k_scales = (uint16_t*)k_scales;
  p->v_scales = (uint16_t*)v_scales;
  p->dev_error = dev_error;
  p->device = dev;
  p->num_sms = sms;
  p->has_tmaps = false;
  p->decode_kernel = INT8KV_DECODE_AUTO;
  for (int k = 0; k < 4; ++k) p->resident[k] = 0;
  p->expire_polls = 0;
  // TMA descriptors for the tensor-core kernels; a 4-bit store is mapped as
  // rows of head_dim / 2 bytes (head_dim 256 only: one 128-byte box a row)
  if (page_size == 64 && (head_dim == 128 || head_dim == 256) && (!v4 || head_dim == 256)) {
    const size_t rows = (size_t)n_layers * n_pages * n_kv_heads * page_size;
    if (rows >= (1ull << 31) ||
        !make_store_map(&p->tmap_k, k_store, k8 || k4, k4 ? head_dim / 2 : head_dim, rows) ||
        !make_store_map(&p->tmap_v, v_store, v8 || v4, v4 ? head_dim / 2 : head_dim, rows)) {
      delete p;
      return INT8KV_ERR_CUDA;
    }
    p->has_tmaps = true;
  }
  *out = p;
  return INT8KV_OK;
}

void kv_pool_destroy(int8kv_pool* pool) { delete pool; }

int kv_quant_append(const int8kv_pool* pool, int layer, const uint16_t* k_new,
                    const uint16_t* v_new, int n_seqs, int n_new, const int32_t* seq_pos,
                    const int32_t* page_table, int max_pages_per_seq, void* stream) {
  if (!pool) return INT8KV_ERR_NULL_PTR;
  if (layer < 0 || layer >= pool->n_layers || n_seqs < 0 || n_new < 0 || max_pages_per_seq <= 0)
    return INT8KV_ERR_INVALID_ARG;
  if ((long long)n_seqs * n_new == 0) return INT8KV_OK;
  if (!k_new || !v_new || !seq_pos || !page_table) return INT8KV_ERR_NULL_PTR;
  if (!aligned16(k_new) || !aligned16(v_new)) return INT8KV_ERR_ALIGNMENT;
  const cudaError_t e = launch_quant_append(layer_view(pool, layer), k_new, v_new, n_seqs, n_new,
                                            seq_pos, page_table, max_pages_per_seq, pool->k_int8,
                                            pool->v_int8, (cudaStream_t)stream);
  return e == cudaSuccess ? INT8KV_OK : INT8KV_ERR_CUDA;
}

int kv_pool_set_decode_kernel(int8kv_pool* pool, int kind) {
  if (!pool) return INT8KV_ERR_NULL_PTR;
  if (kind != INT8KV_DECODE_AUTO && kind != INT8KV_DECODE_WARP_MMA && kind != INT8KV_DECODE_SIMT)
    return INT8KV_ERR_INVALID_ARG;
  const PoolView v = layer_view(pool, 0);
  if (kind == INT8KV_DECODE_WARP_MMA && !(pool->has_tmaps && decode_mma_supported(v, 1)))
    return INT8KV_ERR_UNSUPPORTED;
  pool->decode_kernel = kind;
  return INT8KV_OK;
}

int attn_decode_n_splits(const int8kv_pool* pool, int batch, int max_ctx) {
  if (!pool) return INT8KV_ERR_NULL_PTR;
  if (batch <= 0 || max_ctx < 0) return INT8KV_ERR_INVALID_ARG;
  return decode_splits_heuristic(pool, (long long)batch * pool->n_kv_heads, max_ctx, kMaxSplits);
}

int attn_decode_workspace_bytes(int batch, int n_heads, int n_kv_heads, int head_dim,
                                int n_splits, size_t* out_bytes) {
  if (!out_bytes) return INT8KV_ERR_NULL_PTR;
  if (batch < 0 || n_heads <= 0 || n_kv_heads <= 0 || !valid_head_dim(head_dim) ||
      n_splits < 1 || n_splits > kMaxSplits)
    return INT8KV_ERR_INVALID_ARG;
  *out_bytes = decode_workspace_layout(batch, n_heads, n_kv_heads, head_dim, n_splits, nullptr,
                                       nullptr);
  return INT8KV_OK;
}

static int decode_entry(const int8kv_pool* pool, int layer, const uint16_t* q,
                        const uint16_t* k_new, const uint16_t* v_new, int batch, int q_len,
                        int n_heads, const int32_t* seq_lens, const int32_t* page_table,
                        int max_pages_per_seq, int window, float softmax_scale, int n_splits,
                        float* out, void* workspace, size_t workspace_bytes, void* stream);

int attn_decode_int8(const int8kv_pool* pool, int layer, const uint16_t* q, int batch,
                     int n_heads, const int32_t* seq_lens, const int32_t* page_table,
                     int max_pages_per_seq, int window, float softmax_scale, int n_splits,
                     float* out, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_entry(pool, layer, q, nullptr, nullptr, batch, 1, n_heads, seq_lens,
                      page_table, max_pages_per_seq, window, softmax_scale, n_splits, out,
                      workspace, workspace_bytes, stream);
}

int attn_decode_multi_int8(const int8kv_pool* pool, int layer, const uint16_t* q, int batch,
                           int q_len, int n_heads, const int32_t* seq_lens,
                           const int32_t* page_table, int max_pages_per_seq, float softmax_scale,
                           int n_splits, float* out, void* workspace, size_t workspace_bytes,
                           void* stream) {
  return decode_entry(pool, layer, q, nullptr, nullptr, batch, q_len, n_heads, seq_lens,
                      page_table, max_pages_per_seq, 0, softmax_scale, n_splits, out, workspace,
                      workspace_bytes, stream);
}

int attn_decode_append_int8(const int8kv_pool* pool, int layer, const uint16_t* q,
                            const uint16_t* k_new, const uint16_t* v_new, int batch, int n_heads,
                            const int32_t* seq_lens, const int32_t* page_table,
                            int max_pages_per_seq, int window, float softmax_scale, int n_splits,
                            float* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (batch > 0 && (!k_new || !v_new)) return INT8KV_ERR_NULL_PTR;
  if (!aligned16(k_new) || !aligned16(v_new)) return INT8KV_ERR_ALIGNMENT;
  return decode_entry(pool, layer, q, k_new, v_new, batch, 1, n_heads, seq_lens, page_table,
                      max_pages_per_seq, window, softmax_scale, n_splits, out, workspace,
                      workspace_bytes, stream);
}

static int decode_entry(const int8kv_pool* pool, int layer, const uint16_t* q,
                        const uint16_t* k_new, const uint16_t* v_new, int batch, int q_len,
                        int n_heads, const int32_t* seq_lens, const int32_t* page_table,
                        int max_pages_per_seq, int window, float softmax_scale, int n_splits,
                        float* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (!pool) return INT8KV_ERR_NULL_PTR;
  if (layer < 0 || layer >= pool->n_layers || batch < 0 || n_heads <= 0 ||
      max_pages_per_seq <= 0 || window < 0 || n_splits < 0 || n_splits > kMaxSplits ||
      q_len < 1 || q_len > kMaxQueryWindow || !std::isfinite(softmax_scale))
    return INT8KV_ERR_INVALID_ARG;
  if (n_heads % pool->n_kv_heads != 0) return INT8KV_ERR_INVALID_ARG;
  const int G = n_heads / pool->n_kv_heads;
  if (G > 8) return INT8KV_ERR_UNSUPPORTED;
  // a query window runs on the warp-level tensor-core kernel only
  if (q_len > 1 && decode_kernel_for(pool, G) != INT8KV_DECODE_WARP_MMA)
    return INT8KV_ERR_UNSUPPORTED;
  if (batch == 0) return INT8KV_OK;
  if (!q || !seq_lens || !page_table || !out) return INT8KV_ERR_NULL_PTR;
  if (!aligned16(q) || !aligned16(out)) return INT8KV_ERR_ALIGNMENT;
  const int n_cg = (q_len * G + 7) / 8;   // blocks per (sequence, kv head) sharing the columns
  if (n_splits == 0)
    n_splits = decode_auto_splits(pool, batch, q_len, G, max_pages_per_seq, window, 0);
  DecodeArgs a;
  a.q_len = q_len;
  a.n_cg = n_cg;
  const size_t need = decode_workspace_layout(batch * q_len, n_heads, pool->n_kv_heads,
                                              pool->head_dim, n_splits, &a.ws, workspace);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return INT8KV_ERR_WORKSPACE;
    if (!aligned16(workspace)) return INT8KV_ERR_ALIGNMENT;
  }
  a.pool = layer_view(pool, layer);
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.seq_lens = seq_lens;
  a.page_table = page_table;
  a.out = out;
  a.B = batch;
  a.H = n_heads;
  a.G = G;
  a.max_pages = max_pages_per_seq;
  a.window = window;
  a.n_splits = n_splits;
  const float scale = softmax_scale != 0.f ? softmax_scale : 1.0f / std::sqrt((float)pool->head_dim);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.expire_polls = pool->expire_polls;
  const cudaError_t e = launch_decode(pool, layer, a, (cudaStream_t)stream);
  if (e == cudaErrorNotSupported) return INT8KV_ERR_UNSUPPORTED;
  return e == cudaSuccess ? INT8KV_OK : INT8KV_ERR_CUDA;
}

int attn_prefill_n_splits(const int8kv_pool* pool, int n_new, int n_heads, int start_pos) {
  if (!pool) return INT8KV_ERR_NULL_PTR;
  if (n_new <= 0 || n_heads <= 0 || start_pos < 0 || n_heads % pool->n_kv_heads != 0)
    return INT8KV_ERR_INVALID_ARG;
  const int G = n_heads / pool->n_kv_heads;
  if (G > 8) return INT8KV_ERR_UNSUPPORTED;
  // One block per SM at a time: (query tiles of 128 rows) x kv heads x splits
  // blocks run in ceil(blocks / SMs) waves of ceil(pages / splits) pages each.
  // Take the split count with the shortest such chain, counting two pages of
  // per-block overhead (the q tile, the epilogue) per wave.
  const long long tiles = (n_new + 128 / G - 1) / (128 / G);
  const long long units = tiles * pool->n_kv_heads;
  const int pages = (start_pos + n_new + pool->page_size - 1) / pool->page_size;
  const long long sms = pool->num_sms > 0 ? pool->num_sms : 1;
  const int top = pages < kMaxSplits ? pages : kMaxSplits;
  long long best = -1;
  int n = 1;
  for (int s = 1; s <= top; ++s) {
    const long long waves = (units * s + sms - 1) / sms;
    const long long cost = waves * ((pages + s - 1) / s + 2);
    if (best < 0 || cost < best) {
      best = cost;
      n = s;
    }
  }
  return n;
}

int attn_prefill_workspace_bytes(int n_new, int n_heads, int n_kv_heads, int head_dim,
                                 int n_splits, size_t* out_bytes) {
  return attn_decode_workspace_bytes(n_new, n_heads, n_kv_heads, head_dim, n_splits, out_bytes);
}

int attn_prefill_chunk_int8(const int8kv_pool* pool, int layer, const uint16_t* q, int n_new,
                            int n_heads, int start_pos, const int32_t* page_table,
                            int max_pages_per_seq, float softmax_scale, int n_splits, float* out,
                            void* workspace, size_t workspace_bytes, void* stream) {
  if (!pool) return INT8KV_ERR_NULL_PTR;
  if (layer < 0 || layer >= pool->n_layers || n_new < 0 || n_heads <= 0 || start_pos < 0 ||
      max_pages_per_seq <= 0 || n_splits < 0 || n_splits > kMaxSplits ||
      !std::isfinite(softmax_scale) || n_heads % pool->n_kv_heads != 0)
    return INT8KV_ERR_INVALID_ARG;
  const int G = n_heads / pool->n_kv_heads;
  if (!prefill_supported(pool, G)) return INT8KV_ERR_UNSUPPORTED;
  if (n_new == 0) return INT8KV_OK;
  if ((long long)start_pos + n_new > (long long)max_pages_per_seq * pool->page_size)
    return INT8KV_ERR_CAPACITY;
  if (!q || !page_table || !out) return INT8KV_ERR_NULL_PTR;
  if (!aligned16(q) || !aligned16(out)) return INT8KV_ERR_ALIGNMENT;
  if (n_splits == 0) {
    n_splits = attn_prefill_n_splits(pool, n_new, n_heads, start_pos);
    if (n_splits < 0) return n_splits;
  }
  PrefillArgs a;
  const size_t need = decode_workspace_layout(n_new, n_heads, pool->n_kv_heads, pool->head_dim,
                                              n_splits, &a.ws, workspace);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return INT8KV_ERR_WORKSPACE;
    if (!aligned16(workspace)) return INT8KV_ERR_ALIGNMENT;
  }
  a.pool = layer_view(pool, layer);
  a.q = q;
  a.page_table = page_table;
  a.out = out;
  a.n_new = n_new;
  a.H = n_heads;
  a.G = G;
  a.start = start_pos;
  a.max_pages = max_pages_per_seq;
  a.n_splits = n_splits;
  const float scale =
      softmax_scale != 0.f ? softmax_scale : 1.0f / std::sqrt((float)pool->head_dim);
  a.scale_log2 = scale * 1.4426950408889634f;
  const cudaError_t e = launch_prefill(pool, layer, a, (cudaStream_t)stream);
  if (e == cudaErrorNotSupported) return INT8KV_ERR_UNSUPPORTED;
  return e == cudaSuccess ? INT8KV_OK : INT8KV_ERR_CUDA;
}

int kv_pool_test_expire_waits(int8kv_pool* pool, uint32_t max_polls) {
  if (!pool) return INT8KV_ERR_NULL_PTR;
  if (max_polls != 0 && decode_kernel_for(pool, 1) != INT8KV_DECODE_WARP_MMA)
    return INT8KV_ERR_UNSUPPORTED;
  pool->expire_polls = max_polls;
  return INT8KV_OK;
}

int kv_pool_read_device_error(const int8kv_pool* pool, int32_t* out, void* stream) {
  if (!pool || !out || !pool->dev_error) return INT8KV_ERR_NULL_PTR;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(out, pool->dev_error, sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return INT8KV_ERR_CUDA;
  if (cudaMemsetAsync(pool->dev_error, 0, sizeof(int32_t), s) != cudaSuccess)
    return INT8KV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return INT8KV_ERR_CUDA;
  return INT8KV_OK;
}

}  // extern "C"

namespace int8kv {

int decode_kernel_for(const int8kv_pool* pool, int G) {
  const PoolView v = layer_view(pool, 0);
  const bool mma_ok = pool->has_tmaps && decode_mma_supported(v, G);
  switch (pool->decode_kernel) {
    case INT8KV_DECODE_WARP_MMA:
      if (mma_ok) return INT8KV_DECODE_WARP_MMA;
      break;
    case INT8KV_DECODE_SIMT:
      return INT8KV_DECODE_SIMT;
    default:
      break;
  }
  if (mma_ok) return INT8KV_DECODE_WARP_MMA;
  return INT8KV_DECODE_SIMT;
}

cudaError_t launch_decode(const int8kv_pool* pool, int layer, const DecodeArgs& a_in,
                          cudaStream_t stream) {
  bool k8, v8;
  variant_int8(pool->variant, &k8, &v8);
  DecodeArgs a = a_in;
  const int kind = decode_kernel_for(pool, a.G);
  if (a.k_new && kind != INT8KV_DECODE_WARP_MMA) {
    // only the warp-level kernel fuses the append: append first, at seq_lens[b] - 1
    const cudaError_t e0 = launch_quant_append(a.pool, a.k_new, a.v_new, a.B, 1, a.seq_lens,
                                               a.page_table, a.max_pages, k8, v8, stream, -1);
    if (e0 != cudaSuccess) return e0;
    a.k_new = a.v_new = nullptr;
  }
  cudaError_t e;
  if (kind == INT8KV_DECODE_WARP_MMA) {
    // the first wave prefetches its first pages; the residency query runs once
    // per pool, outside stream capture (inside, three blocks per SM are assumed)
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (pool->resident[kind] == 0 && cudaStreamIsCapturing(stream, &cs) == cudaSuccess &&
        cs == cudaStreamCaptureStatusNone)
      query_residency(pool, kind);
    a.pf_blocks = pool->resident[kind] ? pool->resident[kind] : 3 * pool->num_sms;
    e = launch_decode_mma(a, k8, v8, pool->tmap_k, pool->tmap_v, layer * pool->n_pages, stream);
    // up to 8 splits are combined inside the kernel (one cluster)
    if (e != cudaSuccess || a.n_splits <= 8) return e;
  } else {
    e = launch_decode_simt(a, k8, v8, stream);
    if (e != cudaSuccess || a.n_splits == 1) return e;
  }
  DecodeArgs c = a;   // the combine's rows: [B][q_len][H]
  c.B = a.B * a.q_len;
  return launch_decode_combine(c, stream);
}

}  // namespace int8kv

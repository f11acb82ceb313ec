// Saved images of a pool: the used positions of each sequence, every layer,
// codes and scales together (kv_pool_image_bytes, kv_pool_save, kv_pool_load).
//
// genie-ai-runtime release v0.1.0-alpha.12, "Path F (#45) interop guard": the
// persistent-KV format v2 stored the int8 bytes without the per-head scales
// that attention needs when the cache is hydrated again, so int8 saves were
// skipped; format v3 (#67) persists the scales region too.  Release
// v0.1.0-alpha.11 ("--int8-kv triage") lists the same requirement: save/load
// must carry the scales, or refuse a cache whose int8 setting differs.  The
// alpha.10 Path F table (F3b) packs only the used tokens.  The byte layout is
// this library's own:
//
//   header (48 bytes, little-endian): "I8KV", u32 version 3, u32 variant,
//     u32 n_layers, u32 n_kv_heads, u32 head_dim, u32 group_size, u32 n_seqs,
//     u64 payload bytes, u64 0
//   lengths: int32 [n_seqs], zero-padded to a multiple of 16 bytes
//   payload: per sequence b, per layer: K store [L_b][Hkv][D], V store
//     [L_b][Hkv][D] (int8 codes or fp16 values), then for each int8 store its
//     scales [L_b][Hkv][D / group_size] fp16; each section zero-padded to 16
//     bytes.
//
// The payload is position-major, so an image does not depend on the page size
// or the physical pages it came from.  The device work is a gather (save) or a
// scatter (load) between the pool's pages and a caller-provided device staging
// copy of the image; the host copies the staging copy to or from the caller's
// host buffer on the same stream and waits for it.

#include <cstring>

#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace int8kv {
namespace {

constexpr uint32_t kImageVersion = 3;
constexpr size_t kHeaderBytes = 48;
constexpr int kChunk = 64;          // positions per block
constexpr int kThreadsImg = 256;

__host__ __device__ inline size_t pad16(size_t n) { return (n + 15) / 16 * 16; }

struct ImageShape {
  int n_layers, Hkv, D, ng;
  bool k8, v8, k4, v4;
};

ImageShape shape_of(const int8kv_pool* p) {
  return ImageShape{p->n_layers, p->n_kv_heads, p->head_dim, p->n_groups,
                    p->k_int8, p->v_int8, p->k_q4, p->v_q4};
}

// Bytes of one row (position, kv head) of each region: K store, V store, K
// scales, V scales (0: no such region).
__host__ __device__ inline void row_bytes_of(const ImageShape& s, long long (&r)[4]) {
  r[0] = s.k4 ? s.D / 2 : (long long)s.D * (s.k8 ? 1 : 2);
  r[1] = s.v4 ? s.D / 2 : (long long)s.D * (s.v8 ? 1 : 2);
  r[2] = s.k4 ? (s.D / 32) * 2 : (s.k8 ? s.ng * 2 : 0);
  r[3] = s.v4 ? (s.D / 32) * 2 : (s.v8 ? s.ng * 2 : 0);
}

// Bytes of the four sections of one (sequence, layer) with L positions.
__host__ __device__ inline void section_bytes(const ImageShape& s, long long L, long long (&b)[4]) {
  long long r[4];
  row_bytes_of(s, r);
  for (int i = 0; i < 4; ++i) b[i] = L * s.Hkv * r[i];
}

__host__ __device__ inline long long layer_bytes(const ImageShape& s, long long L) {
  long long b[4];
  section_bytes(s, L, b);
  long long n = 0;
  for (int i = 0; i < 4; ++i) n += (b[i] + 15) / 16 * 16;
  return n;
}

__host__ __device__ inline size_t head_bytes(int n_seqs) { return kHeaderBytes + pad16((size_t)n_seqs * 4); }

size_t payload_bytes(const ImageShape& s, int n_seqs, const int32_t* lens) {
  size_t n = 0;
  for (int b = 0; b < n_seqs; ++b) n += (size_t)s.n_layers * (size_t)layer_bytes(s, lens[b]);
  return n;
}

// One block: positions [chunk*64, chunk*64 + 64) of sequence blockIdx.y, layer
// blockIdx.z.  SAVE: pool -> staging; else staging -> pool.  The sequences'
// lengths are read from the staging copy's length table.
template <bool SAVE>
__global__ void __launch_bounds__(kThreadsImg) image_kernel(PoolView pv, ImageShape s,
                                                            const int32_t* page_table,
                                                            int max_pages, unsigned char* img,
                                                            int n_seqs, size_t pool_layer_rows) {
  const int b = blockIdx.y, layer = blockIdx.z;
  const int32_t* lens = reinterpret_cast<const int32_t*>(img + kHeaderBytes);
  const int L = lens[b];
  const int p0 = blockIdx.x * kChunk;
  if (p0 >= L) return;
  const int np = min(kChunk, L - p0);
  // offset of this (sequence, layer) in the payload
  long long off = (long long)head_bytes(n_seqs);
  for (int j = 0; j < b; ++j) off += (long long)s.n_layers * layer_bytes(s, lens[j]);
  off += (long long)layer * layer_bytes(s, L);
  long long sb[4];
  section_bytes(s, L, sb);
  __shared__ int s_page[kChunk];
  for (int i = threadIdx.x; i < np; i += blockDim.x) {
    const int pos = p0 + i;
    s_page[i] = lookup_page(page_table + (size_t)b * max_pages, pos / pv.ps, max_pages, pv);
  }
  __syncthreads();
  long long rb[4];
  row_bytes_of(s, rb);
  const void* region[4] = {pv.k, pv.v, pv.ks, pv.vs};   // layer 0 of each region
  long long sec = off;
  for (int q = 0; q < 4; ++q) {
    if (sb[q] == 0) continue;
    const int row_bytes = (int)rb[q];                                // bytes of one (position, head) row
    const unsigned char* base =
        (const unsigned char*)region[q] + (size_t)layer * pool_layer_rows * row_bytes;
    unsigned char* dst0 = img + sec + (long long)p0 * s.Hkv * row_bytes;
    if (row_bytes % 16 == 0) {
      const int vpr = row_bytes / 16;                               // 16-byte pieces per row
      const int n = np * s.Hkv * vpr;
      for (int e = threadIdx.x; e < n; e += blockDim.x) {
        const int v = e % vpr, r = e / vpr, h = r % s.Hkv, i = r / s.Hkv;
        const int page = s_page[i];
        if (page < 0) continue;
        const size_t prow = ((size_t)page * s.Hkv + h) * pv.ps + (p0 + i) % pv.ps;
        uint4* pp = (uint4*)(const_cast<unsigned char*>(base) + prow * row_bytes) + v;
        uint4* ip = (uint4*)(dst0 + (size_t)r * row_bytes) + v;
        if (SAVE) *ip = *pp; else *pp = *ip;
      }
    } else {
      const int epr = row_bytes / 2;                                // fp16 elements per row
      const int n = np * s.Hkv * epr;
      for (int e = threadIdx.x; e < n; e += blockDim.x) {
        const int v = e % epr, r = e / epr, h = r % s.Hkv, i = r / s.Hkv;
        const int page = s_page[i];
        if (page < 0) continue;
        const size_t prow = ((size_t)page * s.Hkv + h) * pv.ps + (p0 + i) % pv.ps;
        uint16_t* pp = (uint16_t*)(const_cast<unsigned char*>(base) + prow * row_bytes) + v;
        uint16_t* ip = (uint16_t*)(dst0 + (size_t)r * row_bytes) + v;
        if (SAVE) *ip = *pp; else *pp = *ip;
      }
    }
    sec += (sb[q] + 15) / 16 * 16;
  }
}

cudaError_t launch_image(const int8kv_pool* pool, bool save, const int32_t* page_table,
                         int max_pages, unsigned char* staging, int n_seqs, int max_len,
                         cudaStream_t stream) {
  if (max_len <= 0 || n_seqs <= 0) return cudaSuccess;
  const PoolView v = layer_view(pool, 0);
  const ImageShape s = shape_of(pool);
  const size_t rows = (size_t)pool->n_pages * pool->n_kv_heads * pool->page_size;
  const dim3 grid((max_len + kChunk - 1) / kChunk, n_seqs, pool->n_layers);
  if (save)
    image_kernel<true><<<grid, kThreadsImg, 0, stream>>>(v, s, page_table, max_pages, staging,
                                                          n_seqs, rows);
  else
    image_kernel<false><<<grid, kThreadsImg, 0, stream>>>(v, s, page_table, max_pages, staging,
                                                           n_seqs, rows);
  return cudaGetLastError();
}

void put_u32(unsigned char* p, uint32_t x) {
  for (int i = 0; i < 4; ++i) p[i] = (unsigned char)(x >> (8 * i));
}
void put_u64(unsigned char* p, uint64_t x) {
  for (int i = 0; i < 8; ++i) p[i] = (unsigned char)(x >> (8 * i));
}
uint32_t get_u32(const unsigned char* p) {
  uint32_t x = 0;
  for (int i = 0; i < 4; ++i) x |= (uint32_t)p[i] << (8 * i);
  return x;
}
uint64_t get_u64(const unsigned char* p) {
  uint64_t x = 0;
  for (int i = 0; i < 8; ++i) x |= (uint64_t)p[i] << (8 * i);
  return x;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace int8kv

using namespace int8kv;

extern "C" {

int kv_pool_image_bytes(const int8kv_pool* pool, int n_seqs, const int32_t* seq_lens,
                        size_t* out_bytes) {
  if (!pool || !out_bytes || (n_seqs > 0 && !seq_lens)) return INT8KV_ERR_NULL_PTR;
  if (n_seqs < 0) return INT8KV_ERR_INVALID_ARG;
  for (int b = 0; b < n_seqs; ++b)
    if (seq_lens[b] < 0) return INT8KV_ERR_INVALID_ARG;
  *out_bytes = head_bytes(n_seqs) + payload_bytes(shape_of(pool), n_seqs, seq_lens);
  return INT8KV_OK;
}

int kv_pool_save(const int8kv_pool* pool, int n_seqs, const int32_t* seq_lens,
                 const int32_t* page_table, int max_pages_per_seq, void* staging,
                 size_t staging_bytes, void* image, size_t image_bytes, void* stream) {
  size_t need = 0;
  const int st = kv_pool_image_bytes(pool, n_seqs, seq_lens, &need);
  if (st != INT8KV_OK) return st;
  if (!image || !staging || (n_seqs > 0 && !page_table)) return INT8KV_ERR_NULL_PTR;
  if (max_pages_per_seq <= 0) return INT8KV_ERR_INVALID_ARG;
  if (!aligned16(staging)) return INT8KV_ERR_ALIGNMENT;
  if (image_bytes < need || staging_bytes < need) return INT8KV_ERR_CAPACITY;
  int max_len = 0;
  for (int b = 0; b < n_seqs; ++b) {
    if ((long long)seq_lens[b] > (long long)max_pages_per_seq * pool->page_size)
      return INT8KV_ERR_CAPACITY;
    if (seq_lens[b] > max_len) max_len = seq_lens[b];
  }
  unsigned char* h = (unsigned char*)image;
  const size_t hb = head_bytes(n_seqs);
  std::memset(h, 0, hb);
  std::memcpy(h, "I8KV", 4);
  put_u32(h + 4, kImageVersion);
  put_u32(h + 8, (uint32_t)pool->variant);
  put_u32(h + 12, (uint32_t)pool->n_layers);
  put_u32(h + 16, (uint32_t)pool->n_kv_heads);
  put_u32(h + 20, (uint32_t)pool->head_dim);
  put_u32(h + 24, (uint32_t)pool->group_size);
  put_u32(h + 28, (uint32_t)n_seqs);
  put_u64(h + 32, (uint64_t)(need - hb));
  for (int b = 0; b < n_seqs; ++b) put_u32(h + kHeaderBytes + 4 * b, (uint32_t)seq_lens[b]);
  cudaStream_t s = (cudaStream_t)stream;
  unsigned char* d = (unsigned char*)staging;
  // the padding of every section is zero in the image: clear the payload first
  if (cudaMemcpyAsync(d, h, hb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemsetAsync(d + hb, 0, need - hb, s) != cudaSuccess)
    return INT8KV_ERR_CUDA;
  if (launch_image(pool, true, page_table, max_pages_per_seq, d, n_seqs, max_len, s) !=
      cudaSuccess)
    return INT8KV_ERR_CUDA;
  if (cudaMemcpyAsync(h + hb, d + hb, need - hb, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return INT8KV_ERR_CUDA;
  return INT8KV_OK;
}

int kv_pool_load(const int8kv_pool* pool, const void* image, size_t image_bytes, int n_seqs,
                 const int32_t* page_table, int max_pages_per_seq, void* staging,
                 size_t staging_bytes, int32_t* seq_lens, void* stream) {
  if (!pool || !image || !staging || (n_seqs > 0 && (!page_table || !seq_lens)))
    return INT8KV_ERR_NULL_PTR;
  if (n_seqs < 0 || max_pages_per_seq <= 0) return INT8KV_ERR_INVALID_ARG;
  if (!aligned16(staging)) return INT8KV_ERR_ALIGNMENT;
  const unsigned char* h = (const unsigned char*)image;
  const size_t hb = head_bytes(n_seqs);
  if (image_bytes < hb || std::memcmp(h, "I8KV", 4) != 0) return INT8KV_ERR_FORMAT;
  if (get_u32(h + 4) != kImageVersion || get_u32(h + 8) != (uint32_t)pool->variant ||
      get_u32(h + 12) != (uint32_t)pool->n_layers ||
      get_u32(h + 16) != (uint32_t)pool->n_kv_heads ||
      get_u32(h + 20) != (uint32_t)pool->head_dim ||
      get_u32(h + 24) != (uint32_t)pool->group_size || get_u32(h + 28) != (uint32_t)n_seqs)
    return INT8KV_ERR_FORMAT;
  int max_len = 0;
  for (int b = 0; b < n_seqs; ++b) {
    const int32_t L = (int32_t)get_u32(h + kHeaderBytes + 4 * b);
    if (L < 0) return INT8KV_ERR_FORMAT;
    if ((long long)L > (long long)max_pages_per_seq * pool->page_size) return INT8KV_ERR_CAPACITY;
    seq_lens[b] = L;
    if (L > max_len) max_len = L;
  }
  const size_t pay = payload_bytes(shape_of(pool), n_seqs, seq_lens);
  if (get_u64(h + 32) != (uint64_t)pay || image_bytes < hb + pay) return INT8KV_ERR_FORMAT;
  if (staging_bytes < hb + pay) return INT8KV_ERR_CAPACITY;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(staging, image, hb + pay, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return INT8KV_ERR_CUDA;
  if (launch_image(pool, false, page_table, max_pages_per_seq, (unsigned char*)staging, n_seqs,
                   max_len, s) != cudaSuccess)
    return INT8KV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return INT8KV_ERR_CUDA;
  return INT8KV_OK;
}

}  // extern "C"

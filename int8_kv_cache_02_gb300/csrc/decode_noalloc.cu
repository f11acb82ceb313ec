// attn_decode_int8_noalloc: split-K decode attention without a caller workspace.
//
// attn_decode_int8 keeps its split partials in a workspace the caller
// allocates.  Some callers cannot allocate device memory where they decode:
// code that runs while a CUDA graph is being captured under a framework that
// forbids allocation there, runtimes that reserve all device memory at start-up
// and hand out only fixed tensors, plugins whose host passes in the tensors it
// owns and nothing else, or callers whose allocator must not be re-entered from
// this point.  This entry point serves them with a fixed scratch array that
// belongs to the library: a file-scope __device__ array of kNoAllocScratchBytes
// (4 MiB), which every GPU that loads the library holds until the process
// exits.  The caller still passes q, the pool, the lengths, the page table and
// the output.
//
// The source pages have no counterpart of this call; it reuses the decode path
// of attn_decode_int8 unchanged and only supplies the workspace.

#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "decode_common.cuh"
#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;   // 4 MiB per device
constexpr int kMaxDevices = 64;

// The scratch itself.  Host code must not use this name as an address: on the
// host it is only a stand-in; the device address comes from
// cudaGetSymbolAddress, once per device, with that device current.
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on `dev` (the current device).  The first call
// per device looks it up; later calls reuse it.  The cached address assumes the
// device's primary context lives as long as the process.
int scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return INT8KV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return INT8KV_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return INT8KV_OK;
}

}  // namespace

extern "C" int attn_decode_int8_noalloc(const int8kv_pool* pool, int layer, const uint16_t* q,
                                        int batch, int n_heads, const int32_t* seq_lens,
                                        const int32_t* page_table, int max_pages_per_seq,
                                        int window, float softmax_scale, int n_splits, float* out,
                                        void* stream) {
  if (!pool) return INT8KV_ERR_NULL_PTR;
  if (batch < 0 || n_heads <= 0 || n_splits < 0 || n_splits > int8kv::kMaxSplits ||
      max_pages_per_seq <= 0 || window < 0 || n_heads % pool->n_kv_heads != 0)
    return INT8KV_ERR_INVALID_ARG;
  if (n_heads / pool->n_kv_heads > 8) return INT8KV_ERR_UNSUPPORTED;
  if (batch == 0) return INT8KV_OK;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return INT8KV_ERR_CUDA;
  if (dev != pool->device) return INT8KV_ERR_INVALID_ARG;   // the pool's device must be current
  // n_splits = 0: the count attn_decode_int8 would pick (same window and unit
  // count), or, when that count's partials would not fit in the scratch, the
  // best count among those that do
  if (n_splits == 0)
    n_splits = int8kv::decode_auto_splits(pool, batch, 1, n_heads / pool->n_kv_heads,
                                          max_pages_per_seq, window, kNoAllocScratchBytes);
  int8kv::DecodeWorkspace ws;
  void* base = nullptr;
  const int st = scratch_address(dev, &base);
  if (st != INT8KV_OK) return st;
  const size_t need = int8kv::decode_workspace_layout(batch, n_heads, pool->n_kv_heads,
                                                      pool->head_dim, n_splits, &ws, base);
  if (need > kNoAllocScratchBytes) return INT8KV_ERR_CAPACITY;
  // The scratch keeps whatever the previous call left; nothing in it has to
  // start at zero (every partial a call reads, the same call writes first).
  return attn_decode_int8(pool, layer, q, batch, n_heads, seq_lens, page_table,
                          max_pages_per_seq, window, softmax_scale, n_splits, out,
                          need > 0 ? base : nullptr, need > 0 ? kNoAllocScratchBytes : 0, stream);
}

"""INT8 KV cache and split-K GQA decode attention for NVIDIA GB300 (sm_103a).

The computation lives in ``libint8kv.so`` (hand-written CUDA kernels behind the
C ABI of ``include/int8kv.h``); ``binding`` marshals torch tensors into it.
Importing the package does not load the library: the first call does, and
raises if it has not been built (``int8_kv_cache_02_gb300.build.build()``).
"""

from .binding import (K8V8, K8V16, K16V8, VARIANTS, Int8KVError, KVPool,  # noqa: F401
                      attn_decode_append_int8, attn_decode_int8, attn_decode_int8_noalloc,
                      attn_decode_multi_int8,
                      attn_decode_n_splits,
                      attn_decode_workspace_bytes, attn_prefill_chunk_int8, attn_prefill_n_splits,
                      attn_prefill_workspace_bytes,
                      int8kv_pool_region_bytes, int8kv_status_string, kv_pool_create,
                      kv_pool_destroy, kv_pool_read_device_error, kv_quant_append, lib)

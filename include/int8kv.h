/*
 * int8kv.h -- C ABI of the INT8 KV cache and split-K decode attention library
 * for NVIDIA GB300 (sm_103a).
 *
 * What the library computes
 * -------------------------
 *  1. kv_quant_append: fp16 K/V rows of new tokens become int8 codes with an
 *     fp16 absmax/127 scale, one per (position, kv head) as in the genie-ai-
 *     runtime INT8 KV cache (release v0.1.0-alpha.12, "Path I series", rows
 *     I1-I2; release v0.1.0-alpha.11, "--int8-kv triage": scales are captured
 *     for all n_kv_heads rows, never dropped), or one per 64 values as in
 *     Strata pull request #2698 ("What it does", kKVG = 64).  Rounding:
 *         s = fp16_round_nearest_even(fp32(absmax) / 127.0f)
 *         c = clamp(round_half_even(fp32(x) / fp32(s)), -127, 127), c = 0 if s == 0
 *     Codes go into a paged pool; scales go into a separate region.
 *  2. attn_decode_int8: GQA decode attention over that pool, dequantizing on
 *     load (alpha.12 row I3: the scale of cached row (pos, kv_head) is read
 *     per position), split-K across the key range with an online-softmax
 *     partial per split and a per-head combine (genie-ai-runtime v1.3.0,
 *     "split-K decode attention"), with an optional sliding window (v1.3.0
 *     "Details").  Query head h uses kv head h / (n_heads / n_kv_heads).
 *  3. attn_prefill_chunk_int8: causal attention of a chunk of new queries over
 *     the same int8 cache (Strata #2698: the prompt chunk dequantizes on the
 *     fly; genie-ai-runtime v1.3.1: a fused query-tiled kernel for chunks).
 *  4. attn_decode_multi_int8: decode of a window of queries per sequence,
 *     causal within the window (Strata #2698 "What it does": the verify
 *     windows of speculative decoding go through the decode kernels).
 *
 * Store variants (Strata #2698 "What it does": k8v8, and one-store variants;
 * "Not in this PR": k8v4 with the Hadamard rotation over head_dim 256):
 *     INT8KV_K8V8  K and V int8 with scales
 *     INT8KV_K8V16 K int8 with scales, V fp16
 *     INT8KV_K16V8 K fp16, V int8 with scales
 *     INT8KV_K8V4  K int8 with scales; V rotated by the normalised fast
 *                  Walsh-Hadamard transform over head_dim (y = H v / sqrt(D),
 *                  butterflies in fp32 stage by stage, h = 1, 2, ..., D/2) and
 *                  stored as Q4_0: blocks of 32 values, d = m * (-1/8) with m
 *                  the block's first value of largest magnitude, code
 *                  min(15, floor(fl(fl(x * (1/d)) + 8.5))), stored fp16(d) and
 *                  two codes per byte: byte (D/16)*r + 2g + h of a row holds
 *                  value 32g + 4r + 2h in its low nibble and the next value in
 *                  its high nibble (r = 0..7, h = 0..1, g the 32-value block);
 *                  value (code - 8) * d.  Decode rotates its output back.  No
 *                  prefill chunk.
 *     INT8KV_Q4_0  K and V both as V of INT8KV_K8V4 (Strata #2698 "Not in this
 *                  PR": --kv q4_0): the rows of K are rotated before they are
 *                  stored, decode rotates each query the same way (scores are
 *                  unchanged, the transform being orthonormal) and the output
 *                  back.  At head_dim 256 the tensor-core decode serves it
 *                  (query windows included; a rotated query must stay within
 *                  the fp16 range, as it is fed as an fp16 hi + lo pair); at
 *                  64 and 128 the CUDA-core kernel, one query per sequence.
 *                  No prefill chunk.  group_size is validated but no store
 *                  uses it.
 *
 * Pool layout in device memory (caller-allocated; the library never
 * allocates device memory):
 *     int8 store   int8    [n_layers][n_pages][n_kv_heads][page_size][head_dim]
 *     fp16 store   fp16    [n_layers][n_pages][n_kv_heads][page_size][head_dim]
 *     4-bit store  uint8   [n_layers][n_pages][n_kv_heads][page_size][head_dim/2]
 *     scales       fp16    [n_layers][n_pages][n_kv_heads][page_size][head_dim/group_size]
 *                          (of the 4-bit store: [...][head_dim/32])
 * Position p of sequence b lives on physical page page_table[b*max_pages + p/page_size],
 * slot p % page_size.
 *
 * Conventions
 * -----------
 *  - fp16 arrays are passed as uint16_t* holding IEEE binary16 bit patterns.
 *  - "device" pointers are CUDA device (or managed) memory of the current
 *    device; "host" pointers are ordinary host memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call only enqueues work on it: no call synchronises, no
 *    call allocates, so every call can be captured in a CUDA graph.
 *  - Every function returns an int status: INT8KV_OK (0) or a negative
 *    INT8KV_ERR_* code; int8kv_status_string() names it.  Arguments are
 *    validated on the host before anything is launched; nothing falls back
 *    silently to another path.
 *  - Device-side checks (a page id outside the pool, a sequence length beyond
 *    its page-table row, a wait on an asynchronous copy that does not finish)
 *    never fault: the kernel skips the access, ORs a bit into the pool's device
 *    error word and carries on.  kv_pool_read_device_error() returns the word.
 */
#ifndef INT8KV_H
#define INT8KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define INT8KV_OK                 0
#define INT8KV_ERR_INVALID_ARG   -1  /* a size or index out of range */
#define INT8KV_ERR_NULL_PTR      -2  /* a required pointer is NULL (e.g. scales of an int8 store) */
#define INT8KV_ERR_ALIGNMENT     -3  /* a region or row is not 16-byte aligned */
#define INT8KV_ERR_GROUP         -4  /* head_dim is not a multiple of group_size, or group_size unsupported */
#define INT8KV_ERR_CAPACITY      -5  /* pages, positions or splits exceed what the pool / workspace holds */
#define INT8KV_ERR_UNSUPPORTED   -6  /* a shape the kernels are not built for (see each call) */
#define INT8KV_ERR_CUDA          -7  /* a CUDA runtime call or launch failed */
#define INT8KV_ERR_WORKSPACE     -8  /* workspace NULL or smaller than the *_workspace_bytes query */
#define INT8KV_ERR_FORMAT        -9  /* a pool image that is not format 3, or that was saved from a
                                        pool of another variant or shape */

/* Format version of the images kv_pool_save writes and kv_pool_load reads. */
#define INT8KV_IMAGE_VERSION      3

/* Bits of the device error word. */
#define INT8KV_DEVERR_PAGE_ID     1  /* page-table entry outside [0, n_pages) */
#define INT8KV_DEVERR_LENGTH      2  /* position beyond max_pages_per_seq * page_size */
#define INT8KV_DEVERR_TIMEOUT     4  /* an mbarrier wait on an async copy hit its iteration cap */

typedef enum {
  INT8KV_K8V8 = 0,
  INT8KV_K8V16 = 1,
  INT8KV_K16V8 = 2,
  INT8KV_K8V4 = 3,
  INT8KV_Q4_0 = 4
} int8kv_variant;

/* Regions of a pool, for int8kv_pool_region_bytes. */
#define INT8KV_REGION_K_STORE  0
#define INT8KV_REGION_V_STORE  1
#define INT8KV_REGION_K_SCALES 2
#define INT8KV_REGION_V_SCALES 3

/* Opaque host-side pool descriptor.  It holds the shapes and the caller's
 * device pointers; it owns no device memory. */
typedef struct int8kv_pool int8kv_pool;

/* Bytes of one region of a pool of this shape (0 for the scales of an fp16
 * store).  Writes *out_bytes.  Errors: INVALID_ARG, GROUP, NULL_PTR. */
int int8kv_pool_region_bytes(int n_layers, int n_kv_heads, int head_dim, int group_size,
                             int page_size, int n_pages, int variant, int region,
                             size_t* out_bytes);

/* Create a pool descriptor over caller-allocated device regions: codes in one
 * region, their fp16 scales in a separate one (genie-ai-runtime release
 * v0.1.0-alpha.12, "Path I series" I1: a separate scales region beside the
 * int8 pool; Strata #2698 "What it does": K and V stores that can each be int8
 * or fp16; genie-ai-runtime v1.2.1, "Bugs fixed", first item: the position
 * stride of a cached slot comes from the cache's own layout, never from the
 * query's head_dim).
 *   head_dim    64, 128 or 256
 *   group_size  values per scale: head_dim (one scale per (position, kv head))
 *               or 16/32/64/128 dividing head_dim (64 = Strata's grouping)
 *   page_size   positions per page: 16, 32, 64 or 128
 *   k_store, v_store   device, 16-byte aligned, region bytes as queried
 *   k_scales, v_scales device, 16-byte aligned; required for an int8 store,
 *                      must be NULL for an fp16 store
 *   dev_error   device int32 word (4-byte aligned) for device-side checks, or
 *               NULL to disable reporting (the checks still skip bad accesses)
 * On success *out receives a descriptor to free with kv_pool_destroy.
 * Errors: NULL_PTR, INVALID_ARG, GROUP, ALIGNMENT, UNSUPPORTED. */
int kv_pool_create(int8kv_pool** out, int n_layers, int n_kv_heads, int head_dim,
                   int group_size, int page_size, int n_pages, int variant,
                   void* k_store, void* v_store, void* k_scales, void* v_scales,
                   int32_t* dev_error);

/* Free a descriptor (device regions stay the caller's).  NULL is ignored. */
void kv_pool_destroy(int8kv_pool* pool);

/* Quantize and append n_new tokens for each of n_seqs sequences of one layer
 * (alpha.12 "Path I series" I2; Strata #2698 "What it does").
 *   k_new, v_new  device fp16 [n_seqs][n_new][n_kv_heads][head_dim]
 *   seq_pos       device int32 [n_seqs]: position of each sequence's first new token
 *   page_table    device int32 [n_seqs][max_pages_per_seq]
 * A store that is fp16 receives the values unchanged.  Positions whose page
 * is outside the table row or the pool are skipped and flagged in the device
 * error word.  Errors: NULL_PTR, INVALID_ARG, CUDA. */
int kv_quant_append(const int8kv_pool* pool, int layer, const uint16_t* k_new,
                    const uint16_t* v_new, int n_seqs, int n_new, const int32_t* seq_pos,
                    const int32_t* page_table, int max_pages_per_seq, void* stream);

/* Decode kernels, for kv_pool_set_decode_kernel. */
#define INT8KV_DECODE_AUTO      0  /* the library's choice (the default) */
#define INT8KV_DECODE_WARP_MMA  1  /* warp-level tensor-core kernel (mma.sync): fused append,
                                      splits combined inside the kernel */
#define INT8KV_DECODE_SIMT      3  /* CUDA-core kernel: any shape the pool takes; a combine
                                      kernel reduces its splits */

/* Choose the kernel that serves this pool's decode calls (attn_decode_int8,
 * attn_decode_append_int8, attn_decode_n_splits).  Both kernels compute the same
 * result within the attention tolerance; the choice is for tuning and testing.
 * WARP_MMA needs page_size 64, head_dim 128 or 256 and group_size >= 64; a call
 * whose n_heads / n_kv_heads exceeds 8 uses SIMT whatever the choice.  The
 * split-K scheme both follow is genie-ai-runtime v1.3.0, "split-K decode
 * attention" (a partial per split, combined per head).
 * Errors: NULL_PTR, INVALID_ARG (unknown kind), UNSUPPORTED (the kernel does not
 * serve the pool's shape). */
int kv_pool_set_decode_kernel(int8kv_pool* pool, int kind);

/* Splits the library picks when attn_decode_int8 gets n_splits = 0, for a
 * batch of `batch` sequences of at most max_ctx positions on this pool
 * (genie-ai-runtime v1.3.0, "split-K decode attention": the key range of each
 * head is cut into n_splits pieces so that short batches fill the GPU; there
 * the count was fixed, here it is sized to the GPU).  The (sequence, kv head,
 * split) blocks run in waves of as many blocks as the pool's decode kernel
 * keeps resident on the pool's device (queried once per pool and kernel); the
 * count with the shortest chain of waves x (pages per block + 1), plus 2 when
 * the splits need combining, is returned (the smallest on a tie): at least 1,
 * at most the pages of max_ctx and 256.
 * Returns >= 1, or a negative status (NULL_PTR, INVALID_ARG). */
int attn_decode_n_splits(const int8kv_pool* pool, int batch, int max_ctx);

/* Workspace bytes attn_decode_int8 needs for this shape (0 when n_splits == 1):
 * the split partials of genie-ai-runtime v1.3.0 "split-K decode attention"
 * ((m, l, o) per split and head).  Errors: INVALID_ARG. */
int attn_decode_workspace_bytes(int batch, int n_heads, int n_kv_heads, int head_dim,
                                int n_splits, size_t* out_bytes);

/* Split-K GQA decode attention over the int8 cache of one layer
 * (genie-ai-runtime v1.3.0, "split-K decode attention" and its "Details": a
 * partial per split with its own running max and sum, combined per head; the
 * split ranges come from the length in device memory; optional sliding
 * window), dequantizing each cached row with its own scale as it is loaded
 * (release v0.1.0-alpha.12, "Path I series" I3; Strata #2698 "What it does").
 *   q            device fp16 [batch][n_heads][head_dim]
 *   seq_lens     device int32 [batch]: keys 0..L-1 of sequence b are attended
 *                (read on the device, so a captured graph can be replayed as
 *                lengths grow); L = 0 gives a zero output row
 *   page_table   device int32 [batch][max_pages_per_seq]
 *   window       0 = full context; W > 0 = only the last W positions L-W..L-1
 *   softmax_scale 0 -> 1/sqrt(head_dim)
 *   n_splits     0 -> attn_decode_n_splits() for the longest context the page
 *                table holds (or the window plus one page); 1 -> single pass;
 *                otherwise the P pages that hold the key range [lo, L) are
 *                cut into n_splits runs, split s taking pages
 *                [s*P/n_splits, (s+1)*P/n_splits) (integer division: the
 *                counts differ by at most one), clipped to [lo, L)
 *   out          device fp32 [batch][n_heads][head_dim]
 * *   workspace    device, >= attn_decode_workspace_bytes, 16-byte aligned, any
 *                contents (every partial a call reads, it writes first).  Calls
 *                sharing one workspace must not overlap on the device.
 * With the warp-level tensor-core kernel, up to 8 splits are combined inside
 * the decode kernel (the splits of a (sequence, kv head) form one thread-block
 * cluster and reduce through distributed shared memory); with more, or with the
 * CUDA-core kernel, a combine kernel follows on the stream.
 * n_heads must be a multiple of n_kv_heads with n_heads / n_kv_heads <= 8.
 * Errors: NULL_PTR, INVALID_ARG, UNSUPPORTED, WORKSPACE, CAPACITY, CUDA. */
int attn_decode_int8(const int8kv_pool* pool, int layer, const uint16_t* q, int batch,
                     int n_heads, const int32_t* seq_lens, const int32_t* page_table,
                     int max_pages_per_seq, int window, float softmax_scale, int n_splits,
                     float* out, void* workspace, size_t workspace_bytes, void* stream);

/* One decode step with its append fused: the new token's K and V rows
 *   k_new, v_new  device fp16 [batch][n_kv_heads][head_dim]
 * are quantized (as kv_quant_append does) into position seq_lens[b] - 1 of each
 * sequence, then attn_decode_int8 runs over positions 0 .. seq_lens[b] - 1.  With
 * the warp-level tensor-core kernel the block whose key range holds the new
 * position writes it before streaming its pages, so the whole step is one
 * kernel; otherwise the append kernel runs first on the same stream.  Same arguments, workspace and
 * errors as attn_decode_int8 (a length beyond the page-table row skips the
 * append and is flagged).  Bit-identical to kv_quant_append followed by
 * attn_decode_int8. */
int attn_decode_append_int8(const int8kv_pool* pool, int layer, const uint16_t* q,
                            const uint16_t* k_new, const uint16_t* v_new, int batch, int n_heads,
                            const int32_t* seq_lens, const int32_t* page_table,
                            int max_pages_per_seq, int window, float softmax_scale, int n_splits,
                            float* out, void* workspace, size_t workspace_bytes, void* stream);

/* Decode of a window of q_len queries per sequence, causal within the window:
 * the verify windows of speculative decoding (Strata pull request #2698, "What
 * it does", third bullet: the MTP block and its verify windows go through the
 * same dequantizing decode kernels).  Query i of sequence b sits at position
 * seq_lens[b] - q_len + i and attends keys 0 .. seq_lens[b] - q_len + i of the
 * pool: append the window's K/V with kv_quant_append first.
 *   q            device fp16 [batch][q_len][n_heads][head_dim]
 *   out          device fp32 [batch][q_len][n_heads][head_dim]; a query at a
 *                negative position gets a zero row
 *   q_len        1 .. 64 (1 is attn_decode_int8 without a window)
 *   workspace    >= attn_decode_workspace_bytes(batch * q_len, n_heads, ...,
 *                n_splits), 16-byte aligned, any contents
 *   n_splits     0 -> attn_decode_n_splits(pool, batch * ceil(q_len * G / 8),
 *                longest context of the page table); else as attn_decode_int8
 * The (query, head) pairs of a kv head take the 8 columns of the tensor-core
 * products, eight per block: q_len * G <= 8 reads each page once per split,
 * more reads it once per group of eight pairs.  Served by the warp-level
 * tensor-core kernel only (page_size 64, head_dim 128/256, group_size >= 64, a
 * multiple of 64); other pools return UNSUPPORTED.  No sliding window.
 * Errors: NULL_PTR, INVALID_ARG, UNSUPPORTED, WORKSPACE, ALIGNMENT, CUDA. */
int attn_decode_multi_int8(const int8kv_pool* pool, int layer, const uint16_t* q, int batch,
                           int q_len, int n_heads, const int32_t* seq_lens,
                           const int32_t* page_table, int max_pages_per_seq, float softmax_scale,
                           int n_splits, float* out, void* workspace, size_t workspace_bytes,
                           void* stream);

/* Blocks of the prefill-chunk kernel per (128-row query tile, kv head).  The
 * kernel runs one block per SM at a time, so tiles x kv heads x splits blocks
 * take ceil(blocks / SMs) waves of ceil(pages / splits) pages; the count with
 * the shortest such chain (two pages of per-block overhead added per wave) is
 * returned: at least 1, at most the pages of the context and 256.  Returns
 * >= 1, or NULL_PTR, INVALID_ARG, UNSUPPORTED. */
int attn_prefill_n_splits(const int8kv_pool* pool, int n_new, int n_heads, int start_pos);

/* Workspace bytes attn_prefill_chunk_int8 needs (0 when n_splits == 1): the
 * split partials of the chunk's (query, head) rows, combined per row as in
 * genie-ai-runtime v1.3.0 "split-K decode attention". */
int attn_prefill_workspace_bytes(int n_new, int n_heads, int n_kv_heads, int head_dim,
                                 int n_splits, size_t* out_bytes);

/* Causal attention of a chunk of n_new queries over the int8 cache of one
 * sequence (Strata #2698 "What it does": the prompt chunk dequantizes the cache
 * on the fly; genie-ai-runtime v1.3.1: fused query-tiled kernel for chunks).
 * Query i sits at position start_pos + i and attends keys 0 .. start_pos + i,
 * all read from the pool: append the chunk's own K/V with kv_quant_append
 * first.
 *   q           device fp16 [n_new][n_heads][head_dim]
 *   page_table  device int32 [max_pages_per_seq] of the sequence
 *   softmax_scale 0 -> 1/sqrt(head_dim); n_splits 0 -> attn_prefill_n_splits
 *   out         device fp32 [n_new][n_heads][head_dim]
 *   workspace   device, >= attn_prefill_workspace_bytes (any contents)
 * Built for page_size 64, head_dim 128/256, group_size >= 64 and
 * n_heads / n_kv_heads in {1, 2, 4, 8}; other shapes return UNSUPPORTED.
 * Errors: NULL_PTR, INVALID_ARG, UNSUPPORTED, CAPACITY (start_pos + n_new beyond
 * the page-table row), WORKSPACE, ALIGNMENT, CUDA. */
int attn_prefill_chunk_int8(const int8kv_pool* pool, int layer, const uint16_t* q, int n_new,
                            int n_heads, int start_pos, const int32_t* page_table,
                            int max_pages_per_seq, float softmax_scale, int n_splits,
                            float* out, void* workspace, size_t workspace_bytes, void* stream);

/* attn_decode_int8 for callers that cannot allocate device memory where they
 * decode (inside a graph-capture region of a framework that forbids
 * allocation, runtimes that reserve all device memory up front, plugins that
 * receive only the tensors their host owns).  Same arguments and result as
 * attn_decode_int8 without the workspace: the split partials live in a fixed
 * 4 MiB scratch array inside the library, which every GPU that loads the
 * library holds until the process exits.  No cudaMalloc, cudaFree or other
 * allocating call is made.
 *   - The first call on a device, with that device current, looks up the
 *     scratch's device address; make that first call before any stream
 *     capture.  The pool's device must be the current device.
 *   - Every call on a device shares the one scratch and leaves its contents
 *     there; nothing in it has to start at zero.  Calls that overlap on the GPU
 *     (other streams, other host threads) race on the scratch: serialise them.
 *   - n_splits = 0 takes the count attn_decode_int8 would pick (same window and
 *     batch); when that count's workspace would exceed the scratch, the best
 *     count among those whose workspace fits is taken instead.
 *   - An explicit n_splits whose workspace (attn_decode_workspace_bytes)
 *     exceeds 4 MiB is rejected with INT8KV_ERR_CAPACITY; lower n_splits or
 *     the batch.
 * The source pages have no counterpart of this call.
 * The cached scratch address assumes the device's primary context lives as
 * long as the process.
 * Errors: those of attn_decode_int8, and CAPACITY, INVALID_ARG (pool not on the
 * current device), CUDA. */
int attn_decode_int8_noalloc(const int8kv_pool* pool, int layer, const uint16_t* q, int batch,
                             int n_heads, const int32_t* seq_lens, const int32_t* page_table,
                             int max_pages_per_seq, int window, float softmax_scale,
                             int n_splits, float* out, void* stream);

/* ---- saved pool images ------------------------------------------------
 * The used positions 0 .. L_b - 1 of each sequence, every layer, with the int8
 * codes AND their scales (genie-ai-runtime release v0.1.0-alpha.12, "Path F
 * (#45) interop guard": the persistent-KV format v2 carried the int8 bytes
 * without the scales attention needs when the cache is hydrated again, so int8
 * saves had to be skipped; format v3 (#67) persists the scales region.
 * Release v0.1.0-alpha.11, "--int8-kv triage": save/load must persist the
 * scales, or refuse caches whose int8 setting differs.  The alpha.10 Path F
 * table, F3b: a save packs only the used tokens).  Layout (little-endian,
 * every section 16-byte aligned and zero-padded):
 *   header, 48 bytes: "I8KV", u32 version (3), u32 variant, u32 n_layers,
 *     u32 n_kv_heads, u32 head_dim, u32 group_size, u32 n_seqs,
 *     u64 payload bytes, u64 0
 *   lengths: int32 [n_seqs], padded to 16 bytes
 *   payload: per sequence, per layer: K store [L][n_kv_heads][head_dim], V
 *     store [L][n_kv_heads][head_dim] (int8 codes or fp16 values), then the
 *     scales [L][n_kv_heads][head_dim / group_size] fp16 of each int8 store.
 * The payload is position-major: an image does not depend on the page size or
 * the physical pages of the pool it came from, and loads into any pool of the
 * same variant, n_layers, n_kv_heads, head_dim and group_size. */

/* Bytes of the image of n_seqs sequences of these lengths (host int32
 * [n_seqs]).  Errors: NULL_PTR, INVALID_ARG (a negative length). */
int kv_pool_image_bytes(const int8kv_pool* pool, int n_seqs, const int32_t* seq_lens,
                        size_t* out_bytes);

/* Save the image of positions 0 .. seq_lens[b] - 1 of every layer of each
 * sequence into `image` (host memory, >= kv_pool_image_bytes).
 *   seq_lens    host int32 [n_seqs]
 *   page_table  device int32 [n_seqs][max_pages_per_seq] of the pool
 *   staging     device, 16-byte aligned, >= kv_pool_image_bytes: the image is
 *               assembled there by a gather kernel and copied to `image`
 * Waits for `stream` before returning (the image is complete).  Page-table
 * entries outside the pool are flagged in the device error word and their rows
 * left zero.  Errors: NULL_PTR, INVALID_ARG, ALIGNMENT, CAPACITY (image or
 * staging too small, a length beyond its page-table row), CUDA. */
int kv_pool_save(const int8kv_pool* pool, int n_seqs, const int32_t* seq_lens,
                 const int32_t* page_table, int max_pages_per_seq, void* staging,
                 size_t staging_bytes, void* image, size_t image_bytes, void* stream);

/* Load an image (host memory) into the pool through page_table (device int32
 * [n_seqs][max_pages_per_seq]; the pages may differ from those it was saved
 * from, and so may the page size) and write the sequences' lengths to
 * seq_lens (host int32 [n_seqs]).  staging: device, 16-byte aligned, >= the
 * image's bytes.  Waits for `stream` before returning.  An image of another
 * format version (such as one without scales), variant, n_layers, n_kv_heads,
 * head_dim, group_size or sequence count is refused with INT8KV_ERR_FORMAT and
 * nothing is written.  Errors: NULL_PTR, INVALID_ARG, ALIGNMENT, FORMAT,
 * CAPACITY (staging too small, a length beyond its page-table row), CUDA. */
int kv_pool_load(const int8kv_pool* pool, const void* image, size_t image_bytes, int n_seqs,
                 const int32_t* page_table, int max_pages_per_seq, void* staging,
                 size_t staging_bytes, int32_t* seq_lens, void* stream);

/* Diagnostic for the device-side timeout report (genie-ai-runtime release
 * v0.1.0-alpha.11, "--int8-kv triage": a path that fell back silently ended in
 * a hang; here every wait on an asynchronous copy is bounded and its expiry is
 * reported instead).  With max_polls > 0, the pool's later decode calls on the
 * warp-level tensor-core kernel issue no page copies at all and arm each stage
 * barrier for 16 bytes that never arrive, so every wait gives up after
 * max_polls polls, sets INT8KV_DEVERR_TIMEOUT in the device error word and the
 * call completes (its output is not meaningful).  No copy is in flight when a
 * block gives up.  0 restores normal operation.  Errors: NULL_PTR, UNSUPPORTED
 * (the pool's decode calls do not run on the warp-level kernel). */
int kv_pool_test_expire_waits(int8kv_pool* pool, uint32_t max_polls);

/* Copy the pool's device error word into *out (host) and clear it.  Blocks
 * until `stream` has finished.  Errors: NULL_PTR (no word given), CUDA. */
int kv_pool_read_device_error(const int8kv_pool* pool, int32_t* out, void* stream);

/* Static name of a status code. */
const char* int8kv_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* INT8KV_H */

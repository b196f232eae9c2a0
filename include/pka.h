/*
 * pka.h -- C ABI of the paged-KV attention forward library (libpka.so) for
 * NVIDIA GB300 (sm_103a).
 *
 * One serving step over a continuous batch, in the three-path form of the
 * ROCm attention-backend pages ("Beyond porting: how vLLM orchestrates
 * high-performance inference on AMD ROCm", sections "Key innovations" and
 * "Three-path processing explained"):
 *
 *   pka_cache_write          scatter the new tokens' K/V rows into cache slots
 *                            (the pages' reshape_and_cache_flush, stage 1 of
 *                            the unified backend's forward()).
 *   pka_paged_attn_forward   attention of every new token over its request's
 *                            cached + new keys, routed in three slices of a
 *                            batch ordered [decode : extend : prefill]:
 *                              decode  -> memory-bound split-KV paged kernel
 *                                         (GQA; or MLA's absorbed latent form),
 *                              prefill -> varlen causal kernel,
 *                              extend  -> new tokens over themselves (causal)
 *                                         plus the cached context in fixed
 *                                         chunks, each chunk's (output, LSE)
 *                                         combined by the LSE merge.
 *   pka_merge_attn_states    the LSE merge of two partial results.
 *
 * Conventions for every entry point
 * ---------------------------------
 * - Pointers named as device pointers must be CUDA device (or managed)
 *   memory of the current device; host pointers are not accepted.
 * - bf16 tensors are IEEE bfloat16, row-major, densely packed, and their base
 *   address must be 16-byte aligned.
 * - The caller owns every buffer. The library allocates no device memory;
 *   scratch lives in the caller's `workspace` (see pka_workspace_size).
 * - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *   legacy default stream), except pka_get_error, which synchronises it.
 * - Arguments are validated on the host before anything is launched; a
 *   rejected call launches nothing and returns the status. Metadata that
 *   lives on the device (query_start_loc, seq_lens, block_table,
 *   slot_mapping) is validated by the kernels: a violation sets a bit of the
 *   device error word (PKA_DEVERR_*), the offending work is skipped (never
 *   an out-of-bounds access, never a trap) and the outputs of that call are
 *   unspecified.
 * - Calls are re-entrant; concurrent calls on different streams need
 *   different workspaces.
 */
#ifndef PKA_H_
#define PKA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKA_API __attribute__((visibility("default")))
#else
#define PKA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKA_OK = 0,
    PKA_ERR_INVALID_ARG = 1,          /* null pointer, non-positive size, inconsistent shapes */
    PKA_ERR_UNSUPPORTED = 2,          /* a shape or head size this build has no kernel for */
    PKA_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes < pka_workspace_size(...) */
    PKA_ERR_CUDA = 4,                 /* a CUDA runtime/driver call failed */
    PKA_ERR_DEVICE_METADATA = 5       /* pka_get_error found a device error bit set */
} pka_status;

/* Bits of the device error word. */
#define PKA_DEVERR_QUERY_START_LOC 0x01 /* qsl[0] != 0, a request with no new token, or qsl[B] != num_tokens */
#define PKA_DEVERR_SEQ_LEN 0x02         /* seq_len < query_len, or seq_len > max_seq_len */
#define PKA_DEVERR_ORDER 0x04           /* batch is not [decode : extend : prefill] */
#define PKA_DEVERR_QUERY_LEN 0x08       /* a query_len > max_query_len */
#define PKA_DEVERR_BLOCK_TABLE 0x10     /* seq_len needs more than max_blocks_per_req blocks */
#define PKA_DEVERR_BLOCK_ID 0x20        /* a block id outside [0, num_blocks) */
#define PKA_DEVERR_SLOT 0x40            /* a cache slot >= num_blocks * block_size */
#define PKA_DEVERR_CAPACITY 0x80        /* the plan outgrew the workspace (inconsistent hints) */
#define PKA_DEVERR_TIMEOUT 0x100        /* a pipeline wait gave up (bounded spin); results invalid */
#define PKA_DEVERR_INDEX 0x200          /* pka_gather_rows: a row index outside [0, src_rows) */

/*
 * pka_cache_write -- write the new tokens' K and V rows into the paged cache.
 *
 * Defined by the pages' reshape_and_cache_flush ("Beyond porting", unified
 * backends, stage 1 "save key/value into the KV cache"). Row t of k/v goes to
 * slot s = slot_mapping[t]: block s / block_size, offset s % block_size:
 *     k_cache[s / bs][h][s % bs][:] = k[t][h][:]   for every kv head h
 * and likewise for v. A negative slot skips the token. The copy is bit-exact.
 *
 *   k            device, [num_tokens, num_kv_heads, head_dim] bf16
 *   v            device, [num_tokens, num_kv_heads, head_dim_v] bf16, or NULL
 *                (latent cache: only k is written; v_cache must be NULL too)
 *   slot_mapping device, [num_tokens] int64
 *   k_cache      device, [num_blocks, num_kv_heads, block_size, head_dim] bf16
 *   v_cache      device, [num_blocks, num_kv_heads, block_size, head_dim_v] bf16, or NULL
 *   error_word   device int32, or NULL. A slot >= num_blocks * block_size is
 *                skipped and, when error_word is given, PKA_DEVERR_SLOT is
 *                OR-ed into it (it is never cleared here).
 * head_dim and head_dim_v must be multiples of 8. num_tokens == 0 is a no-op.
 */
PKA_API pka_status pka_cache_write(const void *k, const void *v, const int64_t *slot_mapping,
                           int64_t num_tokens, int num_kv_heads, int head_dim, int head_dim_v,
                           void *k_cache, void *v_cache, int64_t num_blocks, int block_size,
                           int32_t *error_word, void *stream);

/*
 * pka_cache_write_fp8 -- pka_cache_write into an 8-bit cache: the pages'
 * cache write with a quantising KV-cache dtype ("Beyond porting",
 * non-absorbed recipe: the context is gathered from the cache and
 * dequantised, gather_and_maybe_dequant_cache). Every element is stored as
 * an FP8 E4M3 code ("fn" variant: bit 7 sign, 4 exponent bits with bias 7, 3
 * mantissa bits, no infinities, 0x7F/0xFF = NaN, largest finite 448) of one
 * tensor-wide scale per cache:
 *     k_cache[s / bs][h][s % bs][i] = E4M3(k[t][h][i] / k_scale)
 * and likewise v with v_scale. The quotient is formed in float32 (IEEE
 * round to nearest) and rounded to the nearest code, ties to the even code;
 * finite quotients beyond +-448 saturate to +-448. Same arguments, layouts,
 * slot rules and error behaviour as pka_cache_write, except:
 *   k_cache, v_cache  device, [num_blocks, num_kv_heads, block_size, head_dim(_v)]
 *                     uint8 codes, 16-byte aligned; both required (no latent cache)
 *   k_scale, v_scale  finite and > 0, else PKA_ERR_INVALID_ARG
 * head_dim and head_dim_v must be multiples of 8 with head_dim + head_dim_v <= 1024.
 */
PKA_API pka_status pka_cache_write_fp8(const void *k, const void *v, const int64_t *slot_mapping,
                                       int64_t num_tokens, int num_kv_heads, int head_dim, int head_dim_v,
                                       void *k_cache, void *v_cache, int64_t num_blocks, int block_size,
                                       float k_scale, float v_scale, int32_t *error_word, void *stream);

/*
 * pka_workspace_size -- bytes of scratch pka_paged_attn_forward needs for a
 * batch described by the same host hints (see pka_paged_attn_forward). The
 * result depends on the current device's SM count. Never fails; returns 0
 * for hints it would reject.
 */
PKA_API size_t pka_workspace_size(int num_decodes, int num_extends, int num_prefills, int num_tokens,
                          int num_q_heads, int num_kv_heads, int head_dim, int head_dim_v,
                          int max_query_len, int max_seq_len, int context_chunk_tokens);

/*
 * pka_workspace_size_fp8 -- the same for pka_paged_attn_forward_fp8. With
 * extends in the batch it adds the gathered context (the extends' cached
 * positions as bf16, num_extends x ceil(max_seq_len / 128) x 128 rows per kv
 * head, K and V) and its block table. Returns 0 for hints the 8-bit forward
 * would reject.
 */
PKA_API size_t pka_workspace_size_fp8(int num_decodes, int num_extends, int num_prefills, int num_tokens,
                                      int num_q_heads, int num_kv_heads, int head_dim, int head_dim_v,
                                      int max_query_len, int max_seq_len, int context_chunk_tokens);

/*
 * pka_paged_attn_forward -- attention forward of one continuous batch.
 *
 * For new token i of request r (absolute position p = ctx_r + i, where
 * ctx_r = seq_lens[r] - query_len_r is the number of tokens cached before
 * this step) and query head h, with G = num_q_heads / num_kv_heads:
 *     s_j = scale * <q[t][h], K_r[j][h / G]>          for keys j = 0 .. p
 *     out[t][h] = sum_j softmax(s)_j * V_r[j][h / G]
 *     lse[t][h] = log(sum_j exp(s_j))                  (natural log)
 * K_r / V_r are read through block_table (key j of request r lives in block
 * block_table[r][j / block_size] at offset j % block_size). The result is
 * the same for any chunking (the pages' extend path, "each chunk yields an
 * output and an LSE ... merged in a numerically stable way").
 *
 * Batch layout (the model runner's reorder, "Key innovations" item 2): the
 * first num_decodes requests are decodes (query_len == 1), the next
 * num_extends are extends (ctx >= 1; query_len >= 2 normally, but a request
 * with one new token may be placed here too: it then runs through the
 * extend path instead of the decode kernel, which is how a caller gets the
 * single-path "unified" routing of every request with context), the last
 * num_prefills are prefills (ctx == 0). New tokens are contiguous per
 * request: request r owns rows [query_start_loc[r], query_start_loc[r+1]).
 *
 * The cache must already hold every key/value of every request, including
 * the new tokens (call pka_cache_write first). Decode reads only the cache.
 * Prefill and the extend path's new-token stage read the new tokens' K/V
 * from k_new / v_new (token-major, the pages' [num_tokens, num_heads,
 * head_dim] layout) and the extend context from the cache.
 *
 *   q               device, [num_tokens, num_q_heads, head_dim] bf16
 *   k_new, v_new    device, [num_tokens, num_kv_heads, head_dim(_v)] bf16; may be
 *                   NULL when num_extends + num_prefills == 0
 *   k_cache         device, [num_blocks, num_kv_heads, block_size, head_dim] bf16
 *   v_cache         device, [num_blocks, num_kv_heads, block_size, head_dim_v] bf16,
 *                   or NULL for the MLA latent cache (num_kv_heads == 1,
 *                   V = the first head_dim_v entries of each K row)
 *   block_table     device, [B, max_blocks_per_req] int32, B = num_decodes +
 *                   num_extends + num_prefills
 *   query_start_loc device, [B + 1] int32
 *   seq_lens        device, [B] int32 (cached + new tokens)
 *   scale           multiplies q.k (e.g. 1/sqrt(head_dim)); finite and > 0, else PKA_ERR_INVALID_ARG
 *   context_chunk_tokens  context tokens per extend chunk (the pages' ~32K
 *                   per-iteration budget), >= 16
 *   max_query_len, max_seq_len  host upper bounds of query_len and seq_len
 *                   over the batch; they size the plan and the workspace
 *   out             device, [num_tokens, num_q_heads, head_dim_v] bf16
 *   lse             device, [num_tokens, num_q_heads] float32, or NULL
 *   workspace       device scratch of >= pka_workspace_size(...) bytes,
 *                   256-byte aligned; its first 4 bytes are the device error
 *                   word, cleared at the start of every call
 *
 * Supported: (head_dim, head_dim_v) in {(64, 64), (128, 128)} for every
 * slice; (576, 512) with v_cache == NULL, num_q_heads in {16, 32, 64, 128}
 * and num_kv_heads == 1 for decode-only batches. num_q_heads / num_kv_heads
 * <= 16 for the GQA decode. block_size a power of two in [1, 128].
 */
PKA_API pka_status pka_paged_attn_forward(const void *q, const void *k_new, const void *v_new,
                                  const void *k_cache, const void *v_cache,
                                  const int32_t *block_table, int max_blocks_per_req,
                                  const int32_t *query_start_loc, const int32_t *seq_lens,
                                  int num_decodes, int num_extends, int num_prefills,
                                  int num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                                  int head_dim_v, int64_t num_blocks, int block_size, float scale,
                                  int context_chunk_tokens, int max_query_len, int max_seq_len,
                                  void *out, float *lse, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * pka_paged_attn_forward_fp8 -- pka_paged_attn_forward over an 8-bit cache
 * written by pka_cache_write_fp8 (K = k_scale x code, V = v_scale x code).
 *
 * Computes the same definition, with these K and V values for the positions
 * read from the cache ("Beyond porting", absorbed / non-absorbed recipe:
 * the new tokens' attention runs on the step's own K/V, the context chunks
 * on the cache after gather_and_maybe_dequant_cache):
 *   * a decode reads every position from the cache, its own new token
 *     included (written there by pka_cache_write_fp8 first);
 *   * an extend reads its cached positions from the cache and its new
 *     tokens' K/V from k_new / v_new (bf16); a prefill reads only k_new/v_new.
 * For positions from the cache s_j = scale * k_scale * <q[t][h], code_K[j]>
 * and their share of out is v_scale * softmax(s)_j code_V[j].
 *
 * Decode: the codes are widened inside the decode kernel's tile loads (every
 * E4M3 value is exactly an f16 value); the products run on f16 operands with
 * float32 accumulation, so q is converted to f16 once per work unit: decode
 * queries must satisfy |q| < 65504 (larger magnitudes saturate), and q
 * elements below 2^-14 in magnitude are rounded to f16's subnormal spacing.
 * Extend: the extends' cached positions are first gathered into the
 * workspace as bf16 copies of the codes' values (exact), then the bf16
 * prefill/extend kernel runs with the scales applied to the context chunks'
 * scores and outputs.
 *
 * Arguments as in pka_paged_attn_forward, with k_cache / v_cache as uint8 E4M3
 * codes in the same [num_blocks, num_kv_heads, block_size, head_dim] layout and
 * the two scales (finite, > 0). The workspace is sized by
 * pka_workspace_size_fp8. Supported: head_dim == head_dim_v == 128, v_cache
 * not NULL, num_q_heads / num_kv_heads <= 16, block_size a power of two in
 * [1, 128]; other shapes return PKA_ERR_UNSUPPORTED.
 */
PKA_API pka_status pka_paged_attn_forward_fp8(const void *q, const void *k_new, const void *v_new,
                                              const void *k_cache, const void *v_cache,
                                              const int32_t *block_table, int max_blocks_per_req,
                                              const int32_t *query_start_loc, const int32_t *seq_lens,
                                              int num_decodes, int num_extends, int num_prefills,
                                              int num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                                              int head_dim_v, int64_t num_blocks, int block_size, float scale,
                                              float k_scale, float v_scale, int context_chunk_tokens,
                                              int max_query_len, int max_seq_len, void *out, float *lse,
                                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * pka_paged_attn_step / pka_paged_attn_step_fp8 -- one whole serving step:
 * the cache write of the new tokens (pka_cache_write / pka_cache_write_fp8
 * with k_new, v_new and slot_mapping) followed by the forward pass
 * (pka_paged_attn_forward / _fp8), as the pages' unified forward() runs its
 * stage 1 "save key/value into the KV cache" before the attention ("Beyond
 * porting", unified backends). Same results as the two calls in a row; in one
 * call the planner, which reads no cache, runs while the cache write runs
 * (and waits for it before the kernels that read the cache start).
 *
 *   slot_mapping       device int64 [num_tokens], as in pka_cache_write (not NULL)
 *   k_new, v_new       required (v_new NULL with a latent cache, v_cache NULL)
 *   cache_error_word   device int32, or NULL: the cache write's error bits
 *                      (PKA_DEVERR_SLOT), or-ed in; the caller clears it
 *   k_cache, v_cache   written (the new tokens' slots), then read
 * Every other argument, the workspace (pka_workspace_size / _fp8) and the
 * supported shapes are those of the forward call; validation failures return
 * before any launch.
 */
PKA_API pka_status pka_paged_attn_step(const void *q, const void *k_new, const void *v_new,
                                       const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                       const int32_t *block_table, int max_blocks_per_req,
                                       const int32_t *query_start_loc, const int32_t *seq_lens, int num_decodes,
                                       int num_extends, int num_prefills, int num_tokens, int num_q_heads,
                                       int num_kv_heads, int head_dim, int head_dim_v, int64_t num_blocks,
                                       int block_size, float scale, int context_chunk_tokens, int max_query_len,
                                       int max_seq_len, void *out, float *lse, int32_t *cache_error_word,
                                       void *workspace, size_t workspace_bytes, void *stream);
PKA_API pka_status pka_paged_attn_step_fp8(const void *q, const void *k_new, const void *v_new,
                                           const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                           const int32_t *block_table, int max_blocks_per_req,
                                           const int32_t *query_start_loc, const int32_t *seq_lens,
                                           int num_decodes, int num_extends, int num_prefills, int num_tokens,
                                           int num_q_heads, int num_kv_heads, int head_dim, int head_dim_v,
                                           int64_t num_blocks, int block_size, float scale, float k_scale,
                                           float v_scale, int context_chunk_tokens, int max_query_len,
                                           int max_seq_len, void *out, float *lse, int32_t *cache_error_word,
                                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * pka_merge_attn_states -- combine two partial attention results over
 * disjoint key sets (the pages' merge_attn_states, extend path):
 *     m = max(la, lb), wa = exp(la - m), wb = exp(lb - m)
 *     out = (wa * a + wb * b) / (wa + wb),  out_lse = m + log(wa + wb)
 * A side whose lse is -inf contributes nothing; both -inf gives out = 0,
 * out_lse = -inf. Arithmetic is float32.
 *
 *   out, prefix_out, suffix_out  device, [num_rows, head_dim] of io_dtype
 *                                (0 = float32, 1 = bf16); out may alias an input
 *   out_lse                      device float32 [num_rows], or NULL
 *   prefix_lse, suffix_lse       device float32 [num_rows]
 * num_rows = num_tokens * num_heads; head_dim a multiple of 4 (fp32) or 8 (bf16).
 */
PKA_API pka_status pka_merge_attn_states(void *out, float *out_lse, const void *prefix_out,
                                 const float *prefix_lse, const void *suffix_out,
                                 const float *suffix_lse, int64_t num_rows, int head_dim,
                                 int io_dtype, void *stream);

/*
 * pka_get_error -- synchronise `stream` and read the device error word of a
 * workspace (or any device int32 used as cache_write's error_word).
 * Writes the word to *code_out (may be NULL) and returns PKA_OK when it is 0,
 * PKA_ERR_DEVICE_METADATA when a bit is set, PKA_ERR_CUDA on a CUDA failure.
 */
PKA_API pka_status pka_get_error(const void *workspace, int32_t *code_out, void *stream);

/*
 * pka_paged_decode_noalloc -- the split-KV GQA decode of pka_paged_attn_forward
 * for callers that cannot hand the library any scratch memory.
 *
 * The pages have no counterpart to this call; it exists for integration.
 * Some callers cannot allocate device memory when they call into the
 * library: a serving engine that reserved nearly all device memory for its
 * KV-cache pool up front (a cudaMalloc would fail or fragment the pool), or
 * a plugin host that gives its kernels no workspace and forbids allocation
 * on the hot path because cudaMalloc/cudaFree synchronise the device. This
 * entry point needs no workspace: its scratch (work lists, split partials,
 * error word) is a fixed array of PKA_NOALLOC_SCRATCH_BYTES bytes compiled
 * into the library as a static device variable, which every GPU that loads
 * the library keeps until the process exits. It allocates nothing.
 *
 * Computes exactly what pka_paged_attn_forward computes for a batch of
 * num_decodes decode requests (query_len 1 each, so num_tokens ==
 * num_decodes), with the same argument meanings, layouts and supported GQA
 * shapes ((head_dim, head_dim_v) in {(64, 64), (128, 128)}; v_cache must not
 * be NULL). The cache must already hold the new tokens (pka_cache_write).
 *
 *   error_word  device int32 or NULL; receives the call's device error word
 *               (PKA_DEVERR_*; 0 when clean) at the end of the call.
 * Returns PKA_ERR_WORKSPACE_TOO_SMALL, launching nothing, when the batch
 * needs more scratch than PKA_NOALLOC_SCRATCH_BYTES (with 32 query heads of
 * dim 128, up to about 2000 decode requests fit).
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it for the rest of the process; make that first
 * call before any stream capture. The cached address belongs to the device's
 * primary context as it was at that first call: after cudaDeviceReset (or
 * anything else that destroys that context) it is stale, so do not call this
 * entry point again in that process. Every call on a device shares the one array, which keeps the last
 * call's contents (the call clears what must start at zero), so calls whose
 * work overlaps on the GPU -- on different streams, or from different host
 * threads -- race and must be serialised by the caller.
 */
#define PKA_NOALLOC_SCRATCH_BYTES (32u << 20)
PKA_API pka_status pka_paged_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                            const int32_t *block_table, int max_blocks_per_req,
                                            const int32_t *query_start_loc, const int32_t *seq_lens,
                                            int num_decodes, int num_q_heads, int num_kv_heads,
                                            int head_dim, int64_t num_blocks, int block_size,
                                            float scale, int max_seq_len, void *out, float *lse,
                                            int32_t *error_word, void *stream);

/*
 * Kernel timing for benchmarks (not needed for normal use). While enabled,
 * every launch of the selected kernel family is bracketed by a CUDA event
 * pair recorded on the launching stream (events are created once and
 * reused; no device memory is allocated). pka_kernel_timer_read
 * synchronises those events and returns the summed device time in
 * milliseconds and the number of launches since the last reset; up to 4096
 * launches per family are kept, later ones are counted but not timed.
 * Not thread-safe with respect to concurrent forward calls.
 */
typedef enum {
    PKA_KERNEL_CACHE_WRITE = 0,
    PKA_KERNEL_PLANNER = 1,
    PKA_KERNEL_DECODE = 2,          /* GQA or MLA split-KV decode */
    PKA_KERNEL_DECODE_REDUCE = 3,
    PKA_KERNEL_PREFILL_EXTEND = 4,  /* varlen prefill + extend stages */
    PKA_KERNEL_EXTEND_REDUCE = 5,
    PKA_KERNEL_MERGE = 6,
    PKA_KERNEL_GATHER = 7,          /* pka_gather_rows */
    PKA_KERNEL_CTX_DEQUANT = 8,     /* 8-bit cache: the extends' context gather */
    PKA_KERNEL_COUNT = 9
} pka_kernel;

/* enable != 0 turns timing on for `kernel` (and resets it); 0 turns it off. */
PKA_API pka_status pka_kernel_timer(int kernel, int enable);
/* Summed duration (ms) and launch count of `kernel` since it was enabled. */
PKA_API pka_status pka_kernel_timer_read(int kernel, double *total_ms, int *launches, int *timed);

/*
 * pka_batch_order -- put a batch of requests in the order the forward pass
 * needs, [decode : extend : prefill] (the pages' batch reordering before the
 * attention backend; classification with the decode threshold 1: a request
 * with one new token is a decode, one with more new tokens and cached context
 * an extend, one without cached context a prefill). Host-only, no CUDA call.
 *
 *   num_reqs      B >= 1
 *   query_lens    [B] new tokens per request, >= 1 (host)
 *   ctx_lens      [B] cached tokens per request before this step, >= 0 (host)
 *   req_order     [B] out: req_order[i] = original index of the request at
 *                 position i; stable within each class
 *   qsl_ordered   [B+1] out: query_start_loc of the ordered batch
 *   token_src     [T] out (T = sum of query_lens; may be NULL): original
 *                 token row of ordered token row j (gather index for q, k, v)
 *   token_dst     [T] out (may be NULL): ordered token row of original token
 *                 row t (gather index that brings out/lse back)
 *   counts        [3] out: num_decodes, num_extends, num_prefills
 * Returns PKA_ERR_INVALID_ARG for B < 1, a NULL required pointer, a query
 * length < 1 or a context length < 0 (outputs untouched), else PKA_OK.
 */
PKA_API pka_status pka_batch_order(int num_reqs, const int32_t *query_lens, const int32_t *ctx_lens,
                                   int32_t *req_order, int32_t *qsl_ordered, int32_t *token_src,
                                   int32_t *token_dst, int32_t *counts);

/*
 * pka_gather_rows -- dst row i = src row index[i], for i in [0, num_rows):
 * moves token rows (q, k, v, out, lse) or request rows (seq_lens, block
 * table rows) into or out of the order of pka_batch_order. Device pointers;
 * rows are row_bytes long and packed (row i at byte offset i * row_bytes).
 * 16-byte copies when row_bytes and both pointers allow, else 4-byte, else
 * single bytes. A row whose index is outside [0, src_rows) is zero-filled
 * and, when error_word is given, PKA_DEVERR_INDEX is OR-ed into it. dst and
 * src must not overlap. Asynchronous on `stream`.
 * Returns PKA_ERR_INVALID_ARG for NULL dst/src/index, num_rows < 0,
 * src_rows < 0, row_bytes < 1 or a byte size past INT64_MAX, PKA_ERR_CUDA
 * on a launch failure.
 */
PKA_API pka_status pka_gather_rows(void *dst, const void *src, const int32_t *index, int64_t num_rows,
                                   int64_t src_rows, int64_t row_bytes, int32_t *error_word, void *stream);

/*
 * pka_selftest_wait -- the library's bounded pipeline wait (the one every
 * kernel uses between its copy, MMA and softmax roles), run on its own: one
 * warp waits on a shared-memory mbarrier. With arrive != 0 one of its threads
 * completes the barrier's phase first and the wait returns at once; with
 * arrive == 0 nothing ever arrives, so the wait gives up after limit_us
 * microseconds, records PKA_DEVERR_TIMEOUT in the run's device error word and
 * the kernel exits normally (the CUDA context stays usable). The run's error
 * word (0 or PKA_DEVERR_TIMEOUT) is written to *code_out. Synchronises
 * `stream` (NULL = legacy default stream). The run's error word is one
 * device-global int per process: calls must not overlap.
 * Returns PKA_ERR_INVALID_ARG for a NULL code_out or limit_us outside
 * [1, 2000000], PKA_ERR_CUDA on a launch or copy failure, else PKA_OK (also
 * when the wait timed out: that is reported through *code_out).
 */
PKA_API pka_status pka_selftest_wait(int arrive, uint32_t limit_us, int32_t *code_out, void *stream);

/* A static, human-readable name of a status. */
PKA_API const char *pka_status_string(pka_status status);

#ifdef __cplusplus
}
#endif

#endif /* PKA_H_ */

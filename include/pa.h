/*
 * pa.h -- C ABI of the paged-KV attention library (libpa.so) for GB300.
 *
 * The library implements the GPU hot path of one scheduler step of a
 * paged-KV serving engine, as the following pages describe it:
 *
 *  [Anatomy]  "vLLM engine anatomy" (oripoin.cn/posts/vllm-engine-anatomy)
 *  [V1arch]   "vLLM V1 engine architecture: from single process to
 *             multi-process EngineCore" (charlestar.github.io)
 *  [V0vsV1]   "vLLM V0 vs V1" (llm.rainlin.net/.../vllm-v0-v1-comparation)
 *  [Overview] "01. vLLM: a general inference engine that grew out of paged KV"
 *             (niuwancheng.cn/blog/docs/ai/inference-engines/01-vllm.html)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every buffer argument is a DEVICE pointer on the current CUDA device,
 *    allocated and owned by the caller.  The library never allocates,
 *    frees or retains a buffer between calls.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) and performs no host<->device synchronisation,
 *    except pa_get_device_error, which synchronises `stream`.
 *  - Arguments are validated on the host before any launch.  A call that
 *    returns anything other than PA_OK has launched nothing.
 *  - Index values that live in device memory (slots, block ids, sequence
 *    lengths, query offsets) are validated by the kernels themselves: an
 *    out-of-range value is never dereferenced; the kernel skips the access
 *    and records a flag that pa_get_device_error reports.
 *  - Unsupported type / shape combinations return PA_ERR_UNSUPPORTED; there
 *    is no fallback path of any kind.
 *  - The library looks up a few device addresses of its own (the device
 *    error word, the scratch of pa_attention_noalloc) once per device and
 *    keeps them for the life of the process.  cudaDeviceReset invalidates
 *    them: after a reset, make no further call in that process.
 *
 * KV-cache layout (fixed by this library; the pages do not prescribe one):
 *    k_cache, v_cache : [num_blocks][num_kv_heads][block_size][head_dim]
 *  contiguous, elements of type cache_dtype.  One (block, kv head) page of
 *  block_size x head_dim elements is contiguous (4 KiB for bf16/fp16 at
 *  head_dim 128).  Token j of a sequence lives in physical block
 *  block_table[j / block_size] at offset j % block_size ([Anatomy],
 *  "PagedAttention: paging the KV cache", Figure 2).  A slot number is
 *  block * block_size + offset.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same types as cudaStream_t / cudaEvent_t, declared without the CUDA
 * headers. */
typedef struct CUstream_st* pa_stream_t;
typedef struct CUevent_st* pa_event_t;

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1, /* bad pointer, size, alias or value: nothing ran */
  PA_ERR_UNSUPPORTED = 2, /* valid but not implemented combination          */
  PA_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed          */
  PA_ERR_DEVICE = 4       /* a kernel recorded a device-side error flag      */
} pa_status;

typedef enum {
  PA_F32 = 0,
  PA_F16 = 1,
  PA_BF16 = 2,
  PA_FP8_E4M3 = 3, /* OCP FP8 E4M3 "FN": bias 7, max 448, no inf, 0x7f NaN */
  PA_INT4 = 4,     /* cache only: int4_per_token_head (4-bit pages below)  */
  PA_NVFP4 = 5     /* cache only: NVFP4 (4-bit pages below)                */
} pa_dtype;

/*
 * 4-bit KV caches ([Overview], KV cache options table, --kv-cache-dtype:
 * nvfp4, int4_per_token_head).  k_cache and v_cache are then byte arrays of
 * [num_blocks][num_kv_heads][PA_PAGE_BYTES(dtype, head_dim)], one page per
 * (block, KV head), 16-byte aligned:
 *   - codes: 16 tokens x head_dim / 2 bytes, token by token; element 2i of a
 *     token in the low nibble of its byte i, element 2i + 1 in the high one;
 *   - then the scales: PA_INT4, 16 fp32 (one per token); PA_NVFP4, 16 x
 *     head_dim / 16 E4M3 bytes (token by token, one per 16 elements).
 * Values: PA_INT4: scale_t * code (two's complement, -8 .. 7); PA_NVFP4:
 * tensor_scale * e4m3(block scale) * e2m1(code), with the E2M1 element of
 * the OCP Microscaling specification (values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and
 * their negatives) and tensor_scale = k_scale for K, v_scale for V.
 */
#define PA_PAGE_BYTES(dtype, head_dim)                                     \
  ((dtype) == PA_INT4 ? 8 * (head_dim) + 64 : 9 * (head_dim))

/* Device-side error flags (bit mask) reported by pa_get_device_error. */
#define PA_DEV_ERR_SLOT 0x1u      /* slot >= num_blocks * block_size        */
#define PA_DEV_ERR_BLOCK_ID 0x2u  /* block id outside [0, num_blocks)       */
#define PA_DEV_ERR_METADATA 0x4u  /* seq_len / query_start_loc inconsistent */
#define PA_DEV_ERR_TIMEOUT 0x8u   /* a bounded pipeline wait ran out
                                     (pa_set_wait_limit_ns)                   */

/* The only block size supported: 16 tokens per physical block, the default
 * block size named in [Anatomy], "PagedAttention: paging the KV cache", and
 * in [Overview], "KV cache management and prefix caching". */
#define PA_BLOCK_SIZE 16

/* Human-readable name of a status code (static storage, never NULL). */
const char* pa_status_string(pa_status status);

/*
 * pa_reshape_and_cache -- write the K and V of this step's tokens into the
 * paged cache.
 *
 * Defines: every token processed by a forward pass has its key and value
 * written into the KV cache ([Anatomy], "Prefill, decode and the three
 * latency metrics"); the cache is split into fixed 16-token physical blocks
 * and a token's place is (block, offset) through the block table ([Anatomy],
 * "PagedAttention", Figure 2); an FP8 KV cache stores one byte per element
 * ([Overview], KV cache options table, --kv-cache-dtype fp8).
 *
 *   for each token t < num_tokens with slot = slot_mapping[t] >= 0,
 *   for each kv head h and d < head_dim:
 *     k_cache[slot/16][h][slot%16][d] = cvt(key  [t*key_stride   + h*head_dim + d])
 *     v_cache[slot/16][h][slot%16][d] = cvt(value[t*value_stride + h*head_dim + d])
 *
 * key, value    : device, kv_dtype (PA_F32 / PA_F16 / PA_BF16); token t's
 *                 row starts at element t*key_stride (resp. value_stride);
 *                 within a row, [num_kv_heads][head_dim] is contiguous.
 * slot_mapping  : device int64 [num_tokens]; a negative slot marks a padding
 *                 token that is not written.  A slot >= num_blocks*block_size
 *                 is skipped and flagged PA_DEV_ERR_SLOT.
 * cache_dtype   : equal to kv_dtype (the bits are copied exactly), or
 *                 PA_FP8_E4M3: the code is the E4M3 value nearest to
 *                 fl32(x / scale) (one correctly rounded fp32 division),
 *                 ties to even, saturating to +-448; scale = k_scale for K
 *                 and v_scale for V, both finite and > 0.  Or a 4-bit cache
 *                 (layout above), each (token, KV head) quantised on its own:
 *                 PA_INT4: s = fl32(max|x| / 7), code = nearest integer to
 *                 fl32(x / s) (ties to even) in [-7, 7] (s = 0: codes 0;
 *                 k_scale, v_scale unused); PA_NVFP4, per 16 elements: block
 *                 scale b = E4M3 code of fl32(fl32(max|x| / 6) / scale) as
 *                 above, r = fl32(e4m3(b) * scale), code = E2M1 value
 *                 nearest to fl32(x / r), ties to even, saturating at 6
 *                 (r = 0: codes 0); scale = k_scale / v_scale, finite, > 0.
 * Two tokens must not map to the same slot (the order of such writes is
 * unspecified).
 */
pa_status pa_reshape_and_cache(const void* key, const void* value,
                               pa_dtype kv_dtype, int64_t num_tokens,
                               int64_t key_stride, int64_t value_stride,
                               void* k_cache, void* v_cache,
                               pa_dtype cache_dtype, int64_t num_blocks,
                               int block_size, int num_kv_heads, int head_dim,
                               const int64_t* slot_mapping, float k_scale,
                               float v_scale, pa_stream_t stream);

/*
 * pa_copy_blocks -- block-granular copy-on-write.
 *
 * Defines: a shared block is read-only; a sequence that must write into a
 * block other sequences still reference gets its own copy of that block and
 * only its own block table changes ([Anatomy], "PagedAttention", the
 * "copy-on-write" item); V0's scheduler output carries the copies to make as
 * blocks_to_copy ([V0vsV1], section 2.1 and 3.1).
 *
 *   for each pair p < num_pairs: (src, dst) = block_mapping[2p], [2p+1]
 *     k_cache[dst][:][:][:] = k_cache[src][:][:][:]   (all heads, offsets)
 *     v_cache[dst][:][:][:] = v_cache[src][:][:][:]
 *
 * block_mapping : device int64 [num_pairs][2].  Every dst must be distinct
 *                 and no dst may also appear as a src (the pairs run in
 *                 parallel).  An id outside [0, num_blocks) is skipped and
 *                 flagged PA_DEV_ERR_BLOCK_ID.
 * The copy is bit-exact for every cache dtype (4-bit pages: codes and
 * scales together).
 */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, pa_dtype cache_dtype,
                         int64_t num_blocks, int block_size, int num_kv_heads,
                         int head_dim, const int64_t* block_mapping,
                         int64_t num_pairs, pa_stream_t stream);

/*
 * pa_attention_workspace_size -- bytes of device workspace pa_attention
 * needs for the given host-known sizes (work list and split-K partials).
 * The same arguments must be passed to pa_attention.  Result in *bytes.
 */
pa_status pa_attention_workspace_size(int64_t num_tokens, int num_q_heads,
                                      int num_kv_heads, int head_dim,
                                      int num_seqs, int max_query_len,
                                      int max_seq_len, size_t* bytes);

/*
 * pa_attention -- unified paged attention for one scheduler step.
 *
 * Defines: one step is a map {request: number of tokens} that mixes
 * one-token decodes with chunks of long prompts (chunked prefill)
 * ([Anatomy], "V1: unified scheduling of prefill and decode", Figure 3;
 * [V1arch], "Scheduler forms one round of work"); the model runner builds
 * the attention metadata from each request's query length, context length
 * and block table ([V0vsV1], section 3.1); generation is autoregressive, each
 * token attends to the tokens before it ([Anatomy], "Prefill, decode ...");
 * GQA has fewer KV heads than query heads ([Anatomy], Table 1); the
 * attention itself is exact softmax attention, computed tile by tile with an
 * online softmax so the score matrix is never materialised ([Anatomy],
 * "Boundaries: FlashAttention, SGLang ...").
 *
 * For request r: its query tokens are rows [query_start_loc[r],
 * query_start_loc[r+1]) of q (n_r of them) and L_r = seq_lens[r] is its
 * number of keys in the cache, THIS step's tokens included (they must have
 * been written with pa_reshape_and_cache first).  Query i of request r sits
 * at position L_r - n_r + i and sees keys 0 .. L_r - n_r + i.  Query head h
 * uses KV head h / (num_q_heads / num_kv_heads).
 *
 *   s_j = scale * <q, k_j>,   out = sum_j softmax(s)_j * v_j
 *
 * with k_j = k_scale * e4m3(k8_j) and v_j = v_scale * e4m3(v8_j) for an FP8
 * cache (k_scale, v_scale ignored otherwise).
 *
 * q, out          : device [num_tokens][num_q_heads][head_dim] of q_dtype;
 *                   out receives q_dtype values (round to nearest even).
 *                   out must not overlap q, the caches or the workspace.
 *                   Rows of tokens that belong to no request are untouched.
 * q_dtype         : PA_F32 / PA_F16 / PA_BF16.  For a non-FP8 cache it must
 *                   equal cache_dtype.
 * block_tables    : device int32 [num_seqs][max_blocks_per_seq].  Entries
 *                   past ceil(L_r / 16) are never read.
 * seq_lens        : device int32 [num_seqs], 0 <= n_r <= L_r <= max_seq_len.
 * query_start_loc : device int32 [num_seqs + 1], non-decreasing, starting at
 *                   0, query_start_loc[num_seqs] <= num_tokens, every n_r <=
 *                   max_query_len.  A request with n_r = 0 produces nothing.
 * max_query_len, max_seq_len : host upper bounds supplied by the caller (no
 *                   device read-back happens inside); violations found on
 *                   the device are flagged PA_DEV_ERR_METADATA and the
 *                   request is skipped.
 * workspace       : device, >= the size pa_attention_workspace_size returns
 *                   for the same sizes, 256-byte aligned; its contents on
 *                   entry do not matter.
 * Results are bitwise deterministic from run to run.
 *
 * Supported: head_dim 64 or 128; block_size 16; num_q_heads a multiple of
 * num_kv_heads; caches bf16/fp16 (with q of the same type), fp32 (with fp32
 * q), FP8 E4M3, INT4 or NVFP4 (with bf16 or fp16 q).  For a 4-bit cache,
 * k_j and v_j are the decoded values of the layout above (NVFP4: times
 * k_scale, v_scale).
 */
pa_status pa_attention(const void* q, pa_dtype q_dtype, const void* k_cache,
                       const void* v_cache, pa_dtype cache_dtype,
                       int64_t num_blocks, int block_size, int num_q_heads,
                       int num_kv_heads, int head_dim,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* seq_lens,
                       const int32_t* query_start_loc, int num_seqs,
                       int64_t num_tokens, int max_query_len, int max_seq_len,
                       float scale, float k_scale, float v_scale, void* out,
                       void* workspace, size_t workspace_bytes,
                       pa_stream_t stream);

/*
 * pa_attention_window -- pa_attention for a layer with sliding-window
 * attention.
 *
 * Defines: models with sliding-window attention layers, whose KV blocks
 * that fall out of the window the hybrid KV cache manager can release early
 * ([Overview], "KV cache management and prefix caching", the hybrid KV cache
 * manager paragraph).  With a window of W keys, query i of request r (at
 * position p = L_r - n_r + i) sees keys max(0, p - W + 1) .. p: its own key
 * and the W - 1 before it.
 *
 * Arguments and results as pa_attention, plus sliding_window = W >= 0
 * (negative: PA_ERR_INVALID_ARG).  W = 0 is no window, the same computation
 * as pa_attention; a window of max_seq_len keys or more cuts nothing.  The
 * workspace must hold pa_attention_window_workspace_size bytes for the same
 * sizes and window.  Block-table entries of blocks that lie wholly before
 * the first query's window (entries below (L_r - n_r - W + 1) / 16) are
 * never read: those blocks may already be released and reused.
 */
pa_status pa_attention_window(const void* q, pa_dtype q_dtype,
                              const void* k_cache, const void* v_cache,
                              pa_dtype cache_dtype, int64_t num_blocks,
                              int block_size, int num_q_heads, int num_kv_heads,
                              int head_dim, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* seq_lens,
                              const int32_t* query_start_loc, int num_seqs,
                              int64_t num_tokens, int max_query_len,
                              int max_seq_len, float scale, float k_scale,
                              float v_scale, int sliding_window, void* out,
                              void* workspace, size_t workspace_bytes,
                              pa_stream_t stream);

/*
 * pa_attention_window_workspace_size -- bytes of device workspace
 * pa_attention_window needs: pa_attention's, plus each request's block-table
 * row and key count through the window (4 bytes per block of
 * min(max_seq_len, max_query_len + W + 14) keys, and 4, per request).
 */
pa_status pa_attention_window_workspace_size(int64_t num_tokens,
                                             int num_q_heads, int num_kv_heads,
                                             int head_dim, int num_seqs,
                                             int max_query_len, int max_seq_len,
                                             int sliding_window, size_t* bytes);

/*
 * pa_attention_cascade -- pa_attention for a step whose requests all begin
 * with the same cached blocks (a shared prefix).
 *
 * Defines: with prefix caching, requests that share a prompt prefix share
 * its full blocks ([Overview], "KV cache management and prefix caching";
 * [Anatomy], the automatic prefix caching section); cascade attention
 * ([Overview], the attention-backend paragraph, which records its removal
 * from vLLM in 0.32.0) computes the shared prefix's part of the attention
 * once for all queries and merges it with each request's own part, by the
 * same rule as the split-K merge ([Anatomy], "Boundaries: FlashAttention").
 * The result is pa_attention's for the same arguments, up to the rounding
 * order of the merge.
 *
 * Arguments and results as pa_attention, plus common_prefix_blocks = N >= 0
 * (negative, or more than max_blocks_per_seq: PA_ERR_INVALID_ARG).  The
 * caller states that every request's block-table row begins with the same
 * N block ids, and that every request's queries come after those blocks'
 * keys (L_r - n_r >= 16 N).  N = 0 is the plain step.  Where the step's
 * types and shapes have a cascade path (head_dim 128, bf16 / f16 / FP8
 * E4M3 caches, a positive scale, KV heads a multiple of 4, at most 512
 * requests) the N prefix blocks are read once per KV head, for the query
 * rows of every request of at most 8 rows per KV head, on the tensor
 * cores, in up to 32 key ranges of at least 32 blocks each (a partial row
 * per range, merged in range order); elsewhere N is not used.
 *
 * The cascade is the caller's choice, and it is not always the faster one:
 * it adds the prefix tiles' start-up and a merge part per key range.
 * Measured on a GB300 (decode steps of the Llama-3.1-8B shape), with a
 * bf16 cache it beat the plain step wherever N >= 512, or N x (requests of
 * at most 8 rows) >= 8192 (e.g. 1.04x at 512 blocks x 8 requests, 2.8x at
 * 1024 x 32, 12x at 4096 x 128), and lost to it below that with few
 * requests (0.69x at 32 blocks x 2 requests); with an FP8 cache (prefix
 * pages widened on the way, the plain step reading half the bytes) wherever
 * N x requests >= 16384 (1.1x at 512 x 32, 5x at 4096 x 128), and lost below
 * that (0.79x at 1024 x 8).  With a single request nothing is shared: call
 * pa_attention.  The statement is checked on the device:
 * a request whose block-table row or key count breaks it sets
 * PA_DEV_ERR_METADATA (pa_get_device_error) and the step's output is then
 * undefined.  The workspace must hold pa_attention_cascade_workspace_size
 * bytes for the same sizes.
 */
pa_status pa_attention_cascade(const void* q, pa_dtype q_dtype,
                               const void* k_cache, const void* v_cache,
                               pa_dtype cache_dtype, int64_t num_blocks,
                               int block_size, int num_q_heads, int num_kv_heads,
                               int head_dim, const int32_t* block_tables,
                               int max_blocks_per_seq, const int32_t* seq_lens,
                               const int32_t* query_start_loc, int num_seqs,
                               int64_t num_tokens, int max_query_len,
                               int max_seq_len, float scale, float k_scale,
                               float v_scale, int common_prefix_blocks, void* out,
                               void* workspace, size_t workspace_bytes,
                               pa_stream_t stream);

/*
 * pa_attention_cascade_workspace_size -- bytes of device workspace
 * pa_attention_cascade needs: pa_attention's, plus one partial row
 * ((head_dim + 2) x 4 bytes) per token, q head and key range of the shared
 * prefix (the ranges: as many as keep the prefix tiles within one per SM,
 * at most 32, and at most one per 32 blocks of a max_seq_len - 1 key
 * prefix) and 32 per request and group of 4 KV heads for the requests' own
 * parts.
 */
pa_status pa_attention_cascade_workspace_size(int64_t num_tokens,
                                              int num_q_heads, int num_kv_heads,
                                              int head_dim, int num_seqs,
                                              int max_query_len, int max_seq_len,
                                              size_t* bytes);

/*
 * pa_set_wait_limit_ns -- the longest one pipeline wait inside the attention
 * kernels may last (no counterpart on the pages; failure detection).  A
 * kernel whose wait runs out records PA_DEV_ERR_TIMEOUT (pa_get_device_error),
 * lets the copies and tensor-core work it has in flight complete, frees its
 * tensor memory and returns: the CUDA context stays usable and the next
 * call runs normally.  ns = 0 restores the default of 2 s; otherwise 0.1 ms
 * <= ns <= 60 s (else PA_ERR_INVALID_ARG).  Applies to the current device
 * and to kernels launched after the call; it copies to device memory
 * synchronously, so it is a configuration call, not one for the step loop.
 */
pa_status pa_set_wait_limit_ns(uint64_t ns);

/*
 * pa_test_skip_copy -- testing hook for the bounded waits (no counterpart on
 * the pages).  stage >= 0: in every later launch of the pipelined attention
 * kernels (the head-group decode kernel, the tensor-core prefill kernel) on
 * the current device, CTA 0 leaves out the copy of its pipeline stage
 * number `stage` (counted from 0 per CTA), so that the waits on that stage
 * can only run out: the step then reports PA_DEV_ERR_TIMEOUT and its output
 * is undefined.  Nothing faults and nothing is left in flight.  stage = -1
 * (the default) turns the hook off.  Same device-memory copy as
 * pa_set_wait_limit_ns.
 */
pa_status pa_test_skip_copy(int64_t stage);

/*
 * pa_set_debug_bounds -- the device-side index checks of the pages' metadata
 * (block ids, slots, lengths, query offsets; see the conventions above).
 * In this library those checks are compiled into every kernel and cannot be
 * switched off: they are integer compares on values the kernels load anyway,
 * one per physical page or per request, beside 4 KiB page copies.
 * enable != 0: PA_OK (the checks are on).  enable == 0: PA_ERR_UNSUPPORTED,
 * nothing changes.
 */
pa_status pa_set_debug_bounds(int enable);

/*
 * pa_get_device_error -- synchronise `stream`, then read and clear the
 * device-side error flags of the current device (PA_DEV_ERR_* bits, 0 if
 * none) into *flags.  Returns PA_ERR_DEVICE if any flag was set, PA_OK
 * otherwise, PA_ERR_CUDA if the synchronisation itself failed.
 */
pa_status pa_get_device_error(pa_stream_t stream, uint32_t* flags);

/*
 * pa_attention_noalloc -- pa_attention without a caller-provided workspace.
 * No counterpart on the pages: it exists for callers that cannot allocate
 * device memory per step -- for instance an engine that gives all free HBM
 * to its KV-cache pool at start-up, or code that must not call cudaMalloc /
 * cudaFree because they can synchronise the device.
 *
 * Same arguments and results as pa_attention, minus the workspace.  The
 * scratch is one fixed array of PA_NOALLOC_SCRATCH_BYTES in device memory
 * that the library image carries: every GPU that loads the library holds it
 * until the process exits.  The function allocates nothing and calls no
 * allocating routine.
 *
 *  - Sizes whose workspace (pa_attention_workspace_size) exceeds
 *    PA_NOALLOC_SCRATCH_BYTES are rejected with PA_ERR_INVALID_ARG before
 *    anything runs.
 *  - The first call on a device (with that device current) looks up the
 *    array's device address (cudaGetSymbolAddress); make that first call
 *    before any stream capture.  The address is kept until the process
 *    exits; a cudaDeviceReset invalidates it.
 *  - Every decode step needs a fixed floor of split-K partial slots (about
 *    98 KiB per SM: two per resident attention CTA, up to three CTAs per
 *    SM); the scratch size is checked against that floor for up to 160 SMs
 *    when the library is compiled.
 *  - All calls share the one array, which keeps the previous call's
 *    contents (nothing in it needs to start at zero).  Calls whose work
 *    overlaps on the GPU -- on different streams, or from different host
 *    threads without ordering -- race on it: order them.
 */
#define PA_NOALLOC_SCRATCH_BYTES (20u * 1024u * 1024u)

pa_status pa_attention_noalloc(const void* q, pa_dtype q_dtype,
                               const void* k_cache, const void* v_cache,
                               pa_dtype cache_dtype, int64_t num_blocks,
                               int block_size, int num_q_heads,
                               int num_kv_heads, int head_dim,
                               const int32_t* block_tables,
                               int max_blocks_per_seq, const int32_t* seq_lens,
                               const int32_t* query_start_loc, int num_seqs,
                               int64_t num_tokens, int max_query_len,
                               int max_seq_len, float scale, float k_scale,
                               float v_scale, void* out, pa_stream_t stream);

/*
 * pa_set_profile_events -- measurement hook (no counterpart on the pages).
 * When both events are non-NULL, every later pa_attention call on this
 * thread records `start` on its stream immediately before the launch of its
 * attention kernels (the main attention kernel and, when the step has
 * prefill tiles for it, the tensor-core prefill kernel, in the order the
 * step runs them) and `stop` immediately after them, so that
 * cudaEventElapsedTime gives their device time alone (the planning and
 * split-merge launches are outside the pair).  While the events are on,
 * these launches run one after the other: a step that would otherwise run
 * part of its prefill tiles beside the decode kernel runs them all behind it.
 * NULL, NULL turns it off.  The events are owned by the caller and must
 * outlive the calls.
 */
pa_status pa_set_profile_events(pa_event_t start, pa_event_t stop);

/*
 * pa_launch_count -- measurement aid (no counterpart on the pages): the
 * number of kernels this library has launched from the calling host thread
 * since it was loaded, through every entry point (launches captured into a
 * CUDA graph count once, at capture).  count: host pointer.  Never fails
 * except on a NULL pointer (PA_ERR_INVALID_ARG).
 */
pa_status pa_launch_count(uint64_t* count);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */

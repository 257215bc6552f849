// pa_internal.h -- host-side interfaces between the C ABI (pa_api.cu) and the
// translation units that hold the kernels.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// Kernels launched from the calling host thread (pa_launch_count); every
// launch site calls count_launch() once its launch has been accepted.
void count_launch();

// Bounded-wait limit and the skipped-copy testing hook of the pipelined
// kernels, for the current device: attn_fast.cu and attn_prefill_tc.cu each
// hold their own copy (cudaMemcpyToSymbol, synchronous).
cudaError_t set_pipeline_hooks_fast(uint64_t wait_limit_ns, long long skip_copy);
cudaError_t set_pipeline_hooks_tc(uint64_t wait_limit_ns, long long skip_copy);

// ---- cache kernels (cache_kernels.cu) --------------------------------------
cudaError_t launch_reshape_and_cache(const void* key, const void* value,
                                     pa_dtype kv_dtype, int64_t num_tokens,
                                     int64_t key_stride, int64_t value_stride,
                                     void* k_cache, void* v_cache,
                                     pa_dtype cache_dtype, int64_t num_blocks,
                                     int num_kv_heads, int head_dim,
                                     const int64_t* slot_mapping, float k_scale,
                                     float v_scale, bool vector_ok,
                                     unsigned* err, cudaStream_t stream);

// 4-bit caches (PA_INT4, PA_NVFP4): one warp per (token, KV head, K or V)
cudaError_t launch_reshape_4bit(const void* key, const void* value,
                                pa_dtype kv_dtype, int64_t num_tokens,
                                int64_t key_stride, int64_t value_stride,
                                void* k_cache, void* v_cache,
                                pa_dtype cache_dtype, int64_t num_blocks,
                                int num_kv_heads, int head_dim,
                                const int64_t* slot_mapping, float k_scale,
                                float v_scale, unsigned* err,
                                cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, int64_t num_blocks,
                               int64_t block_bytes,
                               const int64_t* block_mapping, int64_t num_pairs,
                               unsigned* err, cudaStream_t stream);

// ---- attention (attn_*.cu) --------------------------------------------------
// One work item of the attention kernel: request r, KV head g, kind
// (0 = decode split, 1 = prefill row tile) and the split / tile index x.
enum : int { kItemDecode = 0, kItemPrefill = 1 };

constexpr int kDecodeMaxRows = 16;   // q_len * group rows handled by one warp
#ifndef PA_CONSUMER_WARPS
#define PA_CONSUMER_WARPS 4
#endif
// rows of a prefill tile: 16 per consumer warp
constexpr int kPrefillTileRows = 16 * PA_CONSUMER_WARPS;

#ifndef PA_CTAS_PER_SM
#define PA_CTAS_PER_SM 2  // resident attention CTAs per SM the kernels are built for
#endif
// the head-group decode kernel over 4-bit caches: three CTAs per SM (a
// smaller ring; the kernel is bound by instruction issue, so more warps)
constexpr int kCtasPerSm4 = 3;
// grid bound of the attention kernels
constexpr int kMaxCtasPerSm = PA_CTAS_PER_SM > kCtasPerSm4 ? PA_CTAS_PER_SM : kCtasPerSm4;

// "No sliding window" inside the kernels: a row with causal limit lim sees
// keys lim - window + 1 .. lim, so a window this wide never cuts.
constexpr int kNoWindow = 1 << 30;

// Rows of one split-K partial slot (a head group's 4 KV heads x 8 rows) and
// the partial-result bytes make_plan reserves per SM whatever the step's
// size: two slots per resident attention CTA, each rows x head_dim 128 fp32
// accumulators plus (m, l).  A batch-1 decode needs this much workspace.
constexpr int kPartialRowsPerSlot = 32;
constexpr size_t kPartialBytesPerSm =
    (size_t)2 * kMaxCtasPerSm * kPartialRowsPerSlot * (128 + 2) * 4;

struct AttnPlan {
  int group;            // Hq / Hkv
  int has_prefill;      // some request may have > 16 query rows
  int has_decode;       // some request may have <= 16 query rows
  int grid_max;         // CTAs of the attention kernel, at most
  int64_t max_atoms;    // prefill tiles, at most
  int64_t max_items;    // work items, at most
  int64_t max_slots;    // partial results, at most (2 per CTA)
  // workspace carve-up (byte offsets, 256-aligned)
  size_t off_atoms, off_atom_start, off_req_dec0, off_req_declen, off_req_rows,
      off_items,
      off_cta_begin, off_seg_info, off_split, off_pref, off_acc, off_ml,
      off_win_sl, off_win_bt, total_bytes;
  // sliding window (0: none): each request's view from the block holding its
  // first query's first key in the window -- block-table rows of win_blocks
  // entries and key counts of at most win_max_seq_len
  int window, win_blocks, win_max_seq_len;
  // shared-prefix (cascade) steps: partial rows after the max_slots slots --
  // unc_slots more slots (one per decode request and head group, for the
  // suffix of a segment that no range boundary cuts), then one row per
  // (token, q head) for the shared prefix (casc_row0 onwards)
  int cascade;
  int64_t unc_slots, casc_row0;
  // the prefix's key ranges (one tile, and one partial row per token and q
  // head, each): room for casc_splits ranges of casc_split_rows rows
  int casc_splits;
  int64_t casc_split_rows;
};

// Shared-prefix tiles split the prefix into key ranges of at least
// kCascMinSplitBlocks blocks (four chunks of the tensor-core kernel), at most
// kCascMaxSplits ranges, so that a long prefix read by few tokens still
// spreads over the SMs.
constexpr int kCascMinSplitBlocks = 32;
constexpr int kCascMaxSplits = 32;

// key ranges of a cascade step's prefix of cascade_blocks blocks (<= the
// plan's casc_splits)
int cascade_splits(const AttnPlan& plan, int cascade_blocks);

// Host planning from host-known sizes only (no device read-back).
// window: the sliding window in keys (0: none; a window of at least
// max_seq_len keys cuts nothing and counts as none).
// cascade: room for a shared-prefix step (pa_attention_cascade).
AttnPlan make_plan(int64_t num_tokens, int num_q_heads, int num_kv_heads,
                   int head_dim, int num_seqs, int max_query_len,
                   int max_seq_len, int num_sms, int window = 0,
                   bool cascade = false);


struct AttnArgs {
  const void* q;
  pa_dtype q_dtype;
  const void* k_cache;
  const void* v_cache;
  pa_dtype cache_dtype;
  int64_t num_blocks;
  int num_q_heads, num_kv_heads, head_dim;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int num_seqs;
  int64_t num_tokens;
  int max_query_len, max_seq_len;
  float scale, k_scale, v_scale;
  void* out;
  void* workspace;
  unsigned* err;
  int window;  // sliding window in keys (0: none)
  int cascade_blocks;  // leading block-table entries all requests share,
                       // computed once for the step (0: no cascade)
};

// true if a shared-prefix step of these types and shapes runs as a cascade
// (prefix tiles on the tensor cores, suffixes on the head-group decode
// kernel); otherwise the prefix hint is not used
bool cascade_supported(const AttnArgs& a);

// true if the TMA + tensor-core kernel covers these types / shapes
bool fast_path_supported(const AttnArgs& a);

// The step's view through a sliding window (plan.window > 0): for every
// request, its block-table row from the block that holds its first query's
// first key inside the window, and its key count from that block on, into
// the workspace at plan.off_win_bt / off_win_sl.
cudaError_t launch_window_view(const AttnArgs& a, const AttnPlan& plan,
                               cudaStream_t stream);

// events recorded around the main attention launch (measurement hook)
struct ProfileEvents {
  cudaEvent_t start = nullptr;
  cudaEvent_t stop = nullptr;
};
ProfileEvents& profile_events();  // thread-local

// tensor maps of the tensor-core prefill kernel: q as [token][head][dim],
// each cache as [row][dim] with 64-column boxes of one page
struct TcMaps {
  CUtensorMap q, k, v;
};

// true if the tensor-core kernel can take the prefill tiles of such a step
bool tc_prefill_supported(const AttnArgs& a);
// query rows of one of its tiles (128 / group tokens x group heads)
int tc_prefill_tile_rows(int group);
bool encode_prefill_tensor_maps(const AttnArgs& a, TcMaps* maps);
// the step's prefill tiles (requests of more than dec_rows_max query rows),
// listed by the kernel itself (self_plan) or by the planner (atoms,
// n_atoms); one persistent CTA per SM.  tile_ctr (zeroed int, or null):
// tiles drawn dynamically; after_decode: launched right behind the step's
// decode kernel, whose output it does not read (starts as its CTAs retire).
// casc_acc / casc_ml: the shared-prefix tiles' partial rows (cascade steps,
// a.cascade_blocks > 0, self-planned only): casc_splits key ranges of the
// prefix, range s at rows s * casc_split_rows + token * num_q_heads + head.
cudaError_t launch_prefill_tc(const AttnArgs& a, const TcMaps& maps,
                              bool self_plan, const int4* atoms,
                              const int* n_atoms, int max_atoms,
                              int dec_rows_max, int* tile_ctr, bool after_decode,
                              int num_sms, cudaStream_t stream,
                              float* casc_acc = nullptr, float* casc_ml = nullptr,
                              int casc_splits = 1, int64_t casc_split_rows = 0);

// plan kernel + (tensor-core prefill kernel) + main kernel + split merge
cudaError_t launch_attention_fast(const AttnArgs& a, const AttnPlan& plan,
                                  const CUtensorMap& tmap_k,
                                  const CUtensorMap& tmap_v, const TcMaps* tc,
                                  int num_sms, cudaStream_t stream);

// warp-per-row kernel for the remaining types / shapes
cudaError_t launch_attention_generic(const AttnArgs& a, cudaStream_t stream);

// Rows of one TMA box of the caches for the attention kernels of this step:
// 16 (one page), or 64 (the pages of four KV heads of a block) when the step
// runs in head groups.
// tc: the step's prefill tiles go to the tensor-core kernel
int decode_box_rows(const AttnArgs& a, bool tc);

// Encode the tensor maps of the two caches for the fast path (boxes of
// box_rows rows of 128-byte segments).
bool encode_cache_tensor_maps(const AttnArgs& a, CUtensorMap* tmap_k,
                              CUtensorMap* tmap_v, int box_rows);

}  // namespace pa

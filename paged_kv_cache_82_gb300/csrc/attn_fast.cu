// attn_fast.cu -- unified paged attention for one scheduler step (sm_103a).
//
// What it computes ("vLLM engine anatomy": PagedAttention section and Figure
// 2 for the paging, Table 1 for GQA, "Boundaries: FlashAttention ..." for
// exact attention with an online softmax; "vLLM V1 engine architecture":
// one step mixes decodes with prefill chunks): for every query token of every
// request, softmax attention over the request's keys 0 .. L - n + i, read
// through the block table from 16-token pages.
//
// How (GB300):
//  * A planner kernel (one CTA) lays the step's work on one line -- prefill
//    tiles of 64 query rows (indivisible, weighted by their key pages), then
//    one segment of key pages per (decode request, KV head) -- and cuts it
//    into equal contiguous ranges, one per resident CTA of the attention
//    kernel (stream-K).  A segment cut by a range boundary is finished by the
//    merge kernel from one partial result per piece.
//  * The attention kernel is persistent: in every CTA a producer warp walks
//    the CTA's items and streams each (block, KV head) page of K and V into
//    a shared-memory ring with TMA (cp.async.bulk.tensor, 128-byte swizzle),
//    completing on mbarriers; four consumer warps run Q.K^T and P.V on the
//    warp-level tensor-core MMA straight from the swizzled pages with an fp32
//    online softmax in registers.  Decode pages go round-robin to the four
//    warps (merged through shared memory at the end of the piece); a prefill
//    tile gives each warp 16 rows and all pages.  The ring streams across
//    item boundaries.
//  * The merge combines the parts of a split segment in a fixed order
//    (deterministic): M = max m_s, out = sum e^{m_s-M} acc_s / sum e^{m_s-M} l_s.
//  * The attention kernel and the merge are launched as programmatic
//    dependents of their predecessors.
//
// Decode is HBM-bound: every page is read from HBM once per step and the MMA
// only keeps the ALU work (group x 128 MACs per key) off the CUDA cores.
#include <float.h>

#include <algorithm>
#include <cmath>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

#ifndef PA_NARROW_MIN_BLOCKS
#define PA_NARROW_MIN_BLOCKS 3  // resident CTAs per SM, <= 8-row kernel
#endif
constexpr int kMinUnitsPerCta = 8;  // smallest cost range given to a CTA
#ifndef PA_SEG_COST
#define PA_SEG_COST 2
#endif
// Cost units a decode segment adds to the in-kernel plan besides its pages
// (the fixed work of starting an item: its Q rows, block ids, state): they
// sit on the line ahead of the segment's pages.
constexpr int kSegCost = PA_SEG_COST;
// requests of a step the attention kernel plans itself (narrow / wide build)
constexpr int kSelfPlanMaxSeqs = 1024;
constexpr int kSelfPlanMaxSeqsWide = 512;
constexpr int kHg = 4;            // KV heads of a head-group decode item
constexpr int kHgMaxSeqs = 512;   // requests of a step the head-group kernel takes
constexpr int kHgPartRows = 32;   // partial rows per slot there: kHg heads x 8
static_assert(kHgPartRows == kPartialRowsPerSlot, "partial slot rows");

#ifndef PA_L2_PREFETCH_PAGES
#define PA_L2_PREFETCH_PAGES 2  // head-group producer, mixed steps: L2 prefetch distance
#endif
#ifndef PA_PRODUCER_PAGES
#define PA_PRODUCER_PAGES 4     // pages the producer issues per step (2 lanes each)
#endif
#ifndef PA_PREFILL_WEIGHT
#define PA_PREFILL_WEIGHT 2     // cost of a prefill tile page vs a decode page
#endif
#ifndef PA_CONSUMER_WARPS
#define PA_CONSUMER_WARPS 4     // consumer warps per CTA (one producer warp)
#endif
#ifndef PA_CTAS_PER_SM
#define PA_CTAS_PER_SM 2        // resident CTAs per SM the kernel is built for
#endif
#ifndef PA_STAGES_16BIT
#define PA_STAGES_16BIT 8       // ring depth in pages, bf16 / fp16 caches
#endif
// head_dim 64 in the head-group kernel: three CTAs per SM with four-stage
// rings (64 KiB) instead of two with six, the same bytes in flight per SM and
// half again the warps (Llama-3.1-8B-shaped batch at D = 64: kernel 0.0560
// -> 0.0539-0.0545 ms)
#ifndef PA_HG_D64_CTAS
#define PA_HG_D64_CTAS 3
#endif
#ifndef PA_HG_D64_STAGES
#define PA_HG_D64_STAGES 4  // (0: the ring's bytes, PA_HG_RING_BYTES)
#endif
#ifndef PA_HG_RING_BYTES
#define PA_HG_RING_BYTES 98304  // ring of the head-group kernel (96 KiB)
#endif

constexpr int kConsumerWarps = PA_CONSUMER_WARPS;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
static_assert(kConsumerWarps == 4 || kConsumerWarps == 8,
              "4 or 8 consumer warps");
constexpr int kPlanThreads = 1024;


// ---------------------------------------------------------------------------
// compile-time traits of the four supported (cache, q) type pairs
// ---------------------------------------------------------------------------
enum : int {
  kKindBF16 = 0, kKindF16 = 1, kKindFp8BF16 = 2, kKindFp8F16 = 3,
  // 4-bit caches (head-group decode kernel only): INT4 / NVFP4, bf16 / f16 q
  kKindI4BF16 = 4, kKindI4F16 = 5, kKindN4BF16 = 6, kKindN4F16 = 7,
  // head_dim 64, bf16 / f16 (head-group decode kernel only)
  kKindBF16D64 = 8, kKindF16D64 = 9
};

template <int kKind>
struct Traits {
  // 0: none, 1: INT4 per token-head, 2: NVFP4 (pages of pa.h)
  static constexpr int k4 = kKind == kKindN4BF16 || kKind == kKindN4F16   ? 2
                          : kKind == kKindI4BF16 || kKind == kKindI4F16 ? 1
                                                                        : 0;
  static constexpr bool kFp8 = kKind == kKindFp8BF16 || kKind == kKindFp8F16;
  static constexpr int kD = kKind >= kKindBF16D64 ? 64 : 128;  // head_dim
  static constexpr bool kMmaBF16 = kKind == kKindBF16 || kKind == kKindBF16D64;
  static constexpr bool kQBF16 = kKind == kKindBF16 || kKind == kKindFp8BF16 ||
                                 kKind == kKindI4BF16 || kKind == kKindN4BF16 ||
                                 kKind == kKindBF16D64;
  // a page's rows are one 128-byte segment (FP8 at head_dim 128, 16-bit at
  // head_dim 64): 2-D TMA boxes, the 128-byte-row token order below
  static constexpr bool kRows128 = kFp8 || kD == 64;
  // q is widened to f16 for a quantised cache (an exact decode to f16)
  static constexpr bool kQToF16 = kFp8 || k4 != 0;
  static constexpr int kRowBytes = k4 ? 64 : kRows128 ? 128 : 256;
  // one (block, head) page; a 4-bit page ends with its scales
  static constexpr int kPageBytes = k4 == 1 ? 16 * 64 + 16 * 4
                                    : k4 == 2 ? 16 * 64 + 16 * 8
                                              : kBS * kRowBytes;
  static constexpr int kStageBytes = 2 * kPageBytes;    // K page + V page
  static constexpr int kStages = kFp8 ? 2 * PA_STAGES_16BIT : PA_STAGES_16BIT;
  static constexpr int kRingBytes = kStages * kStageBytes;  // 64 KiB
  // Token order inside an 8-token MMA tile (row n of the tile holds token
  // perm(n)).  A page sits in shared memory as the TMA wrote it under the
  // 128-byte swizzle: FP8 rows of 128 bytes (16-byte chunk k of token t at
  // chunk k ^ (t & 7)); 16-bit rows of 256 bytes, two 128-byte segments
  // (chunk k of segment h of token t at k ^ ((2t + h) & 7)).  With these
  // orders (0,5,2,7,4,1,6,3 for FP8, 0,2,1,3,6,4,7,5 for 16-bit) the 16-byte
  // fragment reads of K and V are free of bank conflicts; the transposing
  // V reads of the decode path are two-way.
  static constexpr uint32_t kPerm = k4         ? 0x76543210u
                                    : kRows128 ? 0x36147250u
                                               : 0x57463120u;
  // A decode item hands page i to warp i % 4 through slot i % kStages.  The
  // ring depth must be a multiple of the consumer count so that every slot
  // always serves the same warp: otherwise a fast warp can wait one full
  // phase ahead on a slot another warp still owns, the parity wait cannot
  // tell the two phases apart, and the slot's barriers are corrupted.
  static_assert(kStages % kConsumerWarps == 0,
                "ring depth must be a multiple of the consumer warp count");
};

__device__ __forceinline__ int perm_of(uint32_t packed, int n) {
  return (packed >> (4 * n)) & 7;
}

// the two bf16 halves of a packed pair, as fp32 (exact)
__device__ __forceinline__ float bf16_lo(uint32_t x) {
  return __uint_as_float(x << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t x) {
  return __uint_as_float(x & 0xFFFF0000u);
}

struct FastParams {
  const void* q;
  void* out;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;
  const int4* items;      // 2 x int4 per work item (see the planner)
  const int* cta_begin;   // work items of CTA b: [cta_begin[b], cta_begin[b+1])
  const int4* split_list; // segments cut into parts: {r, g, parts, first}
  const int* n_split;
  int max_slots;
  float* ws_acc;          // partial O: [slot][16 rows][128]
  float* ws_ml;           // partial (m, l): [slot][16 rows][2]
  unsigned* err;
  int64_t num_tokens;
  int64_t num_blocks;
  int max_blocks_per_seq;
  int num_seqs;
  int num_q_heads, num_kv_heads, group;
  int max_query_len, max_seq_len;
  float score_scale;  // softmax scale * log2(e) (* k_scale for FP8)
  float out_scale;    // 1, or v_scale for FP8
  int self_plan;      // 1: every CTA plans its own range
  int dec_rows_max;   // decode-class requests have at most this many rows
  int seg_heads;      // KV heads per decode segment (1, or kHg: head groups)
  int attn_grid;      // CTAs of the attention kernel (the merge's plan)
  int no_dep_wait;    // 1: start without waiting for the grid before (it let
                      // this one start only after its own wait)
  int window;         // sliding window in keys (kNoWindow: none): a row with
                      // causal limit lim sees keys lim - window + 1 .. lim
  const uint8_t* k4;  // 4-bit caches: [block][head][page] bytes (bulk copies)
  const uint8_t* v4;
  int head_dim;       // 128, or 64 (16-bit caches, head-group decode kernel)
  int l2_prefetch;    // 1: the head-group producer prefetches pages into L2
                      // PA_L2_PREFETCH_PAGES ahead of its loads
  // shared-prefix (cascade) steps, head-group kernel: every request's first
  // cascade_blocks pages are left to the prefix tiles (partial rows from
  // casc_row0 on: casc_splits key ranges of the prefix, range s at rows
  // s * casc_split_rows + token * num_q_heads + q head); the decode segments
  // cover the pages after them, and a segment that no range boundary cuts
  // writes its partial to slot unc_slot0 + request * (KV heads / kHg) + head
  // group.
  int cascade_blocks;
  int casc_splits;
  int64_t unc_slot0, casc_row0, casc_split_rows;
};

// ---------------------------------------------------------------------------
// planner: one CTA lays the step's work on one line and cuts it into equal
// contiguous ranges, one per CTA of the attention kernel
//
// Work units: a prefill tile (kPrefillTileRows query rows of one KV head,
// all keys up to the tile's causal limit) is indivisible and costs
// `prefill_weight` per key page; a decode-class request (q_len * group <= 16
// rows) contributes one segment per KV head, one unit per key page, which may
// be cut anywhere.  Prefill tiles come first, then the decode segments in
// (request, head) order.  CTA b owns the cost interval [b*C/G, (b+1)*C/G):
// every tile that starts in it, and the pieces of the segments that overlap
// it.  A segment cut by CTA boundaries is finished by the merge kernel from
// one partial result per piece (at most 2G of them in total).
// ---------------------------------------------------------------------------
struct PlanArgs {
  const int32_t* qsl;
  const int32_t* seq_lens;
  unsigned* err;
  int64_t num_tokens;
  int num_seqs, max_query_len, max_seq_len, max_blocks_per_seq;
  int group, num_kv_heads, grid, prefill_weight;
  int tile_rows;          // query rows of a prefill tile
  int prefill_tc;         // 1: prefill tiles go to the tensor-core kernel
  int* n_atoms_out;       // prefill tiles of the step (for that kernel)
  int max_atoms, max_items, max_slots;
  int4* atoms;            // prefill tiles: {r, g, tile, pages}
  long long* atom_start;  // cost offset of each tile
  long long* req_dec0;    // decode-unit offset of each request
  int* req_declen;        // key pages of a decode-class request (0 if none)
  int* req_rows;          // query rows (q_len * group) of each request
  int2* seg_cut;          // per (request, KV head): first partial slot, first CTA
  int4* items;
  int* cta_begin;
  float* ws_ml;           // partial (m, l), initialised here
  int4* split_list;       // segments cut by CTA boundaries: {r, g, parts, first}
  int* n_split;
};

// key pages seen by prefill tile tt of a request (its last row's limit)
__device__ __forceinline__ int tile_pages(const ReqMeta& m, int G, int tt,
                                          int tile_rows) {
  const int last_row = min(m.n * G, (tt + 1) * tile_rows) - 1;
  return (m.L - m.n + last_row / G) / kBS + 1;
}

__device__ __forceinline__ long long cta_lo(int b, long long C, int grid) {
  return (long long)b * C / grid;
}

// last CTA whose range starts at or before cost c (los[b] = start of CTA b)
__device__ __forceinline__ int cta_of(long long c, const long long* los,
                                      int grid) {
  int lo = 0, hi = grid - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (los[mid] <= c) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// first index in [0, n) with a[i] >= x (n if none)
__device__ __forceinline__ int lower_bound_ll(const long long* a, int n,
                                              long long x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

constexpr int kPlanCacheBytes = 40 * 1024;  // dynamic shared memory of the planner

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs pa) {
  extern __shared__ long long plan_cache[];
  // the attention kernel may start its prologue now; it waits for this
  // grid to finish before it reads the plan
  pdl_launch_dependents();
  __shared__ long long ws_ll[32];
  __shared__ int ws_i[32];
  __shared__ long long tot_ll;
  __shared__ int tot_i;
  __shared__ long long s_atoms, s_cost_pre, s_dec_total;
  const int G = pa.group, H = pa.num_kv_heads, W = pa.prefill_weight;
  // ---- 1: per request: prefill tiles (with their costs) and decode pages
  long long run_atoms = 0, run_pcost = 0, run_dec = 0;
  for (int base = 0; base < pa.num_seqs; base += blockDim.x) {
    const int r = base + threadIdx.x;
    ReqMeta m{0, 0, 0, 0, false};
    int tiles = 0, declen = 0;
    long long pcost = 0;
    if (r < pa.num_seqs) {
      m = load_req(pa.qsl, pa.seq_lens, r, pa.num_tokens, pa.max_query_len,
                   pa.max_seq_len, pa.max_blocks_per_seq);
      if (!m.ok) {
        flag_error(pa.err, PA_DEV_ERR_METADATA);
      } else if (m.n > 0) {
        if (m.n * G <= kDecodeMaxRows) {
          declen = m.nb;
        } else {
          tiles = (m.n * G + pa.tile_rows - 1) / pa.tile_rows;
          // tiles run by the tensor-core kernel are not on the cost line
          if (!pa.prefill_tc)
            for (int tt = 0; tt < tiles; ++tt)
              pcost += (long long)tile_pages(m, G, tt, pa.tile_rows) * W;
        }
      }
    }
    const long long atoms_r = (long long)tiles * H;
    const long long pcost_r = pcost * H;
    const long long dec_r = (long long)declen * H;
    const long long ex_atoms = block_scan_excl<long long>(atoms_r, &tot_ll, ws_ll);
    const long long t_atoms = tot_ll;
    __syncthreads();
    const long long ex_pcost = block_scan_excl<long long>(pcost_r, &tot_ll, ws_ll);
    const long long t_pcost = tot_ll;
    __syncthreads();
    const long long ex_dec = block_scan_excl<long long>(dec_r, &tot_ll, ws_ll);
    const long long t_dec = tot_ll;
    __syncthreads();
    if (r < pa.num_seqs) {
      pa.req_dec0[r] = run_dec + ex_dec;
      pa.req_declen[r] = declen;
      pa.req_rows[r] = m.ok ? m.n * G : 0;
      long long a0 = run_atoms + ex_atoms;
      long long c0 = run_pcost + ex_pcost;
      for (int tt = 0; tt < tiles; ++tt) {
        const int pg = tile_pages(m, G, tt, pa.tile_rows);
        const long long c = pa.prefill_tc ? 0 : (long long)pg * W;
        for (int g = 0; g < H; ++g) {
          const long long ai = a0 + (long long)tt * H + g;
          if (ai < pa.max_atoms) {
            pa.atoms[ai] = make_int4(r, g, tt, pg);
            pa.atom_start[ai] = c0 + g * c;
          } else {
            flag_error(pa.err, PA_DEV_ERR_METADATA);
          }
        }
        c0 += c * H;
      }
    }
    run_atoms += t_atoms;
    run_pcost += t_pcost;
    run_dec += t_dec;
  }
  if (threadIdx.x == 0) {
    s_atoms = run_atoms < pa.max_atoms ? run_atoms : pa.max_atoms;
    if (pa.prefill_tc) *pa.n_atoms_out = (int)s_atoms;
    s_cost_pre = run_pcost;
    s_dec_total = run_dec;
  }
  __syncthreads();
  // prefill tiles the attention kernel runs (none when the tensor-core
  // kernel takes them)
  const int n_atoms = pa.prefill_tc ? 0 : (int)s_atoms;
  const long long cost_pre = s_cost_pre, dec_total = s_dec_total;
  const long long C = cost_pre + dec_total;
  // CTAs that get work: every cost range at least kMinUnitsPerCta long, so
  // no range is empty; the others find an empty item list
  long long g_eff = C / kMinUnitsPerCta;
  if (g_eff > pa.grid) g_eff = pa.grid;
  if (g_eff < 1) g_eff = 1;
  const int grid = (int)g_eff;
  // Everything the per-CTA walks below read goes to shared memory when it
  // fits (in 8-byte words): range starts, per-request decode offsets /
  // lengths / rows, per-segment cut info, tile starts; else it stays global.
  long long* los = plan_cache;
  for (int b = threadIdx.x; b <= grid; b += blockDim.x)
    los[b] = C > 0 ? cta_lo(b, C, grid) : 0;
  long long free_ll = kPlanCacheBytes / 8 - (grid + 1);
  long long* next = los + grid + 1;
  const int B = pa.num_seqs;
  const bool req_sm = 2ll * B <= free_ll;  // dec0 + (declen, rows)
  long long* dec0 = req_sm ? next : pa.req_dec0;
  int* declen_a = req_sm ? reinterpret_cast<int*>(next + B) : pa.req_declen;
  int* rows_a = req_sm ? declen_a + B : pa.req_rows;
  if (req_sm) {
    for (int r = threadIdx.x; r < B; r += blockDim.x) {
      dec0[r] = pa.req_dec0[r];
      declen_a[r] = pa.req_declen[r];
      rows_a[r] = pa.req_rows[r];
    }
    next += 2ll * B;
    free_ll -= 2ll * B;
  }
  const long long nseg = (long long)B * H;
  const bool seg_sm = nseg <= free_ll;
  int2* seg_cut = seg_sm ? reinterpret_cast<int2*>(next) : pa.seg_cut;
  if (seg_sm) {
    next += nseg;
    free_ll -= nseg;
  }
  const bool atoms_sm = n_atoms <= free_ll;
  long long* astart = atoms_sm ? next : pa.atom_start;
  if (atoms_sm)
    for (int i = threadIdx.x; i < n_atoms; i += blockDim.x) astart[i] = pa.atom_start[i];
  __syncthreads();
  __syncthreads();
  // ---- 2: decode segments, one thread each: the CTAs that cut it, its
  // first partial slot and its place in the list of split segments.  (Every
  // CTA in a split segment's span owns a non-empty piece of it, so every
  // partial slot is written before the merge reads it.)
  int run_slots = 0, run_split = 0;
  for (long long base = 0; base < nseg; base += blockDim.x) {
    const long long sg = base + threadIdx.x;
    int parts = 0, bf = 0;
    if (sg < nseg) {
      const int r = (int)(sg / H), g = (int)(sg - (long long)r * H);
      const int declen = declen_a[r];
      if (declen > 0) {
        const long long s0 = cost_pre + dec0[r] + (long long)g * declen;
        bf = cta_of(s0, los, grid);
        parts = cta_of(s0 + declen - 1, los, grid) - bf + 1;
      }
    }
    const int nslots = parts > 1 ? parts : 0;
    const int ex_slot = block_scan_excl<int>(nslots, &tot_i, ws_i);
    const int t_slot = tot_i;
    __syncthreads();
    const int ex_split = block_scan_excl<int>(parts > 1 ? 1 : 0, &tot_i, ws_i);
    const int t_split = tot_i;
    __syncthreads();
    if (sg < nseg) {
      int first = -1;
      if (parts > 1) {
        const int slot = run_slots + ex_slot;
        if (slot + parts <= pa.max_slots) {
          first = slot;
          const int k = run_split + ex_split;
          pa.split_list[k] = make_int4((int)(sg / H), (int)(sg % H), parts, first);
        } else {
          flag_error(pa.err, PA_DEV_ERR_METADATA);
        }
      }
      seg_cut[sg] = make_int2(first, bf);
    }
    run_slots += t_slot;
    run_split += t_split;
  }
  if (threadIdx.x == 0) *pa.n_split = run_split;
  __syncthreads();  // seg_cut complete before the walks read it

  // ---- 3: items of every CTA (count, scan, emit)
  int run_items = 0;
  for (int base = 0; base < pa.grid; base += blockDim.x) {
    const int b = base + threadIdx.x;
    long long lo = 0, hi = 0;
    int a0 = 0, a1 = 0;
    if (b < grid && C > 0) {  // CTAs at or past the effective grid: no work
      lo = los[b];
      hi = los[b + 1];
      a0 = lower_bound_ll(astart, n_atoms, lo);
      a1 = lower_bound_ll(astart, n_atoms, hi);
    }
    // decode interval of this CTA, in decode units
    const long long d0 = min(max(lo, cost_pre) - cost_pre, dec_total);
    const long long d1 = min(max(hi, cost_pre) - cost_pre, dec_total);
    int cnt = a1 - a0;
    for (int pass = 0; pass < 2; ++pass) {
      int o = 0;
      if (pass == 1) {
        const int ex = block_scan_excl<int>(cnt, &tot_i, ws_i);
        o = run_items + ex;
        if (b < pa.grid) pa.cta_begin[b] = min(o, pa.max_items);
        for (int a = a0; a < a1; ++a, ++o) {
          if (o < pa.max_items) {
            const int4 at = pa.atoms[a];
            const ReqMeta m = load_req(pa.qsl, pa.seq_lens, at.x, pa.num_tokens,
                                       pa.max_query_len, pa.max_seq_len,
                                       pa.max_blocks_per_seq);
            const int rows =
                min(pa.tile_rows, m.n * G - at.z * pa.tile_rows);
            pa.items[2 * o] = make_int4(at.x, at.y, kItemPrefill, at.z);
            pa.items[2 * o + 1] = make_int4(0, at.w, rows, 0);
          }
        }
      }
      if (d0 < d1) {
        // request holding decode unit d0: last r with req_dec0[r] <= d0
        int lo_r = 0, hi_r = pa.num_seqs - 1;
        while (lo_r < hi_r) {
          const int mid = (lo_r + hi_r + 1) >> 1;
          if (dec0[mid] <= d0) lo_r = mid; else hi_r = mid - 1;
        }
        int r = lo_r;
        long long cur = d0;
        int n_pieces = 0;
        while (cur < d1 && r < pa.num_seqs) {
          const int declen = declen_a[r];
          if (declen == 0) { ++r; continue; }
          const long long rs = dec0[r];
          const int g = (int)((cur - rs) / declen);
          const long long ss = rs + (long long)g * declen;
          const long long se = ss + declen;
          const long long pe = min(se, d1);
          if (pass == 1 && o < pa.max_items) {
            const int2 sc = seg_cut[(long long)r * H + g];
            const int slot = sc.x >= 0 ? sc.x + (b - sc.y) : -1;
            const int rows = rows_a[r];
            pa.items[2 * o] = make_int4(r, g, kItemDecode, slot);
            pa.items[2 * o + 1] = make_int4((int)(cur - ss), (int)(pe - ss), rows, 0);
          }
          ++o;
          ++n_pieces;
          cur = pe;
          if (g + 1 == H) ++r;
        }
        if (pass == 0) cnt += n_pieces;
      } else if (pass == 0) {
        // no decode work for this CTA
      }
      if (pass == 1) {
        const int t = tot_i;
        __syncthreads();
        run_items += t;
      }
    }
  }
  if (threadIdx.x == 0) {
    if (run_items > pa.max_items) flag_error(pa.err, PA_DEV_ERR_METADATA);
    pa.cta_begin[pa.grid] = min(run_items, pa.max_items);
  }
}

// ---------------------------------------------------------------------------
// MMA helpers for the "rows 0..7 only" case (rows 8..15 of the A operand are
// zero and their accumulators are not kept)
// ---------------------------------------------------------------------------
template <bool kBF16>
__device__ __forceinline__ void mma_rows8(float& d0, float& d1, uint32_t a0,
                                          uint32_t a2, uint32_t b0,
                                          uint32_t b1) {
  float x2, x3;
  const uint32_t z = 0;
  if constexpr (kBF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%10,%10};"
        : "+f"(d0), "+f"(d1), "=f"(x2), "=f"(x3)
        : "r"(a0), "r"(z), "r"(a2), "r"(z), "r"(b0), "r"(b1), "f"(0.0f));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%10,%10};"
        : "+f"(d0), "+f"(d1), "=f"(x2), "=f"(x3)
        : "r"(a0), "r"(z), "r"(a2), "r"(z), "r"(b0), "r"(b1), "f"(0.0f));
  }
}

template <bool kBF16, bool kRows16>
__device__ __forceinline__ void mma_acc(float (&d)[4], const uint32_t (&a)[4],
                                        uint32_t b0, uint32_t b1) {
  if constexpr (kRows16) {
    mma16816<kBF16>(d, a, b0, b1);
  } else {
    mma_rows8<kBF16>(d[0], d[1], a[0], a[2], b0, b1);
  }
}

// output column (head-dim index) of accumulator element e (0/1 -> columns
// 2c, 2c+1 of n-tile T)
template <int kKind>
__device__ __forceinline__ int out_col(int T, int e, int c) {
  const int n = 2 * c + (e & 1);
  if constexpr (Traits<kKind>::kFp8) {
    return 16 * n + T;
  } else {
    return 64 * (T >> 3) + 8 * n + (T & 7);
  }
}

// ---------------------------------------------------------------------------
// per-warp state
// ---------------------------------------------------------------------------
struct WarpState {
  float o[16][4];
  float m[2];
  float l[2];
};

// Load the A fragments of Q for this warp's rows.  Row R (request-relative)
// is query R / G, head g*G + R % G.  Rows outside [0, nrows) are zero.
template <int kKind, bool kRows16>
__device__ __forceinline__ void load_q(const FastParams& p, int q0, int g,
                                       int wrow0, int nrows, int lane,
                                       uint32_t (&qa)[8][4], float (&rscale)[2]) {
  using Tr = Traits<kKind>;
  const int r = lane >> 2, c = lane & 3;
  const int G = p.group;
  const int Hq = p.num_q_heads;
  rscale[0] = rscale[1] = 1.0f;
#pragma unroll
  for (int half = 0; half < (kRows16 ? 2 : 1); ++half) {
    const int rr = r + 8 * half;
    const bool valid = rr < nrows;
    const int R = wrow0 + rr;
    const uint4* src = nullptr;
    if (valid) {
      const int i = R / G;
      const int h = g * G + (R - i * G);
      src = reinterpret_cast<const uint4*>(
          static_cast<const uint16_t*>(p.q) +
          ((int64_t)(q0 + i) * Hq + h) * Tr::kD);
    }
    uint4 ch[4];
    if constexpr (!Tr::kFp8) {
      // 16-bit cache: chunk 4j + c of the row (8 elements) feeds k-steps
      // 2j and 2j+1
      constexpr int kJ = Tr::kD / 32;
#pragma unroll
      for (int j = 0; j < kJ; ++j)
        ch[j] = valid ? __ldg(src + 4 * j + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        qa[2 * j][half] = ch[j].x;
        qa[2 * j][2 + half] = ch[j].y;
        qa[2 * j + 1][half] = ch[j].z;
        qa[2 * j + 1][2 + half] = ch[j].w;
      }
    } else {
      // FP8 cache: elements 16(c + 4h) .. +16 feed k-steps 4h .. 4h+3
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        ch[2 * hh] = valid ? __ldg(src + 2 * (c + 4 * hh)) : make_uint4(0, 0, 0, 0);
        ch[2 * hh + 1] =
            valid ? __ldg(src + 2 * (c + 4 * hh) + 1) : make_uint4(0, 0, 0, 0);
      }
      uint32_t w[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w[4 * k + 0] = ch[k].x;
        w[4 * k + 1] = ch[k].y;
        w[4 * k + 2] = ch[k].z;
        w[4 * k + 3] = ch[k].w;
      }
      if constexpr (Tr::kQBF16) {
        // bf16 -> f16 with a per-row power-of-two shift so that the row's
        // largest |q| stays inside the f16 range; the shift is undone on the
        // scores.
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          amax = fmaxf(amax, fabsf(__uint_as_float(w[k] << 16)));
          amax = fmaxf(amax, fabsf(__uint_as_float(w[k] & 0xFFFF0000u)));
        }
        amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, 2));
        int e = 0;
        if (amax > 16384.f) e = ilogbf(amax) - 13;  // amax * 2^-e < 2^15
        const float down = exp2f((float)-e);
        rscale[half] = exp2f((float)e);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float lo = __uint_as_float(w[k] << 16) * down;
          const float hi = __uint_as_float(w[k] & 0xFFFF0000u) * down;
          w[k] = pack2<false>(lo, hi);
        }
      }
      // step 4hh + tt: a0 = pair 2tt, a2 = pair 2tt + 1 of half hh
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
          qa[4 * hh + tt][half] = w[8 * hh + 2 * tt];
          qa[4 * hh + tt][2 + half] = w[8 * hh + 2 * tt + 1];
        }
    }
  }
  if constexpr (!kRows16) {
#pragma unroll
    for (int s = 0; s < 8; ++s) qa[s][1] = qa[s][3] = 0u;
  }
}

// S^T = Q.K^T for one page: rows are query rows, columns the 16 keys (two
// 8-key tiles; column n of tile nt is key nt * 8 + perm(n)).  Two
// accumulators per tile (even / odd k-steps) keep four MMA chains in flight.
template <int kKind, bool kRows16>
__device__ __forceinline__ void qk_page(uint32_t k_base,
                                        const uint32_t (&qa)[8][4],
                                        float (&s)[2][4], int lane) {
  using Tr = Traits<kKind>;
  constexpr bool kB = Tr::kMmaBF16;
  constexpr uint32_t P = Tr::kPerm;
  const int r = lane >> 2, c = lane & 3;
  // Q.K^T: two accumulators per 8-key tile (even / odd k-steps) so that four
  // independent MMA chains are in flight
  float s2[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) s[nt][e] = s2[nt][e] = 0.f;
    const int t = nt * 8 + perm_of(P, r);
    if constexpr (!Tr::kFp8 && Tr::kD == 64) {
      // 128-byte rows: chunk u of token t at u ^ (t & 7)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int u = (j << 2) | c;
        const uint4 kv = lds128(k_base + t * 128 + ((u ^ (t & 7)) << 4));
        mma_acc<kB, kRows16>(s[nt], qa[2 * j], kv.x, kv.y);
        mma_acc<kB, kRows16>(s2[nt], qa[2 * j + 1], kv.z, kv.w);
      }
    } else if constexpr (!Tr::kFp8) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int dhi = j >> 1;
        const int u = ((j & 1) << 2) | c;
        const uint4 kv = lds128(k_base + t * 256 + dhi * 128 +
                                ((u ^ (((t << 1) | dhi) & 7)) << 4));
        mma_acc<kB, kRows16>(s[nt], qa[2 * j], kv.x, kv.y);
        mma_acc<kB, kRows16>(s2[nt], qa[2 * j + 1], kv.z, kv.w);
      }
    } else {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int phys = (c + 4 * hh) ^ (t & 7);
        const uint4 kv = lds128(k_base + t * 128 + phys * 16);
        const uint32_t wv[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
          uint32_t b0, b1;
          e4m3x4_to_f16x2x2(wv[tt], b0, b1);
          if (tt & 1)
            mma_acc<false, kRows16>(s2[nt], qa[4 * hh + tt], b0, b1);
          else
            mma_acc<false, kRows16>(s[nt], qa[4 * hh + tt], b0, b1);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) s[nt][e] += s2[nt][e];
  }
}

// Process one page (16 keys) held in shared memory at k_base / v_base.
template <int kKind, bool kRows16>
__device__ __forceinline__ void process_page(uint32_t k_base, uint32_t v_base,
                                             const uint32_t (&qa)[8][4],
                                             WarpState& st, int key0,
                                             int valid_keys, bool need_mask,
                                             int lim0, int lim1, int win,
                                             float sscale0, float sscale1,
                                             int lane) {
  using Tr = Traits<kKind>;
  constexpr bool kB = Tr::kMmaBF16;
  constexpr uint32_t P = Tr::kPerm;
  const int r = lane >> 2, c = lane & 3;
  float s[2][4];
  qk_page<kKind, kRows16>(k_base, qa, s, lane);
  // scale, mask
  const int tA = perm_of(P, 2 * c), tB = perm_of(P, 2 * c + 1);
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v = s[nt][e] * (e < 2 ? sscale0 : sscale1);
      if (need_mask) {
        // visible: lim - win < key <= lim (the causal limit, the window)
        const int key = key0 + nt * 8 + ((e & 1) ? tB : tA);
        const int lim = e < 2 ? lim0 : lim1;
        if (key > lim || key <= lim - win) v = -INFINITY;
      }
      s[nt][e] = v;
    }
  // online softmax (base 2), per row
  float alpha[2];
#pragma unroll
  for (int half = 0; half < (kRows16 ? 2 : 1); ++half) {
    const int e0 = 2 * half;
    float mx = fmaxf(fmaxf(s[0][e0], s[0][e0 + 1]), fmaxf(s[1][e0], s[1][e0 + 1]));
    mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 2));
    const float mnew = fmaxf(st.m[half], mx);
    const float muse = mnew == -INFINITY ? 0.f : mnew;
    alpha[half] = exp2f(st.m[half] - muse);
    st.m[half] = mnew;
    float sum = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = e0; e < e0 + 2; ++e) {
        s[nt][e] = exp2f(s[nt][e] - muse);
        sum += s[nt][e];
      }
    st.l[half] = st.l[half] * alpha[half] + sum;
  }
#ifndef PA_SKIP_RESCALE
#define PA_SKIP_RESCALE 1
#endif
  const bool moved = alpha[0] != 1.f || (kRows16 && alpha[1] != 1.f);
  if (!PA_SKIP_RESCALE || __any_sync(~0u, moved)) {
#pragma unroll
    for (int T = 0; T < 16; ++T) {
      st.o[T][0] *= alpha[0];
      st.o[T][1] *= alpha[0];
      if constexpr (kRows16) {
        st.o[T][2] *= alpha[1];
        st.o[T][3] *= alpha[1];
      }
    }
  }
  // P as the A operand of P.V (k = key within the page).  With bf16 MMA
  // operands P is split into a bf16 head and a bf16 tail (p = hi + lo), so
  // that P.V keeps ~16 bits of P instead of 8.
  uint32_t pa[4], pl[4];
  pa[0] = pack2<kB>(s[0][0], s[0][1]);
  pa[2] = pack2<kB>(s[1][0], s[1][1]);
  if constexpr (kRows16) {
    pa[1] = pack2<kB>(s[0][2], s[0][3]);
    pa[3] = pack2<kB>(s[1][2], s[1][3]);
  } else {
    pa[1] = pa[3] = 0u;
  }
  if constexpr (kB) {
    pl[0] = pack2<true>(s[0][0] - bf16_lo(pa[0]), s[0][1] - bf16_hi(pa[0]));
    pl[2] = pack2<true>(s[1][0] - bf16_lo(pa[2]), s[1][1] - bf16_hi(pa[2]));
    if constexpr (kRows16) {
      pl[1] = pack2<true>(s[0][2] - bf16_lo(pa[1]), s[0][3] - bf16_hi(pa[1]));
      pl[3] = pack2<true>(s[1][2] - bf16_lo(pa[3]), s[1][3] - bf16_hi(pa[3]));
    } else {
      pl[1] = pl[3] = 0u;
    }
  }
  // V fragments: keys tA, tB, 8 + tA, 8 + tB
  const int tk[4] = {tA, tB, 8 + tA, 8 + tB};
  if constexpr (!Tr::kFp8) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int t = tk[k];
        v[k] = lds128(v_base + t * 256 + h * 128 +
                      ((r ^ (((t << 1) | h) & 7)) << 4));
      }
      if (valid_keys < kBS) {  // last page: slots past the sequence end
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (tk[k] >= valid_keys) v[k] = make_uint4(0, 0, 0, 0);
      }
      const uint32_t va[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
      const uint32_t vb[4] = {v[1].x, v[1].y, v[1].z, v[1].w};
      const uint32_t vc[4] = {v[2].x, v[2].y, v[2].z, v[2].w};
      const uint32_t vd[4] = {v[3].x, v[3].y, v[3].z, v[3].w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int T = 8 * h + 2 * w;
        const uint32_t b00 = __byte_perm(va[w], vb[w], 0x5410);
        const uint32_t b01 = __byte_perm(vc[w], vd[w], 0x5410);
        const uint32_t b10 = __byte_perm(va[w], vb[w], 0x7632);
        const uint32_t b11 = __byte_perm(vc[w], vd[w], 0x7632);
        mma_acc<kB, kRows16>(st.o[T], pa, b00, b01);
        mma_acc<kB, kRows16>(st.o[T + 1], pa, b10, b11);
        if constexpr (kB) {
          mma_acc<kB, kRows16>(st.o[T], pl, b00, b01);
          mma_acc<kB, kRows16>(st.o[T + 1], pl, b10, b11);
        }
      }
    }
  } else {
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = tk[k];
      const int phys = r ^ (t & 7);
      v[k] = lds128(v_base + t * 128 + phys * 16);
    }
    if (valid_keys < kBS) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (tk[k] >= valid_keys) v[k] = make_uint4(0, 0, 0, 0);
    }
    const uint32_t va[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
    const uint32_t vb[4] = {v[1].x, v[1].y, v[1].z, v[1].w};
    const uint32_t vc[4] = {v[2].x, v[2].y, v[2].z, v[2].w};
    const uint32_t vd[4] = {v[3].x, v[3].y, v[3].z, v[3].w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t ab01 = __byte_perm(va[w], vb[w], 0x5140);
      const uint32_t ab23 = __byte_perm(va[w], vb[w], 0x7362);
      const uint32_t cd01 = __byte_perm(vc[w], vd[w], 0x5140);
      const uint32_t cd23 = __byte_perm(vc[w], vd[w], 0x7362);
      const int T = 4 * w;
      uint32_t x[8];
      e4m3x4_to_f16x2x2(ab01, x[0], x[1]);
      e4m3x4_to_f16x2x2(cd01, x[2], x[3]);
      e4m3x4_to_f16x2x2(ab23, x[4], x[5]);
      e4m3x4_to_f16x2x2(cd23, x[6], x[7]);
      mma_acc<false, kRows16>(st.o[T], pa, x[0], x[2]);
      mma_acc<false, kRows16>(st.o[T + 1], pa, x[1], x[3]);
      mma_acc<false, kRows16>(st.o[T + 2], pa, x[4], x[6]);
      mma_acc<false, kRows16>(st.o[T + 3], pa, x[5], x[7]);
    }
  }
}

// ---------------------------------------------------------------------------
// decode items with at most 8 query rows: S^T = Q.K^T as above, then
// O^T = V^T.P^T -- the accumulator fragment of S^T is, element for element,
// the B operand of P^T, and V^T comes from transposing matrix loads, so P.V
// needs 8 MMAs per page (M = 16 head-dim rows, N = 8 query rows, K = 16 keys)
// and no register shuffles.
// ---------------------------------------------------------------------------
struct NarrowState {
  float o[8][4];  // O^T: tile mt holds 16 head-dim rows x query rows 2c, 2c+1
  float m, l;     // softmax state of query row lane / 4
};

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&a)[4], uint32_t addr) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
      : "r"(addr));
}

// head-dim index of O^T element e of tile mt for thread (r, c)
template <int kKind>
__device__ __forceinline__ int narrow_col(int mt, int e, int r) {
  if constexpr (Traits<kKind>::kFp8 || Traits<kKind>::k4) {
    return 16 * r + 2 * mt + (e >> 1);
  } else {
    return 16 * mt + r + 8 * (e >> 1);
  }
}

template <int kKind>
__device__ __forceinline__ void process_page_narrow(
    uint32_t k_base, uint32_t v_base, const uint32_t (&qa)[8][4],
    NarrowState& st, int key0, int valid_keys, bool need_mask, int lim,
    int win, float sscale, int lane) {
  using Tr = Traits<kKind>;
  constexpr bool kB = Tr::kMmaBF16;
  constexpr uint32_t P = Tr::kPerm;
  const int r = lane >> 2, c = lane & 3;
  float s[2][4];
  qk_page<kKind, false>(k_base, qa, s, lane);
  const int tA = perm_of(P, 2 * c), tB = perm_of(P, 2 * c + 1);
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = s[nt][e] * sscale;
      if (need_mask) {
        // visible: lim - win < key <= lim (the causal limit, the window)
        const int key = key0 + nt * 8 + (e ? tB : tA);
        if (key > lim || key <= lim - win) v = -INFINITY;
      }
      s[nt][e] = v;
    }
  // online softmax (base 2) of query row r
  float mx = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
  mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 2));
  const float mnew = fmaxf(st.m, mx);
  const float muse = mnew == -INFINITY ? 0.f : mnew;
  const float alpha = exp2f(st.m - muse);
  st.m = mnew;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) s[nt][e] = exp2f(s[nt][e] - muse);
  st.l = st.l * alpha + ((s[0][0] + s[0][1]) + (s[1][0] + s[1][1]));
  // this thread's O^T columns are query rows 2c and 2c + 1
  const float a_lo = __shfl_sync(~0u, alpha, 8 * c);
  const float a_hi = __shfl_sync(~0u, alpha, 8 * c + 4);
  if (__any_sync(~0u, a_lo != 1.f || a_hi != 1.f)) {
#pragma unroll
    for (int mt = 0; mt < Tr::kD / 16; ++mt) {
      st.o[mt][0] *= a_lo;
      st.o[mt][1] *= a_hi;
      st.o[mt][2] *= a_lo;
      st.o[mt][3] *= a_hi;
    }
  }
  // P^T as the B operand: b0 = keys (tA, tB), b1 = keys (8 + tA, 8 + tB) of
  // query row r; with bf16 operands a bf16 head and tail of P
  const uint32_t b0 = pack2<kB>(s[0][0], s[0][1]);
  const uint32_t b1 = pack2<kB>(s[1][0], s[1][1]);
  uint32_t b0l = 0, b1l = 0;
  if constexpr (kB) {
    b0l = pack2<true>(s[0][0] - bf16_lo(b0), s[0][1] - bf16_hi(b0));
    b1l = pack2<true>(s[1][0] - bf16_lo(b1), s[1][1] - bf16_hi(b1));
  }
  // keys past the sequence end (last page only) hold NaN: clear them in V
  uint32_t m01 = ~0u, m23 = ~0u;
  if (valid_keys < kBS) {
    m01 = (tA < valid_keys ? 0x0000FFFFu : 0u) | (tB < valid_keys ? 0xFFFF0000u : 0u);
    m23 = (8 + tA < valid_keys ? 0x0000FFFFu : 0u) |
          (8 + tB < valid_keys ? 0xFFFF0000u : 0u);
  }
  if constexpr (!Tr::kFp8) {
    // matrix g (lanes 8g..8g+7) row i: key (g >> 1) * 8 + perm(i), head-dim
    // chunk 2 * (mt & 3) + (g & 1) of segment mt >> 2
    const int g8 = lane >> 3, i8 = lane & 7;
    const int tok = ((g8 >> 1) << 3) + perm_of(P, i8);
    constexpr int kRowB = Tr::kD == 64 ? 128 : 256;  // bytes of a token's row
    const uint32_t row = v_base + tok * kRowB;
    const int tx = Tr::kD == 64 ? (tok & 7) : ((tok << 1) & 7), gb = g8 & 1;
#pragma unroll
    for (int mt = 0; mt < Tr::kD / 16; ++mt) {
      uint32_t a[4];
      const int ch = 2 * (mt & 3) + gb;
      const int dhi = mt >> 2;
      ldsm_x4_trans(a, row + dhi * 128 + ((ch ^ (tx | dhi)) << 4));
      a[0] &= m01;
      a[1] &= m01;
      a[2] &= m23;
      a[3] &= m23;
      mma16816<kB>(st.o[mt], a, b0, b1);
      if constexpr (kB) mma16816<true>(st.o[mt], a, b0l, b1l);
    }
  } else {
    // thread (r, c) reads head-dim bytes 16r .. 16r+15 of keys tA, tB, 8+tA,
    // 8+tB; tile mt row r is head-dim 16r + 2mt, row r + 8 is 16r + 2mt + 1
    const int tk[4] = {tA, tB, 8 + tA, 8 + tB};
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = tk[k];
      v[k] = lds128(v_base + t * 128 + ((r ^ (t & 7)) << 4));
    }
    if (valid_keys < kBS) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (tk[k] >= valid_keys) v[k] = make_uint4(0, 0, 0, 0);
    }
    const uint32_t va[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
    const uint32_t vb[4] = {v[1].x, v[1].y, v[1].z, v[1].w};
    const uint32_t vc[4] = {v[2].x, v[2].y, v[2].z, v[2].w};
    const uint32_t vd[4] = {v[3].x, v[3].y, v[3].z, v[3].w};
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
      const uint32_t ab = __byte_perm(va[mt >> 1], vb[mt >> 1], sel);
      const uint32_t cd = __byte_perm(vc[mt >> 1], vd[mt >> 1], sel);
      uint32_t a[4];
      e4m3x4_to_f16x2x2(ab, a[0], a[1]);
      e4m3x4_to_f16x2x2(cd, a[2], a[3]);
      mma16816<false>(st.o[mt], a, b0, b1);
    }
  }
}

template <typename TOut>
__device__ __forceinline__ void store_out(void* out, int64_t idx, float v) {
  static_cast<TOut*>(out)[idx] = from_f32<TOut>(v);
}

template <int kKind>
using OutT = typename std::conditional<Traits<kKind>::kQBF16, __nv_bfloat16,
                                       __half>::type;

// Shared-memory carve-up of one CTA (offsets from a 1024-aligned base).
template <int kKind, bool kWide>
struct Layout {
  using Tr = Traits<kKind>;
  static constexpr int kE = kWide ? 4 : 2;  // accumulator rows kept per lane
  // (the narrow state, 8 tiles x 4 per lane, has the size of 16 x 2)
  static constexpr int kRing = 0;
  static constexpr int kScratch = Tr::kRingBytes;                 // partial O
  static constexpr int kScratchBytes = kConsumerWarps * 16 * kE * 32 * 4;
  static constexpr int kML = kScratch + kScratchBytes;            // m, l
  static constexpr int kMLBytes = kConsumerWarps * 16 * 2 * 4;
  static constexpr int kBars = kML + kMLBytes;                    // 8 B each
  static constexpr int kNumBars = 2 * Tr::kStages;
  static constexpr int kIds = kBars + 8 * kNumBars;               // int [2][32]
  static constexpr int kAbort = kIds + 2 * 32 * 4;
  // narrow kernel: the CTA's own plan (per-request decode offset, pages,
  // rows) and scan scratch
  static constexpr int kPlan = kAbort + 16;
  static constexpr int kMaxSeqs = kWide ? kSelfPlanMaxSeqsWide : kSelfPlanMaxSeqs;
  static constexpr int kPlanBytes = kMaxSeqs * 16;
  static constexpr int kScan = kPlan + kPlanBytes;
  static constexpr int kScanBytes = 34 * 8;
  static constexpr int kBytes = kScan + kScanBytes;
  static constexpr int kSmemBytes = 1024 + kBytes;  // + alignment slack
};

struct Smem {
  uint32_t base;          // shared address, 1024-aligned
  uint8_t* ptr;           // generic pointer to the same byte
  int stages;
  __device__ uint32_t full(int s) const { return bars + 8 * s; }
  __device__ uint32_t empty(int s) const { return bars + 8 * (stages + s); }
  uint32_t bars;
  int* ids;
  volatile int* abort_flag;
  float* scratch;
  float* ml;
};

__device__ __forceinline__ void mbar_arrive_cnt(uint32_t bar, uint32_t cnt) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   bar),
               "r"(cnt)
               : "memory");
}

__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Barrier of the consumer warps that also ORs a predicate over all of them,
// so that every consumer takes the same decision.
__device__ __forceinline__ bool consumers_sync_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(kConsumerWarps * 32)
      : "memory");
  return r != 0;
}

// Geometry of a work item: its pages and its query rows.
struct ItemGeom {
  int page0, npages, row0, rows;
};

// rec0 = {request, KV head, kind, tile (prefill) or partial slot (decode,
// -1: write the output)}, rec1 = {first page, end page, query rows}
__device__ __forceinline__ ItemGeom item_geom(const FastParams& p,
                                              const int4& rec0,
                                              const int4& rec1,
                                              const ReqMeta& rm) {
  ItemGeom ig;
  ig.page0 = rec1.x;
  ig.npages = rec1.y - rec1.x;
  (void)rm;
  ig.rows = rec1.z;
  ig.row0 = rec0.z == kItemDecode ? 0 : rec0.w * kPrefillTileRows;
  return ig;
}

// One consumer warp's share of one work item.  Pages are numbered by the
// CTA-wide counter c0 + j; in a decode item page c goes to warp c % W (the
// same warp for a given ring slot, since the ring depth is a multiple of W),
// in a prefill tile every warp reads every page for its own 16 rows.
template <int kKind, bool kRows16, bool kWide>
__device__ void consume_item(const FastParams& p, const Smem& sm,
                             const ReqMeta& rm, int r, int g, int kind, int x,
                             const ItemGeom& ig, uint32_t c0, int warp,
                             int lane) {
  using Tr = Traits<kKind>;
  using Ly = Layout<kKind, kWide>;
  constexpr int S = Tr::kStages;
  const int rq = lane >> 2, c = lane & 3;
  const int G = p.group;
  const bool decode = kind == kItemDecode;
  const int wrow0 = decode ? 0 : ig.row0 + 16 * warp;
  const int wrows = decode ? ig.rows : max(0, min(16, ig.rows - 16 * warp));
  uint32_t qa[8][4];
  float rscale[2];
  load_q<kKind, kRows16>(p, rm.q0, g, wrow0, wrows, lane, qa, rscale);
  int lim[2];
  int my_min = INT_MAX, my_max = -1;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int rr = rq + 8 * half;
    lim[half] = rm.L - 1;
    if (rr < wrows) {
      lim[half] = rm.L - rm.n + (wrow0 + rr) / G;
      my_min = min(my_min, lim[half]);
      my_max = max(my_max, lim[half]);
    }
  }
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    my_min = min(my_min, __shfl_xor_sync(~0u, my_min, d));
    my_max = max(my_max, __shfl_xor_sync(~0u, my_max, d));
  }
  const int min_lim = min(my_min, rm.L - 1);
  // keys at or below this are outside some row's window
  const int win_edge = my_max - p.window;
  const float ss0 = p.score_scale * rscale[0];
  const float ss1 = p.score_scale * rscale[1];

  WarpState st;
#pragma unroll
  for (int T = 0; T < 16; ++T)
    st.o[T][0] = st.o[T][1] = st.o[T][2] = st.o[T][3] = 0.f;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.f;

  const int first =
      decode ? (int)((warp - (int)(c0 % kConsumerWarps) + kConsumerWarps) %
                     kConsumerWarps)
             : 0;
  const int stride = decode ? kConsumerWarps : 1;
  bool alive = *sm.abort_flag == 0;
  for (int j = first; j < ig.npages && alive; j += stride) {
    const uint32_t cc = c0 + j;
    const int slot = cc % S;
    if (!__all_sync(~0u, mbar_wait_bounded(sm.full(slot), (cc / S) & 1))) {
      if (lane == 0) {
        flag_error(p.err, PA_DEV_ERR_TIMEOUT);
        *sm.abort_flag = 1;
      }
      alive = false;
      break;
    }
    const int key0 = (ig.page0 + j) * kBS;
    const int valid = min(kBS, rm.L - key0);
    const bool need_mask = key0 + kBS - 1 > min_lim || key0 <= win_edge;
    const uint32_t kb = sm.base + Ly::kRing + slot * Tr::kStageBytes;
    process_page<kKind, kRows16>(kb, kb + Tr::kPageBytes, qa, st, key0, valid,
                                 need_mask, lim[0], lim[1], p.window, ss0, ss1,
                                 lane);
    __syncwarp();
    if (lane == 0) mbar_arrive_cnt(sm.empty(slot), decode ? kConsumerWarps : 1);
  }
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    st.l[half] += __shfl_xor_sync(~0u, st.l[half], 1);
    st.l[half] += __shfl_xor_sync(~0u, st.l[half], 2);
  }
  const int Hq = p.num_q_heads;
  constexpr int kE = kRows16 ? 4 : 2;

  if (!decode) {
#pragma unroll
    for (int T = 0; T < 16; ++T)
#pragma unroll
      for (int e = 0; e < kE; ++e) {
        const int rr = rq + (e >> 1) * 8;
        if (rr >= wrows) continue;
        const int R = wrow0 + rr;
        const int i = R / G;
        const int h = g * G + (R - i * G);
        const float v = st.o[T][e] / st.l[e >> 1] * p.out_scale;
        store_out<OutT<kKind>>(p.out,
                               ((int64_t)(rm.q0 + i) * Hq + h) * 128 +
                                   out_col<kKind>(T, e, c),
                               v);
      }
    return;
  }

  // decode item: merge the four warps' partial states in shared memory (the
  // scratch is free: every warp passed the item-start barrier after its last
  // read of it)
  float* of = sm.scratch;
  float* ml = sm.ml;
#pragma unroll
  for (int T = 0; T < 16; ++T)
#pragma unroll
    for (int e = 0; e < kE; ++e)
      of[((warp * 16 + T) * Ly::kE + e) * 32 + lane] = st.o[T][e];
  if (c == 0) {
    ml[(warp * 16 + rq) * 2 + 0] = st.m[0];
    ml[(warp * 16 + rq) * 2 + 1] = st.l[0];
    if (kRows16) {
      ml[(warp * 16 + rq + 8) * 2 + 0] = st.m[1];
      ml[(warp * 16 + rq + 8) * 2 + 1] = st.l[1];
    }
  }
  consumers_sync();
  const int slot = x;  // partial slot, -1: this item covers the whole segment
#pragma unroll
  for (int Tq = 0; Tq < 16 / kConsumerWarps; ++Tq) {
    const int T = warp * (16 / kConsumerWarps) + Tq;
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      const int rr = rq + (e >> 1) * 8;
      if (rr >= wrows) continue;
      float mw[kConsumerWarps], M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        mw[w] = ml[(w * 16 + rr) * 2];
        M = fmaxf(M, mw[w]);
      }
      float num = 0.f, den = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float a = mw[w] == -INFINITY ? 0.f : exp2f(mw[w] - M);
        num += a * of[((w * 16 + T) * Ly::kE + e) * 32 + lane];
        den += a * ml[(w * 16 + rr) * 2 + 1];
      }
      const int i = rr / G;
      const int h = g * G + (rr - i * G);
      const int64_t row = (int64_t)(rm.q0 + i) * Hq + h;
      const int col = out_col<kKind>(T, e, c);
      if (slot < 0) {
        store_out<OutT<kKind>>(p.out, row * 128 + col, num / den * p.out_scale);
      } else {
        const int64_t pr = (int64_t)slot * 16 + rr;
        p.ws_acc[pr * 128 + col] = num;
        if (T == 0 && (e & 1) == 0 && c == 0) {
          p.ws_ml[pr * 2 + 0] = M;
          p.ws_ml[pr * 2 + 1] = den;
        }
      }
    }
  }
}

// One consumer warp's share of a decode item with at most 8 query rows
// (pages c0 + j with (c0 + j) % W == warp), merged across the W warps in
// shared memory at the end.
template <int kKind, bool kWide>
__device__ void consume_item_narrow(const FastParams& p, const Smem& sm,
                                    const ReqMeta& rm, int r, int g, int x,
                                    const ItemGeom& ig, uint32_t c0, int warp,
                                    int lane) {
  using Tr = Traits<kKind>;
  using Ly = Layout<kKind, kWide>;
  constexpr int S = Tr::kStages;
  const int rq = lane >> 2, c = lane & 3;
  const int G = p.group;
  const int rows = ig.rows;
  uint32_t qa[8][4];
  float rscale[2];
  load_q<kKind, false>(p, rm.q0, g, 0, rows, lane, qa, rscale);
  const int lim = rq < rows ? rm.L - rm.n + rq / G : rm.L - 1;
  int min_lim = rq < rows ? lim : INT_MAX;
  int max_lim = rq < rows ? lim : -1;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    min_lim = min(min_lim, __shfl_xor_sync(~0u, min_lim, d));
    max_lim = max(max_lim, __shfl_xor_sync(~0u, max_lim, d));
  }
  min_lim = min(min_lim, rm.L - 1);
  // keys at or below this are outside some row's window
  const int win_edge = max_lim - p.window;
  const float ss = p.score_scale * rscale[0];

  NarrowState st;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
    st.o[mt][0] = st.o[mt][1] = st.o[mt][2] = st.o[mt][3] = 0.f;
  st.m = -INFINITY;
  st.l = 0.f;

  const int first = (int)((warp - (int)(c0 % kConsumerWarps) + kConsumerWarps) %
                          kConsumerWarps);
  bool alive = *sm.abort_flag == 0;
  for (int j = first; j < ig.npages && alive; j += kConsumerWarps) {
    const uint32_t cc = c0 + j;
    const int slot = cc % S;
    if (!__all_sync(~0u, mbar_wait_bounded(sm.full(slot), (cc / S) & 1))) {
      if (lane == 0) {
        flag_error(p.err, PA_DEV_ERR_TIMEOUT);
        *sm.abort_flag = 1;
      }
      alive = false;
      break;
    }
    const int key0 = (ig.page0 + j) * kBS;
    const int valid = min(kBS, rm.L - key0);
    const bool need_mask = key0 + kBS - 1 > min_lim || key0 <= win_edge;
    const uint32_t kb = sm.base + Ly::kRing + slot * Tr::kStageBytes;
    process_page_narrow<kKind>(kb, kb + Tr::kPageBytes, qa, st, key0, valid,
                               need_mask, lim, p.window, ss, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive_cnt(sm.empty(slot), kConsumerWarps);
  }
  st.l += __shfl_xor_sync(~0u, st.l, 1);
  st.l += __shfl_xor_sync(~0u, st.l, 2);

  // merge the four warps' states (scratch free since the item-start barrier)
  float* of = sm.scratch;  // [warp][mt][e][lane]
  float* ml = sm.ml;       // [warp][16 rows][m, l]
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      of[((warp * 8 + mt) * 4 + e) * 32 + lane] = st.o[mt][e];
  if (c == 0) {
    ml[(warp * 16 + rq) * 2 + 0] = st.m;
    ml[(warp * 16 + rq) * 2 + 1] = st.l;
  }
  consumers_sync();
  const int slot = x;  // partial slot, -1: this item covers the whole segment
  const int Hq = p.num_q_heads;
#pragma unroll
  for (int k = 0; k < 8 / kConsumerWarps; ++k) {
    const int mt = warp * (8 / kConsumerWarps) + k;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int qrow = 2 * c + (e & 1);
      if (qrow >= rows) continue;
      float mw[kConsumerWarps], M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        mw[w] = ml[(w * 16 + qrow) * 2];
        M = fmaxf(M, mw[w]);
      }
      float num = 0.f, den = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float a = mw[w] == -INFINITY ? 0.f : exp2f(mw[w] - M);
        num += a * of[((w * 8 + mt) * 4 + e) * 32 + lane];
        den += a * ml[(w * 16 + qrow) * 2 + 1];
      }
      const int i = qrow / G;
      const int h = g * G + (qrow - i * G);
      const int64_t orow = (int64_t)(rm.q0 + i) * Hq + h;
      const int col = narrow_col<kKind>(mt, e, rq);
      if (slot < 0) {
        store_out<OutT<kKind>>(p.out, orow * 128 + col, num / den * p.out_scale);
      } else {
        const int64_t pr = (int64_t)slot * 16 + qrow;
        p.ws_acc[pr * 128 + col] = num;
        if (mt == 0 && (e >> 1) == 0 && rq == 0) {
          p.ws_ml[pr * 2 + 0] = M;
          p.ws_ml[pr * 2 + 1] = den;
        }
      }
    }
  }
}

// Where a CTA's work items come from: the planner's list, or (decode-only
// steps, self_plan) the CTA's own stream-K range over the per-request page
// prefix it computed in its prologue.  Every warp of the CTA keeps its own
// copy and draws the same sequence.
struct ItemSource {
  // planner list
  const int4* items;
  int k, end;
  // own range
  bool self;
  const long long* dec0;
  const int* declen;
  const int* rows;
  long long cur, lo, hi;
  int r, B, H, b;
  // cascade steps: pages start after the shared prefix, and an uncut piece
  // goes to its own slot (the merge adds the prefix's part)
  bool casc;
  int pg_off;
  int64_t unc_slot0;

  __device__ bool next(int4& rec0, int4& rec1) {
    if (!self) {
      if (k >= end) return false;
      rec0 = __ldg(items + 2 * k);
      rec1 = __ldg(items + 2 * k + 1);
      ++k;
      return true;
    }
    if (cur >= hi) return false;
    while (r < B && declen[r] == 0) ++r;
    if (r >= B) return false;
    const long long rs = dec0[r];
    const int dl = declen[r];  // segment length on the line: kSegCost + pages
    const int g = (int)((cur - rs) / dl);
    const long long ss = rs + (long long)g * dl, se = ss + dl;
    const long long pe = se < hi ? se : hi;
    // pages of the piece (its line range minus the segment's leading cost
    // units; a piece inside those units has none and writes an empty part)
    const long long p0 = ss + kSegCost;
    const int pg_begin = (int)(cur > p0 ? cur - p0 : 0);
    const int pg_end = (int)(pe > p0 ? pe - p0 : 0);
    // a piece that continues a segment begun in an earlier range is this
    // CTA's "head" part (slot 2b); one that continues into a later range is
    // its "tail" part (slot 2b + 1)
    const bool before = cur == lo && ss < lo;
    const bool after = pe == hi && se > hi;
    const int slot = before ? 2 * b
                            : (after ? 2 * b + 1 : (casc ? (int)(unc_slot0 + r * H + g) : -1));
    rec0 = make_int4(r, g, kItemDecode, slot);
    rec1 = make_int4(pg_begin + pg_off, pg_end + pg_off, rows[r], 0);
    cur = pe;
    if (pe == se && g + 1 == H) ++r;
    return true;
  }
};

// Per-request decode segments of the step and their prefix on the cost line
// (per segment kSegCost + its key pages; one segment per KV head, or per
// group of KV heads) into shared memory; all threads of the block take part.
// Returns the total.  Requests with invalid metadata contribute nothing.
__device__ long long plan_prefix(const FastParams& p, long long* dec0,
                                 int* declen, int* rows, long long* scan_tot,
                                 long long* scan_ws) {
  long long run = 0;
  for (int base = 0; base < p.num_seqs; base += blockDim.x) {
    const int r = base + threadIdx.x;
    int dl = 0, rw = 0;
    if (r < p.num_seqs) {
      const ReqMeta m = load_req(p.qsl, p.seq_lens, r, p.num_tokens,
                                 p.max_query_len, p.max_seq_len,
                                 p.max_blocks_per_seq);
      if (m.ok && m.n > 0 && m.n * p.group <= p.dec_rows_max) {
        dl = kSegCost + m.nb - p.cascade_blocks;
        rw = m.n * p.group;
        // a cascade step's shared prefix must lie before the queries
        if (p.cascade_blocks > 0 && m.L - m.n < p.cascade_blocks * kBS) {
          if (blockIdx.x == 0) flag_error(p.err, PA_DEV_ERR_METADATA);
          dl = rw = 0;
        }
      } else if (!m.ok && blockIdx.x == 0) {
        flag_error(p.err, PA_DEV_ERR_METADATA);
      }
    }
    const long long ex =
        block_scan_excl<long long>((long long)dl * (p.num_kv_heads / p.seg_heads),
                                   scan_tot, scan_ws);
    const long long tot = *scan_tot;
    __syncthreads();
    if (r < p.num_seqs) {
      dec0[r] = run + ex;
      declen[r] = dl;
      rows[r] = rw;
    }
    run += tot;
  }
  __syncthreads();
  return run;
}

__device__ __forceinline__ int self_plan_grid(long long C, int grid) {
  long long g = C / kMinUnitsPerCta;
  if (g > grid) g = grid;
  if (g < 1) g = 1;
  return (int)g;
}

// first request whose decode range holds unit u (skipping empty requests)
__device__ __forceinline__ int request_of(const long long* dec0, int B,
                                          long long u) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (dec0[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// kWide = false: every work item has at most 8 query rows (decode steps with
// q_len * group <= 8) -- half the accumulators.
// kWide = true: any item (up to 16 rows per warp, prefill tiles).
//
// Persistent: each CTA claims work items from a device-wide counter until
// none are left.  Warp 4 (producer) claims items, publishes them through a
// small shared-memory queue and streams their pages into the ring; warps 0-3
// consume.  The ring keeps streaming across item boundaries.
template <int kKind, bool kWide>
__global__ void __launch_bounds__(kThreads, PA_CTAS_PER_SM)
attn_fast_kernel(const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v,
                 const __grid_constant__ FastParams p) {
  using Tr = Traits<kKind>;
  using Ly = Layout<kKind, kWide>;
  constexpr int S = Tr::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  Smem sm;
  sm.base = (raw + 1023u) & ~1023u;
  sm.ptr = smem_raw + (sm.base - raw);
  sm.stages = S;
  sm.bars = sm.base + Ly::kBars;
  sm.ids = reinterpret_cast<int*>(sm.ptr + Ly::kIds);
  sm.abort_flag = reinterpret_cast<volatile int*>(sm.ptr + Ly::kAbort);
  sm.scratch = reinterpret_cast<float*>(sm.ptr + Ly::kScratch);
  sm.ml = reinterpret_cast<float*>(sm.ptr + Ly::kML);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(sm.full(i), 1);
      mbar_init(sm.empty(i), kConsumerWarps);
    }
    *sm.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();               // the planner (and everything before it) is done
  // the merge may be scheduled behind this grid; it reads the step's
  // metadata before its own wait, which is safe from here on
  pdl_launch_dependents();
  ItemSource src{};
  src.self = false;
  {
    if (p.self_plan) {
      long long* dec0 = reinterpret_cast<long long*>(sm.ptr + Ly::kPlan);
      int* declen = reinterpret_cast<int*>(dec0 + Ly::kMaxSeqs);
      int* rows = declen + Ly::kMaxSeqs;
      long long* scan = reinterpret_cast<long long*>(sm.ptr + Ly::kScan);
      const long long C = plan_prefix(p, dec0, declen, rows, scan + 32, scan);
      const int g_eff = self_plan_grid(C, gridDim.x);
      src.self = true;
      src.dec0 = dec0;
      src.declen = declen;
      src.rows = rows;
      src.B = p.num_seqs;
      src.H = p.num_kv_heads / p.seg_heads;
      src.b = blockIdx.x;
      src.lo = src.hi = 0;
      if ((int)blockIdx.x < g_eff && C > 0) {
        src.lo = (long long)blockIdx.x * C / g_eff;
        src.hi = (long long)(blockIdx.x + 1) * C / g_eff;
      }
      src.cur = src.lo;
      src.r = p.num_seqs > 0 ? request_of(dec0, p.num_seqs, src.lo) : 0;
    }
  }
  if (!src.self) {
    src.items = p.items;
    src.k = __ldg(p.cta_begin + blockIdx.x);
    src.end = __ldg(p.cta_begin + blockIdx.x + 1);
  }

  if (warp == kConsumerWarps) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
    }
    uint32_t c = 0;     // pages issued
    int go = 1;
    int4 rec0, rec1;
    while (go && src.next(rec0, rec1)) {
      // the narrow kernel never gets prefill tiles or items over 8 rows (the
      // host guarantees it); both sides skip them the same way
      if (!kWide && (rec0.z == kItemPrefill || rec1.z > 8)) continue;
      const int32_t* bt =
          p.block_tables + (int64_t)rec0.x * p.max_blocks_per_seq + rec1.x;
      // Block ids go through shared memory 32 at a time (the next chunk is
      // loaded while the current one is issued).  Lanes 0 and 1 issue each
      // page together: lane 0 its K page and the expected byte count, lane
      // 1 its V page.
      const int n = rec1.y - rec1.x;
      sm.ids[lane] = lane < n ? __ldg(bt + lane) : 0;
      __syncwarp();
      for (int j0 = 0; j0 < n && go; j0 += 32) {
        const int buf = (j0 >> 5) & 1;
        const int nidx = j0 + 32 + lane;
        const int nreg = nidx < n ? __ldg(bt + nidx) : 0;
        // lanes 2k and 2k+1 issue page j + k of each group of PP pages (PP
        // distinct ring slots)
        constexpr int PP = PA_PRODUCER_PAGES;
        static_assert(PP <= S, "pages per producer step exceed the ring");
        constexpr unsigned kMask = (PP >= 16) ? 0xFFFFFFFFu : ((1u << (2 * PP)) - 1u);
        if (lane < 2 * PP) {
          const int* cur = sm.ids + buf * 32;
          const int cnt = min(32, n - j0);
          const int kk = lane >> 1;        // page within the group
          const int kv = lane & 1;         // 0: K page, 1: V page
          const CUtensorMap* map = kv ? &tmap_v : &tmap_k;
          for (int jj = 0; jj < cnt; jj += PP) {
            const bool mine = jj + kk < cnt;
            const uint32_t cc = c + kk;
            const int slot = cc % S;
            const bool ok = !mine || cc < (uint32_t)S ||
                            mbar_wait_bounded(sm.empty(slot), ((cc / S) - 1) & 1);
            if (__any_sync(kMask, !ok)) {
              if (lane == 0) {
                flag_error(p.err, PA_DEV_ERR_TIMEOUT);
                *sm.abort_flag = 1;
              }
              go = 0;
              break;
            }
            if (mine) {
              int blk = cur[jj + kk];
              if (blk < 0 || (int64_t)blk >= p.num_blocks) {
                if (kv == 0) flag_error(p.err, PA_DEV_ERR_BLOCK_ID);
                blk = 0;
              }
              const int row = (blk * p.num_kv_heads + rec0.y) * kBS;
              const uint32_t dst =
                  sm.base + Ly::kRing + slot * Tr::kStageBytes + kv * Tr::kPageBytes;
              if (kv == 0) mbar_arrive_expect_tx(sm.full(slot), Tr::kStageBytes);
              __syncwarp(__activemask());
              if constexpr (Tr::kFp8)
                tma_load_2d(dst, map, sm.full(slot), 0, row);
              else
                tma_load_3d(dst, map, sm.full(slot), 0, 0, row);
            }
            c += min(PP, cnt - jj);
          }
        }
        __syncwarp();
        go = __shfl_sync(~0u, go, 0);
        c = __shfl_sync(~0u, c, 0);
        sm.ids[(buf ^ 1) * 32 + lane] = nreg;
        __syncwarp();
      }
    }
    // after an abort, let the copies already in flight land before exiting
    if (!go && lane == 0) {
      const uint32_t from = c > (uint32_t)S ? c - S : 0;
      for (uint32_t i = from; i < c; ++i)
        mbar_wait_bounded(sm.full(i % S), (i / S) & 1);
    }
    return;
  }

  // ------------------------------ consumers -------------------------------
  uint32_t c = 0;  // pages consumed (CTA-wide numbering, as issued)
  int4 rec0, rec1;
  while (src.next(rec0, rec1)) {
    // every consumer warp meets here once per item: decisions below are
    // uniform, the previous item's shared scratch is no longer read, and all
    // earlier pages have been consumed by their owners
    if (consumers_sync_any(*sm.abort_flag != 0)) break;
    const ReqMeta rm = load_req(p.qsl, p.seq_lens, rec0.x, p.num_tokens,
                                p.max_query_len, p.max_seq_len,
                                p.max_blocks_per_seq);
    const ItemGeom ig = item_geom(p, rec0, rec1, rm);
    if (!kWide && (rec0.z == kItemPrefill || rec1.z > 8)) {
      if (threadIdx.x == 0) flag_error(p.err, PA_DEV_ERR_METADATA);
      continue;
    }
    if (rec0.z == kItemDecode && ig.rows <= 8) {
      consume_item_narrow<kKind, kWide>(p, sm, rm, rec0.x, rec0.y, rec0.w, ig,
                                        c, warp, lane);
    } else if constexpr (kWide) {
      consume_item<kKind, true, true>(p, sm, rm, rec0.x, rec0.y, rec0.z,
                                      rec0.w, ig, c, warp, lane);
    } else {
      // the host never sends such an item to the narrow kernel
      if (threadIdx.x == 0) flag_error(p.err, PA_DEV_ERR_METADATA);
      continue;
    }
    c += ig.npages;
  }
}

// ---------------------------------------------------------------------------
// split-K merge: CTA k finishes split segment k (request r, KV head g): one
// warp per query row, parts combined in slot order (deterministic)
template <typename TOut>
__global__ void __launch_bounds__(128)
merge_kernel(FastParams p) {
  pdl_wait();  // the attention grid has finished writing the parts
  if ((int)blockIdx.x >= min(*p.n_split, p.max_slots)) return;
  const int4 sg = p.split_list[blockIdx.x];
  const int r = sg.x, g = sg.y, parts = sg.z, first = sg.w;
  const int lane = threadIdx.x & 31;
  const ReqMeta rm = load_req(p.qsl, p.seq_lens, r, p.num_tokens, p.max_query_len,
                              p.max_seq_len, p.max_blocks_per_seq);
  const int rows = rm.n * p.group;
  for (int rr = threadIdx.x >> 5; rr < rows; rr += blockDim.x >> 5) {
    const int i = rr / p.group;
    const int h = g * p.group + (rr - i * p.group);
    const int64_t row = (int64_t)(rm.q0 + i) * p.num_q_heads + h;
    float M = -INFINITY;
    for (int s = lane; s < parts; s += 32)
      M = fmaxf(M, p.ws_ml[((int64_t)(first + s) * 16 + rr) * 2]);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) M = fmaxf(M, __shfl_xor_sync(~0u, M, d));
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float den = 0.f;
    for (int s = 0; s < parts; ++s) {
      const int64_t pr = (int64_t)(first + s) * 16 + rr;
      const float ms = p.ws_ml[pr * 2];
      if (ms == -INFINITY) continue;  // a part with no keys
      const float w = exp2f(ms - M);
      den += w * p.ws_ml[pr * 2 + 1];
      const float4 v = *reinterpret_cast<const float4*>(p.ws_acc + pr * 128 + 4 * lane);
      acc[0] += w * v.x;
      acc[1] += w * v.y;
      acc[2] += w * v.z;
      acc[3] += w * v.w;
    }
    const float inv = p.out_scale / den;
    TOut* o = static_cast<TOut*>(p.out) + row * 128 + 4 * lane;
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = from_f32<TOut>(acc[k] * inv);
  }
}

// Split-K merge of a self-planned decode step: CTA b looks at the range
// boundary b; if it cuts a segment, the CTA merges its share of that
// segment's rows from the segment's parts, combined in a fixed order.
#ifndef PA_MERGE_THREADS
#define PA_MERGE_THREADS 256
#endif
constexpr int kMergeThreads = PA_MERGE_THREADS;  // merge_self_kernel CTA

// (at most 64 registers a thread: a merge CTA fits beside the two decode
// CTAs of an SM, so that its plan runs while the attention kernel does)
// kCasc: a cascade step (p.cascade_blocks > 0); the plain steps' build has
// none of the cascade's code
template <typename TOut, bool kCasc>
__global__ void __launch_bounds__(kMergeThreads, 4)
merge_self_kernel(FastParams p) {
  extern __shared__ long long mplan[];
  __shared__ long long scan[34];
  // The plan needs only the step's metadata, complete before the attention
  // grid let this grid start: it overlaps the attention kernel.
  long long* dec0 = mplan;
  int* declen = reinterpret_cast<int*>(dec0 + p.num_seqs);
  int* rows = declen + p.num_seqs;
  const long long C = plan_prefix(p, dec0, declen, rows, scan + 32, scan);
  const int g_eff = self_plan_grid(C, p.attn_grid);
  if (C <= 0) return;
  const int lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int D = p.head_dim;
  const bool act = 4 * lane < D;  // lanes holding 4 of the row's D columns
  // rows of every KV head of a segment (one head, or a head group whose
  // partial slots hold kHg x 8 rows)
  const int sh = p.seg_heads;
  const int part_rows = sh == 1 ? 16 : kHgPartRows;
  if constexpr (kCasc) {
    // a cascade step's requests all start with request 0's first
    // cascade_blocks block-table entries (checked while the attention runs)
    const int64_t total = (int64_t)p.num_seqs * p.cascade_blocks;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total;
         x += (int64_t)gridDim.x * blockDim.x) {
      const int r = (int)(x / p.cascade_blocks);
      const int j = (int)(x - (int64_t)r * p.cascade_blocks);
      if (r > 0 && __ldg(p.block_tables + (int64_t)r * p.max_blocks_per_seq + j) !=
                       __ldg(p.block_tables + j))
        flag_error(p.err, PA_DEV_ERR_METADATA);
    }
  }
  // One output row from np partial rows (row_of(s): row index into ws_acc /
  // ws_ml), combined in part order: M = max m_s, out = sum 2^(m_s - M) acc_s
  // / sum 2^(m_s - M) l_s.  A part with m = -inf has no visible key.
  auto combine = [&](int np, auto row_of, int64_t orow) {
    float M = -INFINITY, den = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (np <= 32) {
      // lane s holds part s's (m, l): one round trip gives M and the
      // denominator; the weights go round by shuffle, so the numerator's
      // loads are independent of each other.  The first four parts' rows
      // are loaded together with (m, l).
      float4 vpre[4];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        vpre[s] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s < np && act)
          vpre[s] = __ldg(reinterpret_cast<const float4*>(p.ws_acc + row_of(s) * D) + lane);
      }
      float ms = -INFINITY, ls = 0.f;
      if (lane < np) {
        const float2 ml = __ldg(reinterpret_cast<const float2*>(p.ws_ml) + row_of(lane));
        ms = ml.x;
        ls = ml.y;
      }
      M = ms;
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) M = fmaxf(M, __shfl_xor_sync(~0u, M, d));
      const float w = ms == -INFINITY ? 0.f : exp2f(ms - M);
      den = w * ls;
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) den += __shfl_xor_sync(~0u, den, d);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const float wgt = __shfl_sync(~0u, w, s);
        if (s < np) {
          acc[0] += wgt * vpre[s].x;
          acc[1] += wgt * vpre[s].y;
          acc[2] += wgt * vpre[s].z;
          acc[3] += wgt * vpre[s].w;
        }
      }
#pragma unroll 4
      for (int s = 4; s < np; ++s) {
        const float wgt = __shfl_sync(~0u, w, s);
        const float4 v = act ? __ldg(reinterpret_cast<const float4*>(p.ws_acc + row_of(s) * D) + lane)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        acc[0] += wgt * v.x;
        acc[1] += wgt * v.y;
        acc[2] += wgt * v.z;
        acc[3] += wgt * v.w;
      }
    } else {
      // M and the denominator with the parts spread over the lanes
      for (int s = lane; s < np; s += 32) M = fmaxf(M, __ldg(p.ws_ml + row_of(s) * 2));
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) M = fmaxf(M, __shfl_xor_sync(~0u, M, d));
      for (int s = lane; s < np; s += 32) {
        const int64_t pr = row_of(s);
        const float ms = __ldg(p.ws_ml + pr * 2);
        if (ms != -INFINITY) den += exp2f(ms - M) * __ldg(p.ws_ml + pr * 2 + 1);
      }
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) den += __shfl_xor_sync(~0u, den, d);
      // the numerator in part order, loads of several parts in flight
#pragma unroll 4
      for (int s = 0; s < np; ++s) {
        const int64_t pr = row_of(s);
        const float ms = __ldg(p.ws_ml + pr * 2);
        const float4 v = act ? __ldg(reinterpret_cast<const float4*>(p.ws_acc + pr * D) + lane)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        const float wgt = ms == -INFINITY ? 0.f : exp2f(ms - M);
        acc[0] += wgt * v.x;
        acc[1] += wgt * v.y;
        acc[2] += wgt * v.z;
        acc[3] += wgt * v.w;
      }
    }
    const float inv = p.out_scale / den;
    TOut* o = static_cast<TOut*>(p.out) + orow * D + 4 * lane;
    if (act) {
#pragma unroll
      for (int k = 0; k < 4; ++k) o[k] = from_f32<TOut>(acc[k] * inv);
    }
  };
  // the output row of segment row rr (kv head w of the segment's group)
  struct SegRow {
    int prow;
    int64_t row;
  };
  auto seg_row = [&](int g, int x, int nrows, int q0) -> SegRow {
    const int w = x / nrows, rr = x - w * nrows;
    const int i = rr / p.group;
    const int h = (g * sh + w) * p.group + (rr - i * p.group);
    return SegRow{sh == 1 ? rr : w * 8 + rr, (int64_t)(q0 + i) * p.num_q_heads + h};
  };
  // the prefix's parts (one per key range, in range order) come first
  const int c0 = kCasc ? p.casc_splits : 0;
  // this CTA takes range boundaries blockIdx.x, + gridDim.x, ...
  for (int b = blockIdx.x; b < g_eff; b += gridDim.x) {
    if (b == 0) continue;
    const long long lo_b = (long long)b * C / g_eff;
    int r = request_of(dec0, p.num_seqs, lo_b);
    while (r < p.num_seqs && declen[r] == 0) ++r;
    if (r >= p.num_seqs) continue;
    const int dl = declen[r];
    const int g = (int)((lo_b - dec0[r]) / dl);
    const long long ss = dec0[r] + (long long)g * dl, se = ss + dl;
    if (ss >= lo_b) continue;  // boundary b does not cut a segment
    // the boundaries that cut this segment: b0 .. b1-1.  Its parts, in order:
    // (cascade steps: the shared prefix's,) the tail piece of range b0-1
    // (slot 2(b0-1)+1), then the head pieces of ranges b0 .. b1-1 (slots
    // 2k).  The b1-b0 CTAs of these boundaries share the segment's rows.
    int b0 = b;
    while (b0 > 1 && (long long)(b0 - 1) * C / g_eff > ss) --b0;
    int b1 = b + 1;
    while (b1 < g_eff && (long long)b1 * C / g_eff < se) ++b1;
    const int np = 1 + (b1 - b0);
    const ReqMeta rm = load_req(p.qsl, p.seq_lens, r, p.num_tokens, p.max_query_len,
                                p.max_seq_len, p.max_blocks_per_seq);
    pdl_wait();  // the attention grid has finished writing the parts
    const int total = sh * rows[r];
    for (int x = (b - b0) * nwarps + (threadIdx.x >> 5); x < total;
         x += (b1 - b0) * nwarps) {
      const SegRow sr = seg_row(g, x, rows[r], rm.q0);
      const int64_t pr_tail = (int64_t)(2 * (b0 - 1) + 1) * part_rows + sr.prow;
      const int64_t pr_head = (int64_t)(2 * b0) * part_rows + sr.prow;
      const int64_t pr_step = 2 * (int64_t)part_rows;
      const int64_t pr_casc = p.casc_row0 + sr.row;
      combine(np + c0,
              [&](int s) -> int64_t {
                if (s < c0) return pr_casc + s * p.casc_split_rows;
                s -= c0;
                return s == 0 ? pr_tail : pr_head + (s - 1) * pr_step;
              },
              sr.row);
    }
  }  // boundaries
  if constexpr (kCasc) {
    // cascade steps: a segment that no boundary cuts has one part of its
    // own (its uncut slot), merged here after the prefix's
    const int H = p.num_kv_heads / sh;
    const int64_t npairs = (int64_t)p.num_seqs * H;
    for (int64_t x = blockIdx.x; x < npairs; x += gridDim.x) {
      const int r = (int)(x / H), g = (int)(x - (int64_t)r * H);
      if (declen[r] == 0) continue;
      const long long ss = dec0[r] + (long long)g * declen[r], se = ss + declen[r];
      // the range holding unit ss; the segment is cut if the range ends
      // before it does (handled above)
      int k = (int)(ss * g_eff / C);
      while (k + 1 < g_eff && (long long)(k + 1) * C / g_eff <= ss) ++k;
      while (k > 0 && (long long)k * C / g_eff > ss) --k;
      if ((long long)(k + 1) * C / g_eff < se) continue;
      const ReqMeta rm = load_req(p.qsl, p.seq_lens, r, p.num_tokens, p.max_query_len,
                                  p.max_seq_len, p.max_blocks_per_seq);
      pdl_wait();
      const int64_t unc = (p.unc_slot0 + (int64_t)r * H + g) * part_rows;
      for (int y = threadIdx.x >> 5; y < sh * rows[r]; y += nwarps) {
        const SegRow sr = seg_row(g, y, rows[r], rm.q0);
        const int64_t pr_casc = p.casc_row0 + sr.row, pr_unc = unc + sr.prow;
        combine(c0 + 1,
                [&](int s) -> int64_t {
                  return s < c0 ? pr_casc + s * p.casc_split_rows : pr_unc;
                },
                sr.row);
      }
    }
  }
}


// ---------------------------------------------------------------------------
// Decode steps by head groups.  An item is a range of key pages of one
// (request, group of kHg KV heads).  The group's kHg pages of a block lie
// next to each other in the cache, so one TMA box per cache brings all of
// them, and consumer warp w owns KV head kHg * group + w for the whole item:
// its own query rows and softmax state, no merge across warps.  A quarter of
// the TMA instructions per byte of the one-head items; used for steps of
// <= 8-row requests whose KV head count is a multiple of kHg.
// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// 4-bit caches in the head-group decode kernel
//
// Every INT4 and NVFP4 value is exact in f16 (a 4-bit code; an E2M1 value
// times an E4M3 block scale), so the contraction runs on f16 MMAs with q
// widened to f16 as for FP8 caches.  INT4 per-token scales multiply the
// scores (K) and the probabilities (V); NVFP4 block scales multiply the
// decoded pairs; NVFP4's per-tensor scales are folded into the score and
// output scales.
//
// Head-dim order: thread (r, c) supplies dims 32c + 4s .. 32c + 4s + 3 of
// k-step s of Q.K^T (b0 the first two, b1 the last two): the 16-byte chunk
// c of a key's 64 code bytes.  V^T tile mt row r is head dim 16r + 2mt and
// row r + 8 is 16r + 2mt + 1: byte mt of the code bytes 8r .. 8r + 7.
// ---------------------------------------------------------------------------
// Q rows of a narrow item in that order; rows >= nrows are zero.
template <int kKind>
__device__ __forceinline__ void load_q4(const FastParams& p, int q0, int g,
                                        int nrows, int lane,
                                        uint32_t (&qa)[8][4], float& rscale,
                                        float& qbias) {
  using Tr = Traits<kKind>;
  const int r = lane >> 2, c = lane & 3;
  const int G = p.group;
  const bool valid = r < nrows;
  uint32_t w[16];
  if (valid) {
    const int i = r / G, h = g * G + (r - i * G);
    const uint4* src = reinterpret_cast<const uint4*>(
        static_cast<const uint16_t*>(p.q) + ((int64_t)(q0 + i) * p.num_q_heads + h) * 128 +
        32 * c);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = __ldg(src + k);
      w[4 * k] = v.x;
      w[4 * k + 1] = v.y;
      w[4 * k + 2] = v.z;
      w[4 * k + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k) w[k] = 0u;
  }
  rscale = 1.f;
  if constexpr (Tr::kQBF16) {
    // bf16 -> f16 with a per-row power-of-two shift that keeps the row's
    // largest |q| inside the f16 range; the shift is undone on the scores
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w[k] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w[k] & 0xFFFF0000u)));
    }
    amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, 2));
    int e = 0;
    if (amax > 16384.f) e = ilogbf(amax) - 13;
    const float down = exp2f((float)-e);
    rscale = exp2f((float)e);
#pragma unroll
    for (int k = 0; k < 16; ++k)
      w[k] = pack2<false>(__uint_as_float(w[k] << 16) * down,
                          __uint_as_float(w[k] & 0xFFFF0000u) * down);
  }
  if constexpr (Tr::k4 == 1) {
    // INT4: the K decode gives each eight elements as the pairs (0, 4),
    // (1, 5), (2, 6), (3, 7); Q goes in the same order (the dot product is
    // the same sum)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      qa[2 * j][0] = __byte_perm(w[4 * j], w[4 * j + 2], 0x5410);
      qa[2 * j][2] = __byte_perm(w[4 * j], w[4 * j + 2], 0x7632);
      qa[2 * j + 1][0] = __byte_perm(w[4 * j + 1], w[4 * j + 3], 0x5410);
      qa[2 * j + 1][2] = __byte_perm(w[4 * j + 1], w[4 * j + 3], 0x7632);
    }
    // The K decode leaves each code c as its f16 pattern: 1032 + c for an
    // even element (low nibble), 1152 + 16 c for an odd one (high nibble).
    // Q's odd elements are taken / 16 (exact), so that a score comes out as
    // Q.K + 1032 * sum(even q) + 1152 * sum(odd q / 16): that sum, the row's
    // bias, is taken off each score.
    const __half2 sixteenth = __floats2half2_rn(0.0625f, 0.0625f);
    float even = 0.f, odd = 0.f;
#pragma unroll
    for (int st = 0; st < 8; ++st) {
      __half2 h = __hmul2(*reinterpret_cast<const __half2*>(&qa[st][2]), sixteenth);
      qa[st][2] = *reinterpret_cast<uint32_t*>(&h);
      const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&qa[st][0]));
      const float2 o = __half22float2(h);
      even += e.x + e.y;
      odd += o.x + o.y;
    }
    qbias = 1032.f * even + 1152.f * odd;
    qbias += __shfl_xor_sync(~0u, qbias, 1);
    qbias += __shfl_xor_sync(~0u, qbias, 2);
  } else {
#pragma unroll
    for (int st = 0; st < 8; ++st) {
      qa[st][0] = w[2 * st];
      qa[st][2] = w[2 * st + 1];
    }
  }
#pragma unroll
  for (int st = 0; st < 8; ++st) qa[st][1] = qa[st][3] = 0u;
}

// Offset binary of a masked nibble pair under the f16 pattern of 1024 in
// one logic operation: (x ^ 0x8 per nibble) & mask | 0x6400 per half equals
// (x & mask) ^ (0x8 per nibble | 0x6400 per half), the 0x6400 bits lying
// outside the mask.
constexpr uint32_t kNibLo = 0x000F000Fu, kNibLoFlip = 0x64086408u;  // low nibbles
constexpr uint32_t kNibHi = 0x00F000F0u, kNibHiFlip = 0x64806480u;  // high nibbles

// eight INT4 K codes (one word, element 2i in the low nibble of byte i) ->
// the f16 pairs (0, 4), (1, 5), (2, 6), (3, 7): each nibble pair masked in
// place under the f16 pattern of 1024, offset binary code + 8, and left
// there — 1032 + c for a low nibble, 1152 + 16 c for a high one, exact f16
// values; the Q side absorbs the 16, and the offsets become a per-row bias
// taken off the scores (load_q4)
__device__ __forceinline__ void decode8_int4_k(uint32_t w, uint32_t (&f)[4]) {
  const uint32_t y = w >> 8;
  f[0] = (w & kNibLo) ^ kNibLoFlip;
  f[1] = (w & kNibHi) ^ kNibHiFlip;
  f[2] = (y & kNibLo) ^ kNibLoFlip;
  f[3] = (y & kNibHi) ^ kNibHiFlip;
}

// eight 4-bit codes (one word, element 2i in the low nibble of byte i) ->
// four f16 pairs of consecutive elements (exact)
template <int kK4>
__device__ __forceinline__ void decode8(uint32_t w, uint32_t (&f)[4]) {
  if constexpr (kK4 == 1) {
    // two's complement -> offset binary (code + 8), then 1024 + n as f16
    // bits 0x6400 | n, minus 1032
    const uint32_t x = w ^ 0x88888888u;
    const uint32_t y = x >> 4;
    const __half2 off = __floats2half2_rn(1032.f, 1032.f);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      // byte b's low nibble into the low half, its high nibble (the low
      // nibble of byte b of y) into the high half
      const uint32_t t = (__byte_perm(x, y, (uint32_t)(b | ((4 + b) << 8))) & 0x000F000Fu) |
                         0x64006400u;
      __half2 hv = __hsub2(*reinterpret_cast<const __half2*>(&t), off);
      f[b] = *reinterpret_cast<uint32_t*>(&hv);
    }
  } else {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(f[0]), "=r"(f[1]), "=r"(f[2]), "=r"(f[3])
        : "r"(w));
  }
}

// the two E2M1 codes of byte b of w (low nibble first) -> f16 pair (exact);
// b is a constant after unrolling, so the switch folds away
__device__ __forceinline__ uint32_t e2m1x2_byte(uint32_t w, int b) {
  uint32_t r;
  switch (b) {
    case 0:
      asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\t"
          "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t}" : "=r"(r) : "r"(w));
      break;
    case 1:
      asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\t"
          "cvt.rn.f16x2.e2m1x2 %0, b1;\n\t}" : "=r"(r) : "r"(w));
      break;
    case 2:
      asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\t"
          "cvt.rn.f16x2.e2m1x2 %0, b2;\n\t}" : "=r"(r) : "r"(w));
      break;
    default:
      asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\t"
          "cvt.rn.f16x2.e2m1x2 %0, b3;\n\t}" : "=r"(r) : "r"(w));
      break;
  }
  return r;
}

__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a),
                      *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// two E4M3 bytes (low byte first) -> f16 pair
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  asm("{\n\t.reg .b16 l;\n\tcvt.u16.u32 l, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t}"
      : "=r"(r)
      : "r"(two));
  return r;
}

// one 4-bit page (16 keys) of a narrow item
template <int kKind>
__device__ __forceinline__ void process_page_4bit(
    uint32_t k_base, uint32_t v_base, const uint32_t (&qa)[8][4],
    NarrowState& st, int key0, int valid_keys, bool need_mask, int lim,
    int win, float sscale, int lane, float qbias) {
  using Tr = Traits<kKind>;
  constexpr int K4 = Tr::k4;
  constexpr int kCodes = 16 * 64;  // the scales follow the codes
  const int r = lane >> 2, c = lane & 3;
  // ---- S = Q.K^T: key nt * 8 + r, dims 32c .. 32c + 31
  float s[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    float s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
    const int t = nt * 8 + r;
    const uint4 kc = lds128(k_base + t * 64 + c * 16);
    const uint32_t kw[4] = {kc.x, kc.y, kc.z, kc.w};
    uint32_t bsc[2] = {0u, 0u};
    if constexpr (K4 == 2) {
      // block scales of dims 32c .. 32c + 15 and 32c + 16 .. 32c + 31
      uint32_t two;
      asm volatile("ld.shared.u16 %0, [%1];" : "=r"(two) : "r"(k_base + kCodes + t * 8 + 2 * c));
      const uint32_t sp = e4m3x2_to_f16x2(two);
      bsc[0] = __byte_perm(sp, sp, 0x1010);
      bsc[1] = __byte_perm(sp, sp, 0x3232);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t f[4];
      if constexpr (K4 == 1)
        decode8_int4_k(kw[j], f);
      else
        decode8<K4>(kw[j], f);
      if constexpr (K4 == 2) {
#pragma unroll
        for (int q = 0; q < 4; ++q) f[q] = hmul2u(f[q], bsc[j >> 1]);
      }
      mma_acc<false, false>(s[nt], qa[2 * j], f[0], f[1]);
      mma_acc<false, false>(s2, qa[2 * j + 1], f[2], f[3]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) s[nt][e] += s2[e];
  }
  // keys (2c, 2c + 1) of tile nt for row r: INT4 key scales on the scores
  float ks[2][2] = {{1.f, 1.f}, {1.f, 1.f}};
  if constexpr (K4 == 1) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      float2 v;
      asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];"
                   : "=f"(v.x), "=f"(v.y)
                   : "r"(k_base + kCodes + 4 * (nt * 8 + 2 * c)));
      ks[nt][0] = v.x;
      ks[nt][1] = v.y;
    }
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = (K4 == 1 ? s[nt][e] - qbias : s[nt][e]) * (sscale * ks[nt][e]);
      const int key = key0 + nt * 8 + 2 * c + e;
      // keys past the sequence end (their scales may be NaN), past the
      // causal limit or outside the window
      if ((need_mask && (key > lim || key <= lim - win)) || nt * 8 + 2 * c + e >= valid_keys)
        v = -INFINITY;
      s[nt][e] = v;
    }
  // ---- online softmax (base 2) of query row r
  float mx = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
  mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 2));
  const float mnew = fmaxf(st.m, mx);
  const float muse = mnew == -INFINITY ? 0.f : mnew;
  const float alpha = exp2f(st.m - muse);
  st.m = mnew;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) s[nt][e] = exp2f(s[nt][e] - muse);
  st.l = st.l * alpha + ((s[0][0] + s[0][1]) + (s[1][0] + s[1][1]));
  const float a_lo = __shfl_sync(~0u, alpha, 8 * c);
  const float a_hi = __shfl_sync(~0u, alpha, 8 * c + 4);
  if (__any_sync(~0u, a_lo != 1.f || a_hi != 1.f)) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      st.o[mt][0] *= a_lo;
      st.o[mt][1] *= a_hi;
      st.o[mt][2] *= a_lo;
      st.o[mt][3] *= a_hi;
    }
  }
  // ---- O^T += V^T.P^T; keys 2c, 2c + 1, 8 + 2c, 9 + 2c; INT4 value scales
  // go into P (a key past the sequence end gets P = 0 whatever its scale)
  const int tk[4] = {2 * c, 2 * c + 1, 8 + 2 * c, 9 + 2 * c};
  float pv[4] = {s[0][0], s[0][1], s[1][0], s[1][1]};
  if constexpr (K4 == 1) {
#pragma unroll
    for (int k = 0; k < 4; k += 2) {
      float2 v;
      asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];"
                   : "=f"(v.x), "=f"(v.y)
                   : "r"(v_base + kCodes + 4 * tk[k]));
      pv[k] = tk[k] < valid_keys ? pv[k] * v.x : 0.f;
      pv[k + 1] = tk[k + 1] < valid_keys ? pv[k + 1] * v.y : 0.f;
    }
  }
  const uint32_t b0 = pack2<false>(pv[0], pv[1]);
  const uint32_t b1 = pack2<false>(pv[2], pv[3]);
  uint2 vw[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                 : "=r"(vw[k].x), "=r"(vw[k].y)
                 : "r"(v_base + tk[k] * 64 + 8 * r));
  }
  uint32_t vsc[2] = {0u, 0u};  // NVFP4: block r of keys (0, 1) and (2, 3)
  if constexpr (K4 == 2) {
    uint32_t sb[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      asm volatile("ld.shared.u8 %0, [%1];" : "=r"(sb[k]) : "r"(v_base + kCodes + tk[k] * 8 + r));
      if (tk[k] >= valid_keys) sb[k] = 0u;  // past the end: scale 0, not NaN
    }
    vsc[0] = e4m3x2_to_f16x2(sb[0] | (sb[1] << 8));
    vsc[1] = e4m3x2_to_f16x2(sb[2] | (sb[3] << 8));
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int m = mt & 3;
    const uint32_t sel = (uint32_t)(m | (m << 4) | ((4 + m) << 8) | ((4 + m) << 12));
    const uint32_t wa = (mt >> 2) ? vw[0].y : vw[0].x;
    const uint32_t wb = (mt >> 2) ? vw[1].y : vw[1].x;
    const uint32_t wc = (mt >> 2) ? vw[2].y : vw[2].x;
    const uint32_t wd = (mt >> 2) ? vw[3].y : vw[3].x;
    uint32_t a[4];
    if constexpr (K4 == 1) {
      // byte mt of keys (0, 1) in bytes 0 and 2, of keys (2, 3) likewise
      const uint32_t xab = __byte_perm(wa, wb, sel);
      const uint32_t xcd = __byte_perm(wc, wd, sel);
      const __half2 off = __floats2half2_rn(1032.f, 1032.f);
      const __half2 sixteenth = __floats2half2_rn(0.0625f, 0.0625f);
      const __half2 off16 = __floats2half2_rn(-72.f, -72.f);
      uint32_t t0 = (xab & kNibLo) ^ kNibLoFlip, t1 = (xab & kNibHi) ^ kNibHiFlip;
      uint32_t t2 = (xcd & kNibLo) ^ kNibLoFlip, t3 = (xcd & kNibHi) ^ kNibHiFlip;
      __half2 h0 = __hsub2(*reinterpret_cast<__half2*>(&t0), off);
      __half2 h1 = __hfma2(*reinterpret_cast<__half2*>(&t1), sixteenth, off16);
      __half2 h2 = __hsub2(*reinterpret_cast<__half2*>(&t2), off);
      __half2 h3 = __hfma2(*reinterpret_cast<__half2*>(&t3), sixteenth, off16);
      a[0] = *reinterpret_cast<uint32_t*>(&h0);
      a[1] = *reinterpret_cast<uint32_t*>(&h1);
      a[2] = *reinterpret_cast<uint32_t*>(&h2);
      a[3] = *reinterpret_cast<uint32_t*>(&h3);
    } else {
      // each key's byte mt -> its (row r, row r + 8) pair, then the pairs of
      // keys (0, 1) and (2, 3) regrouped by row
      const uint32_t k0 = e2m1x2_byte(wa, m), k1 = e2m1x2_byte(wb, m);
      const uint32_t k2 = e2m1x2_byte(wc, m), k3 = e2m1x2_byte(wd, m);
      a[0] = hmul2u(__byte_perm(k0, k1, 0x5410), vsc[0]);
      a[1] = hmul2u(__byte_perm(k0, k1, 0x7632), vsc[0]);
      a[2] = hmul2u(__byte_perm(k2, k3, 0x5410), vsc[1]);
      a[3] = hmul2u(__byte_perm(k2, k3, 0x7632), vsc[1]);
    }
    mma16816<false>(st.o[mt], a, b0, b1);
  }
}

template <int kKind>
struct HgLayout {
  using Tr = Traits<kKind>;
  static constexpr int kPageBytes = Tr::kPageBytes;          // one KV head
  static constexpr int kStageBytes = 2 * kHg * kPageBytes;   // K, V of a group
  // 4-bit pages: seven stages (~60 KiB), so that three CTAs fit on an SM
  static constexpr int kCtasPerSm =
      Tr::k4 ? kCtasPerSm4 : (Tr::kD == 64 ? PA_HG_D64_CTAS : PA_CTAS_PER_SM);
  static constexpr int kStages =
      Tr::k4 ? 7
             : (Tr::kD == 64 && PA_HG_D64_STAGES > 0 ? PA_HG_D64_STAGES
                                                      : PA_HG_RING_BYTES / kStageBytes);
  static constexpr int kRing = 0;
  static constexpr int kBars = kRing + kStages * kStageBytes;
  static constexpr int kIds = kBars + 8 * 2 * kStages;       // int [2][32]
  static constexpr int kAbort = kIds + 2 * 32 * 4;
  static constexpr int kPlan = kAbort + 16;  // dec0, declen, rows per request
  static constexpr int kScan = kPlan + kHgMaxSeqs * 16;
  static constexpr int kBytes = kScan + 34 * 8;
  static constexpr int kSmemBytes = 1024 + kBytes;           // + alignment slack
  // (228 KiB of shared memory per SM, 1 KiB of it reserved per CTA)
  static_assert(kCtasPerSm * (kSmemBytes + 1024) <= 228 * 1024,
                "head-group CTAs per SM do not fit");
  static_assert(kCtasPerSm <= kMaxCtasPerSm, "partial slots sized for fewer CTAs per SM");
};

// One consumer warp's part of an item: every page of the item, its own KV
// head g; the output rows of that head (or its partial, slot >= 0).
template <int kKind>
__device__ void consume_hg_item(const FastParams& p, uint32_t ring,
                                uint32_t bars, volatile int* abort_flag,
                                const ReqMeta& rm, int g, int slot, int page0,
                                int npages, int rows, uint32_t c0, int warp,
                                int lane) {
  using Ly = HgLayout<kKind>;
  constexpr int S = Ly::kStages;
  const int rq = lane >> 2, c = lane & 3;
  const int G = p.group;
  uint32_t qa[8][4];
  float rscale[2];
  float qbias = 0.f;  // INT4: the row's score bias (load_q4)
  if constexpr (Traits<kKind>::k4) {
    load_q4<kKind>(p, rm.q0, g, rows, lane, qa, rscale[0], qbias);
    rscale[1] = rscale[0];
  } else {
    load_q<kKind, false>(p, rm.q0, g, 0, rows, lane, qa, rscale);
  }
  const int lim = rq < rows ? rm.L - rm.n + rq / G : rm.L - 1;
  int min_lim = rq < rows ? lim : INT_MAX;
  int max_lim = rq < rows ? lim : -1;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    min_lim = min(min_lim, __shfl_xor_sync(~0u, min_lim, d));
    max_lim = max(max_lim, __shfl_xor_sync(~0u, max_lim, d));
  }
  min_lim = min(min_lim, rm.L - 1);
  // keys at or below this are outside some row's window
  const int win_edge = max_lim - p.window;
  const float ss = p.score_scale * rscale[0];

  NarrowState st;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
    st.o[mt][0] = st.o[mt][1] = st.o[mt][2] = st.o[mt][3] = 0.f;
  st.m = -INFINITY;
  st.l = 0.f;
  for (int j = 0; j < npages; ++j) {
    const uint32_t cc = c0 + j;
    const int s = cc % S;
    if (!__all_sync(~0u, mbar_wait_bounded(bars + 8 * s, (cc / S) & 1))) {
      if (lane == 0) {
        flag_error(p.err, PA_DEV_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      return;
    }
    const int key0 = (page0 + j) * kBS;
    const int valid = min(kBS, rm.L - key0);
    const bool need_mask = key0 + kBS - 1 > min_lim || key0 <= win_edge;
    const uint32_t kb = ring + s * Ly::kStageBytes + warp * Ly::kPageBytes;
    if constexpr (Traits<kKind>::k4)
      process_page_4bit<kKind>(kb, kb + kHg * Ly::kPageBytes, qa, st, key0,
                               valid, need_mask, lim, p.window, ss, lane, qbias);
    else
      process_page_narrow<kKind>(kb, kb + kHg * Ly::kPageBytes, qa, st, key0,
                                 valid, need_mask, lim, p.window, ss, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (S + s));
  }
  st.l += __shfl_xor_sync(~0u, st.l, 1);
  st.l += __shfl_xor_sync(~0u, st.l, 2);
  // row 2c + h of O^T is held here; its (m, l) by lanes 4 (2c + h) ..
  float mq[2], lq[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    mq[h] = __shfl_sync(~0u, st.m, (2 * c + h) * 4);
    lq[h] = __shfl_sync(~0u, st.l, (2 * c + h) * 4);
  }
  const int Hq = p.num_q_heads;
  constexpr int kD = Traits<kKind>::kD;
#pragma unroll
  for (int mt = 0; mt < kD / 16; ++mt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int qrow = 2 * c + (e & 1);
      if (qrow >= rows) continue;
      const int col = narrow_col<kKind>(mt, e, rq);
      if (slot < 0) {
        const int i = qrow / G;
        const int h = g * G + (qrow - i * G);
        const int64_t orow = (int64_t)(rm.q0 + i) * Hq + h;
        store_out<OutT<kKind>>(p.out, orow * kD + col,
                               st.o[mt][e] / lq[e & 1] * p.out_scale);
      } else {
        const int64_t pr = (int64_t)slot * kHgPartRows + warp * 8 + qrow;
        p.ws_acc[pr * kD + col] = st.o[mt][e];
        if (mt == 0 && (e >> 1) == 0 && rq == 0) {
          p.ws_ml[pr * 2 + 0] = mq[e & 1];
          p.ws_ml[pr * 2 + 1] = lq[e & 1];
        }
      }
    }
  }
}

template <int kKind>
__global__ void __launch_bounds__(kThreads, HgLayout<kKind>::kCtasPerSm)
attn_decode_hg_kernel(const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v,
                      const __grid_constant__ FastParams p) {
  using Tr = Traits<kKind>;
  using Ly = HgLayout<kKind>;
  constexpr int S = Ly::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const sp = smem_raw + (base - raw);
  const uint32_t bars = base + Ly::kBars;  // full[S], then empty[S]
  int* ids = reinterpret_cast<int*>(sp + Ly::kIds);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sp + Ly::kAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(bars + 8 * i, 1);
      mbar_init(bars + 8 * (S + i), kHg);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // everything before this grid is done (when a prefill grid runs ahead of
  // it, that grid let this one start only after its own wait)
  if (!p.no_dep_wait) pdl_wait();
  pdl_launch_dependents();  // the next grid may be scheduled behind this one
  // this CTA's stream-K range over the (request, head group) segments
  long long* dec0 = reinterpret_cast<long long*>(sp + Ly::kPlan);
  int* declen = reinterpret_cast<int*>(dec0 + kHgMaxSeqs);
  int* rows = declen + kHgMaxSeqs;
  long long* scan = reinterpret_cast<long long*>(sp + Ly::kScan);
  const long long C = plan_prefix(p, dec0, declen, rows, scan + 32, scan);
  const int g_eff = self_plan_grid(C, gridDim.x);
  ItemSource src{};
  src.self = true;
  src.dec0 = dec0;
  src.declen = declen;
  src.rows = rows;
  src.B = p.num_seqs;
  src.H = p.num_kv_heads / kHg;
  src.b = blockIdx.x;
  src.lo = src.hi = 0;
  if ((int)blockIdx.x < g_eff && C > 0) {
    src.lo = (long long)blockIdx.x * C / g_eff;
    src.hi = (long long)(blockIdx.x + 1) * C / g_eff;
  }
  src.cur = src.lo;
  src.r = p.num_seqs > 0 ? request_of(dec0, p.num_seqs, src.lo) : 0;
  src.casc = p.cascade_blocks > 0;
  src.pg_off = p.cascade_blocks;
  src.unc_slot0 = p.unc_slot0;

  if (warp == kConsumerWarps) {
    // ------------------------------ producer ------------------------------
    if (lane == 0 && !Tr::k4) {
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
    }
    uint32_t c = 0;  // stages issued
    int go = 1;
    int4 rec0, rec1;
    const long long skip = skipped_copy();
    while (go && src.next(rec0, rec1)) {
      const int32_t* bt =
          p.block_tables + (int64_t)rec0.x * p.max_blocks_per_seq + rec1.x;
      // block ids through shared memory 32 at a time; lanes 2k, 2k+1 issue
      // the K and V boxes of page k of each group of PP pages
      const int n = rec1.y - rec1.x;
      ids[lane] = lane < n ? __ldg(bt + lane) : 0;
      // pages of one step go to distinct ring slots (a lane must never wait
      // for the slot another lane of the same step is about to fill)
      constexpr int PP = PA_PRODUCER_PAGES < S ? PA_PRODUCER_PAGES : S;
      // L2 prefetch, PF pages ahead of the loads: the lanes of page k of a
      // step hold the block id of page k + PF, read one step early
      constexpr int PF = PA_L2_PREFETCH_PAGES;
      const bool pf_on = PF > 0 && p.l2_prefetch != 0;
      int pf_blk = -1;
      if (pf_on && lane < 2 * PP) {
        const int t = (lane >> 1) + PF;
        pf_blk = t < n ? __ldg(bt + t) : -1;
      }
      __syncwarp();
      for (int j0 = 0; j0 < n && go; j0 += 32) {
        const int buf = (j0 >> 5) & 1;
        const int nidx = j0 + 32 + lane;
        const int nreg = nidx < n ? __ldg(bt + nidx) : 0;
        constexpr unsigned kMask = (PP >= 16) ? 0xFFFFFFFFu : ((1u << (2 * PP)) - 1u);
        if (lane < 2 * PP) {
          const int* cur = ids + buf * 32;
          const int cnt = min(32, n - j0);
          const int kk = lane >> 1;
          const int kv = lane & 1;
          const CUtensorMap* map = kv ? &tmap_v : &tmap_k;
          for (int jj = 0; jj < cnt; jj += PP) {
            const bool mine = jj + kk < cnt;
            const uint32_t cc = c + kk;
            const int s = cc % S;
            const bool ok = !mine || cc < (uint32_t)S ||
                            mbar_wait_bounded(bars + 8 * (S + s), ((cc / S) - 1) & 1);
            if (__any_sync(kMask, !ok)) {
              if (lane == 0) {
                flag_error(p.err, PA_DEV_ERR_TIMEOUT);
                *abort_flag = 1;
              }
              go = 0;
              break;
            }
            if (mine && (long long)cc != skip) {
              int blk = cur[jj + kk];
              if (blk < 0 || (int64_t)blk >= p.num_blocks) {
                if (kv == 0) flag_error(p.err, PA_DEV_ERR_BLOCK_ID);
                blk = 0;
              }
              const int row = (blk * p.num_kv_heads + rec0.y * kHg) * kBS;
              const uint32_t dst = base + Ly::kRing + s * Ly::kStageBytes +
                                   kv * kHg * Ly::kPageBytes;
              if (kv == 0) mbar_arrive_expect_tx(bars + 8 * s, Ly::kStageBytes);
              __syncwarp(__activemask());
              if constexpr (Tr::k4) {
                // the group's four pages (codes and scales) are contiguous
                const uint8_t* src =
                    (kv ? p.v4 : p.k4) +
                    ((int64_t)blk * p.num_kv_heads + rec0.y * kHg) * Ly::kPageBytes;
                bulk_load(dst, src, kHg * Ly::kPageBytes, bars + 8 * s);
              } else if constexpr (Tr::kRows128) {
                tma_load_2d(dst, map, bars + 8 * s, 0, row);
              } else {
                tma_load_3d(dst, map, bars + 8 * s, 0, 0, row);
              }
            }
            if (pf_on) {
              if (pf_blk >= 0 && (int64_t)pf_blk < p.num_blocks) {
                const int prow = (pf_blk * p.num_kv_heads + rec0.y * kHg) * kBS;
                if constexpr (Tr::k4) {
                  bulk_prefetch_l2((kv ? p.v4 : p.k4) +
                                       ((int64_t)pf_blk * p.num_kv_heads + rec0.y * kHg) *
                                           Ly::kPageBytes,
                                   kHg * Ly::kPageBytes);
                } else if constexpr (Tr::kRows128) {
                  tma_prefetch_l2_2d(map, 0, prow);
                } else {
                  tma_prefetch_l2_3d(map, 0, 0, prow);
                }
              }
              // the page this lane loads next (this buffer, else the next one)
              const int nj = (jj + PP < cnt ? j0 + jj + PP : j0 + 32) + kk;
              pf_blk = nj + PF < n ? __ldg(bt + nj + PF) : -1;
            }
            c += min(PP, cnt - jj);
          }
        }
        __syncwarp();
        go = __shfl_sync(~0u, go, 0);
        c = __shfl_sync(~0u, c, 0);
        ids[(buf ^ 1) * 32 + lane] = nreg;
        __syncwarp();
      }
    }
    // after an abort, let the copies already in flight land before exiting
    if (!go && lane == 0) {
      const uint32_t from = c > (uint32_t)S ? c - S : 0;
      for (uint32_t i = from; i < c; ++i)
        mbar_wait_bounded(bars + 8 * (i % S), (i / S) & 1);
    }
    return;
  }

  // ------------------------------ consumers -------------------------------
  uint32_t c = 0;  // stages consumed (every warp reads every stage)
  int4 rec0, rec1;
  while (src.next(rec0, rec1)) {
    if (consumers_sync_any(*abort_flag != 0)) break;
    const ReqMeta rm = load_req(p.qsl, p.seq_lens, rec0.x, p.num_tokens,
                                p.max_query_len, p.max_seq_len,
                                p.max_blocks_per_seq);
    consume_hg_item<kKind>(p, base + Ly::kRing, bars, abort_flag, rm,
                           rec0.y * kHg + warp, rec0.w, rec1.x, rec1.y - rec1.x,
                           rec1.z, c, warp, lane);
    c += rec1.y - rec1.x;
  }
}

template <int kKind, bool kWide>
cudaError_t prepare_kernel(int* grid) {
  using Ly = Layout<kKind, kWide>;
  static int blocks_per_sm[64] = {0};
  static int sms[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (blocks_per_sm[dev] == 0) {
    e = cudaFuncSetAttribute(attn_fast_kernel<kKind, kWide>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Ly::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_fast_kernel<kKind, kWide>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int nb = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &nb, attn_fast_kernel<kKind, kWide>, kThreads, Ly::kSmemBytes);
    if (e != cudaSuccess) return e;
    int n_sm = 0;
    e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sms[dev] = n_sm;
    blocks_per_sm[dev] = nb > 0 ? nb : 1;
  }
  *grid = blocks_per_sm[dev] * sms[dev];
  return cudaSuccess;
}

template <int kKind>
cudaError_t prepare_hg(int* grid) {
  using Ly = HgLayout<kKind>;
  static int blocks_per_sm[64] = {0};
  static int sms[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (blocks_per_sm[dev] == 0) {
    e = cudaFuncSetAttribute(attn_decode_hg_kernel<kKind>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Ly::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_decode_hg_kernel<kKind>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int nb = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &nb, attn_decode_hg_kernel<kKind>, kThreads, Ly::kSmemBytes);
    if (e != cudaSuccess) return e;
    int n_sm = 0;
    e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sms[dev] = n_sm;
    blocks_per_sm[dev] = nb > 0 ? nb : 1;
  }
  *grid = blocks_per_sm[dev] * sms[dev];
  return cudaSuccess;
}

// decode-only steps (<= 8 rows per request) in head groups: KV heads a
// multiple of kHg, up to kHgMaxSeqs requests
// Steps whose decode work runs in KV-head groups: KV heads a multiple of
// kHg, at most kHgMaxSeqs requests, and every request of more than 8 query
// rows (if any) handled by the tensor-core prefill kernel.
bool use_head_groups(const AttnArgs& a, bool tc) {
  const int G = a.num_q_heads / a.num_kv_heads;
  if (a.num_kv_heads % kHg != 0 || a.num_seqs > kHgMaxSeqs) return false;
  return (int64_t)a.max_query_len * G <= 8 || tc;
}

// SMs that run prefill tiles while the decode kernel of a mixed step runs on
// the others.  The tiles' share of the step's time from host-known sizes:
// per key, a prefill token costs 4 D Hq flops on the tensor cores (~1e15
// flop/s in this kernel) and a decode request 2 D Hkv x 2 bytes from HBM
// (~6e12 B/s), so the prefill : decode time ratio is about
// r = G x (prefill tokens / requests) x 0.006, the key counts taken as equal
// and tokens beyond one per request counted as prefill tokens.  The decode
// kernel slows almost in proportion to the SMs it loses, so the split gives
// the tiles half their balanced share: the rest run behind the decode kernel
// on every SM, which measured best (a 1022-token chunk beside 120 decodes:
// 13 SMs, step 437 -> 428 us; 20 SMs or more were slower than none).
//
// Cascade steps: the decode segments lose the shared prefix (their keys
// taken as max_seq_len - 16 N against the prefill rows' max_seq_len), and
// the decode kernel, prefetching into L2 (l2_prefetch) and reading no
// prefix from L2, keeps HBM busy on fewer SMs: the tiles get their whole
// balanced share (the 120-decode mixed step after a 125-block prefix: 31
// SMs; measured 13 -> 0.409 ms, 28 -> 0.387-0.392, 36-44 -> 0.394).  The
// prefix tiles add their own time: a tile's chunk of 8 blocks takes about
// 1 us whatever its rows (its TMA copies; FP8 pages about twice that, with
// the widening), per 128-row tile of the decode tokens (one per request
// taken) and KV head.
int prefill_ctas_ahead(const AttnArgs& a, int num_sms) {
  const int64_t n_pf = a.num_tokens - a.num_seqs + 1;
  if (n_pf <= 0 || a.num_seqs <= 0 || num_sms < 16) return 0;
  const double G = (double)a.num_q_heads / a.num_kv_heads;
  double r = G * (double)n_pf / (double)a.num_seqs * 0.006;
  double share = 0.5;
  if (a.cascade_blocks > 0) {
    const double K = (double)a.max_seq_len;
    const double Kd = std::max(1.0, K - (double)a.cascade_blocks * kBS);
    r *= K / Kd;
    const bool fp8 = a.cache_dtype == PA_FP8_E4M3;
    const double elem = fp8 ? 1.0 : 2.0;
    const double t_dec =
        (double)a.num_seqs * Kd * a.num_kv_heads * a.head_dim * 2.0 * elem / 6e12;
    const double tpt = std::max(1.0, 128.0 / G);
    const double ctiles = std::ceil((double)std::min<int64_t>(a.num_tokens, a.num_seqs) / tpt);
    const double t_pre = ctiles * a.num_kv_heads * a.cascade_blocks *
                         (fp8 ? 0.25e-6 : 0.125e-6) / num_sms;
    r += t_pre / t_dec;
    share = 1.0;
  }
  int p = (int)(share * num_sms * r / (1.0 + r) + 0.5);
  if (p < 4) p = 4;
  if (p > num_sms / 4) p = num_sms / 4;
  return p;
}

template <int kKind>
cudaError_t launch_hg(const AttnArgs& a, const FastParams& fp,
                      const AttnPlan& plan, const CUtensorMap& tk,
                      const CUtensorMap& tv, const TcMaps* tc, int num_sms,
                      cudaStream_t stream) {
  int grid = 0;
  cudaError_t e = prepare_hg<kKind>(&grid);
  if (e != cudaSuccess) return e;
  if (grid > plan.grid_max) grid = plan.grid_max;
  FastParams f = fp;
  f.self_plan = 1;
  f.dec_rows_max = 8;
  f.seg_heads = kHg;
  f.attn_grid = grid;
  // steps with prefill tiles beside the decode kernel: prefetching two pages
  // ahead into L2 measured 5.7 % faster on the 120-decode mixed step with a
  // shared 2000-token prefix, and neutral on decode-only steps (not used there)
  f.l2_prefetch = tc != nullptr ? 1 : 0;
  const ProfileEvents& pe = profile_events();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pe.start == nullptr ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = HgLayout<kKind>::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // With prefill tiles (requests of more than 8 query rows) the tensor-core
  // kernel and the decode kernel share the GPU, the tiles drawn from one
  // step-wide counter (zeroed here):
  //  1. a prefill grid of P CTAs (one per SM) goes first; it waits for the
  //     step's inputs and then lets the next grid start;
  //  2. the decode kernel, on the other SMs (its CTAs do not fit next to a
  //     prefill CTA), starts without a wait of its own;
  //  3. a second prefill grid, behind the decode kernel, takes the SMs its
  //     CTAs leave and draws whatever tiles are left (none: it exits).
  // The merge, a plain launch, waits for all three.
  int* tile_ctr = nullptr;
  int pf_ctas = 0;
  if (tc) {
    tile_ctr = reinterpret_cast<int*>(static_cast<uint8_t*>(a.workspace) +
                                      plan.off_pref) + 1;
    e = cudaMemsetAsync(tile_ctr, 0, sizeof(int), stream);
    if (e != cudaSuccess) return e;
    // A step of one request with more than 8 query rows per KV head has no
    // decode work (its rows all go to the tiles): the tensor-core kernel runs
    // alone, one CTA per SM, with no decode kernel and no merge.
    const int G = a.num_q_heads / a.num_kv_heads;
    if (a.num_seqs == 1 && a.num_tokens * G > 8 && f.cascade_blocks == 0) {
      if (pe.start) cudaEventRecord(pe.start, stream);
      e = launch_prefill_tc(a, *tc, true, nullptr, nullptr, (int)plan.max_atoms, 8,
                            tile_ctr, false, num_sms, stream);
      if (pe.stop) cudaEventRecord(pe.stop, stream);
      return e;
    }
    // (with the profiling events on, launches are plain and run one after
    // the other: no grid ahead, the tiles all behind the decode kernel)
    pf_ctas = pe.start == nullptr ? prefill_ctas_ahead(a, num_sms) : 0;
    const int per_sm = num_sms > 0 && grid >= num_sms ? grid / num_sms : 1;
    const int dec_grid = per_sm * (num_sms - pf_ctas);
    if (dec_grid >= 1 && dec_grid < grid) grid = dec_grid;
    f.attn_grid = grid;
    f.no_dep_wait = (pe.start == nullptr && pf_ctas > 0) ? 1 : 0;
    cfg.gridDim = dim3(grid);
  }
  if (pe.start) cudaEventRecord(pe.start, stream);
  // (cascade steps: the shared-prefix tiles' partial rows)
  float* casc_acc = f.cascade_blocks > 0 ? f.ws_acc + f.casc_row0 * 128 : nullptr;
  float* casc_ml = f.cascade_blocks > 0 ? f.ws_ml + f.casc_row0 * 2 : nullptr;
  if (tc && pf_ctas > 0) {
    e = launch_prefill_tc(a, *tc, true, nullptr, nullptr, (int)plan.max_atoms, 8,
                          tile_ctr, false, pf_ctas, stream, casc_acc, casc_ml,
                          f.casc_splits, f.casc_split_rows);
    if (e != cudaSuccess) return e;
  }
  e = cudaLaunchKernelEx(&cfg, attn_decode_hg_kernel<kKind>, tk, tv, f);
  if (e != cudaSuccess) return e;
  count_launch();
  if (tc) {
    e = launch_prefill_tc(a, *tc, true, nullptr, nullptr, (int)plan.max_atoms, 8,
                          tile_ctr, pe.start == nullptr, num_sms, stream, casc_acc,
                          casc_ml, f.casc_splits, f.casc_split_rows);
    if (e != cudaSuccess) return e;
  }
  if (pe.stop) cudaEventRecord(pe.stop, stream);
  // one merge CTA per range boundary
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = (size_t)f.num_seqs * 16;
  attr[0].val.programmaticStreamSerializationAllowed =
      (pe.start == nullptr && !tc) ? 1 : 0;
  e = f.cascade_blocks > 0
          ? cudaLaunchKernelEx(&cfg, merge_self_kernel<OutT<kKind>, true>, f)
          : cudaLaunchKernelEx(&cfg, merge_self_kernel<OutT<kKind>, false>, f);
  if (e == cudaSuccess) count_launch();
  return e;
}

template <int kKind>
cudaError_t launch_kind(const AttnArgs& a, const FastParams& fp, PlanArgs pa,
                        const AttnPlan& plan, const CUtensorMap& tk,
                        const CUtensorMap& tv, const TcMaps* tc, int num_sms,
                        cudaStream_t stream) {
  // the narrow kernel covers steps whose every item has <= 8 rows
  const bool wide = (int64_t)fp.max_query_len * fp.group > 8;
  int grid = 0;
  cudaError_t e = wide ? prepare_kernel<kKind, true>(&grid)
                       : prepare_kernel<kKind, false>(&grid);
  if (e != cudaSuccess) return e;
  if (grid > plan.grid_max) grid = plan.grid_max;
  pa.grid = grid;
  // Steps whose decode work is all the attention kernel has to do (no
  // prefill tiles, or prefill tiles on the tensor-core kernel) plan inside
  // the kernels, up to a request count; the rest go through the planner.
  FastParams f = fp;
  f.attn_grid = grid;
  f.dec_rows_max = wide ? kDecodeMaxRows : 8;
  f.self_plan = fp.num_seqs <= (wide ? kSelfPlanMaxSeqsWide : kSelfPlanMaxSeqs) &&
                (!plan.has_prefill || tc != nullptr);
  if (!f.self_plan) {
    plan_kernel<<<1, kPlanThreads, kPlanCacheBytes, stream>>>(pa);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launch();
  }
  // The attention kernel and the merge are launched as programmatic
  // dependents: each may start while its predecessor runs and waits (on the
  // device) for it to finish before touching its results.  With the
  // profiling hook on, plain launches keep the events around the kernel.
  const ProfileEvents& pe = profile_events();
  const bool pdl = pe.start == nullptr;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (pe.start) cudaEventRecord(pe.start, stream);
  if (tc) {
    // prefill tiles on the tensor cores, ahead of the decode work
    e = launch_prefill_tc(a, *tc, f.self_plan != 0, pa.atoms, pa.n_atoms_out,
                          pa.max_atoms, kDecodeMaxRows, nullptr, false, num_sms,
                          stream);
    if (e != cudaSuccess) return e;
  }
  if (wide) {
    cfg.dynamicSmemBytes = Layout<kKind, true>::kSmemBytes;
    e = cudaLaunchKernelEx(&cfg, attn_fast_kernel<kKind, true>, tk, tv, f);
  } else {
    cfg.dynamicSmemBytes = Layout<kKind, false>::kSmemBytes;
    e = cudaLaunchKernelEx(&cfg, attn_fast_kernel<kKind, false>, tk, tv, f);
  }
  if (pe.stop) cudaEventRecord(pe.stop, stream);
  if (e != cudaSuccess) return e;
  count_launch();
  if (plan.has_decode) {
    // split segments: at most one fewer than the CTAs that got work
    if (f.self_plan) {
      cfg.blockDim = dim3(kMergeThreads);
      cfg.dynamicSmemBytes = (size_t)f.num_seqs * 16;
      e = cudaLaunchKernelEx(&cfg, merge_self_kernel<OutT<kKind>, false>, f);
    } else {
      cfg.blockDim = dim3(128);
      cfg.dynamicSmemBytes = 0;
      e = cudaLaunchKernelEx(&cfg, merge_kernel<OutT<kKind>>, f);
    }
    if (e == cudaSuccess) count_launch();
  }
  return e;
}

}  // namespace

int decode_box_rows(const AttnArgs& a, bool tc) {
  return use_head_groups(a, tc) ? kHg * kBS : kBS;
}

int cascade_splits(const AttnPlan& plan, int cascade_blocks) {
  const int want = (cascade_blocks + kCascMinSplitBlocks - 1) / kCascMinSplitBlocks;
  return std::max(1, std::min(plan.casc_splits, want));
}

bool cascade_supported(const AttnArgs& a) {
  return a.cascade_blocks > 0 && a.window <= 0 && fast_path_supported(a) &&
         tc_prefill_supported(a) && use_head_groups(a, true);
}

bool fast_path_supported(const AttnArgs& a) {
  // head_dim 64, bf16 / f16: decode-only steps in KV-head groups
  if (a.head_dim == 64)
    return (a.cache_dtype == PA_BF16 || a.cache_dtype == PA_F16) &&
           a.q_dtype == a.cache_dtype && use_head_groups(a, false);
  if (a.head_dim != 128) return false;
  // 4-bit caches: decode-only steps in KV-head groups
  if (is_4bit(a.cache_dtype))
    return (a.q_dtype == PA_BF16 || a.q_dtype == PA_F16) && use_head_groups(a, false);
  if (a.cache_dtype == PA_BF16 && a.q_dtype == PA_BF16) return true;
  if (a.cache_dtype == PA_F16 && a.q_dtype == PA_F16) return true;
  if (a.cache_dtype == PA_FP8_E4M3 && (a.q_dtype == PA_BF16 || a.q_dtype == PA_F16))
    return true;
  return false;
}

AttnPlan make_plan(int64_t num_tokens, int num_q_heads, int num_kv_heads,
                   int head_dim, int num_seqs, int max_query_len,
                   int max_seq_len, int num_sms, int window, bool cascade) {
  AttnPlan pl{};
  pl.cascade = cascade && window <= 0 ? 1 : 0;
  pl.window = window > 0 && window < max_seq_len ? window : 0;
  pl.group = num_q_heads / num_kv_heads;
  pl.has_prefill = (int64_t)max_query_len * pl.group > kDecodeMaxRows;
  pl.has_decode = pl.group <= kDecodeMaxRows;
  pl.grid_max = num_sms * kMaxCtasPerSm;
  pl.max_atoms =
      pl.has_prefill
          ? (int64_t)num_kv_heads *
                ((num_tokens * pl.group + kPrefillTileRows - 1) / kPrefillTileRows +
                 num_seqs)
          : 0;
  pl.casc_splits = 1;
  if (pl.cascade) {
    // shared-prefix tiles: the step's tokens, per KV head, in tiles of
    // 128 / group tokens (128 query rows), for each of up to casc_splits key
    // ranges of the prefix: as many as keep the tiles within one per SM,
    // ranges of at least kCascMinSplitBlocks blocks of the longest prefix
    // the step allows (its keys lie before some query: < max_seq_len)
    const int64_t tpt = std::max(1, 128 / pl.group);
    const int64_t tiles = (int64_t)num_kv_heads * ((num_tokens + tpt - 1) / tpt);
    const int64_t max_blocks = std::max<int64_t>(1, ((int64_t)max_seq_len - 1) / kBS);
    int64_t sp = tiles > 0 ? num_sms / tiles : 1;
    sp = std::min<int64_t>(sp, (max_blocks + kCascMinSplitBlocks - 1) / kCascMinSplitBlocks);
    pl.casc_splits = (int)std::max<int64_t>(1, std::min<int64_t>(sp, kCascMaxSplits));
    pl.max_atoms += tiles * pl.casc_splits;
  }
  pl.max_items = pl.max_atoms + (pl.has_decode ? (int64_t)num_seqs * num_kv_heads : 0) +
                 pl.grid_max;
  pl.max_slots = 2 * (int64_t)pl.grid_max;
  pl.unc_slots = pl.cascade && pl.has_decode ? (int64_t)num_seqs * (num_kv_heads / kHg) : 0;
  // partial rows: the slots', then (cascade) one per key range, token and
  // q head
  pl.casc_row0 = (pl.max_slots + pl.unc_slots) * kHgPartRows;
  pl.casc_split_rows = num_tokens * num_q_heads;
  const int64_t part_rows =
      pl.has_decode
          ? pl.casc_row0 + (pl.cascade ? pl.casc_splits * pl.casc_split_rows : 0)
          : 0;
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  size_t off = 0;
  pl.off_atoms = off;       off = up(off + (size_t)pl.max_atoms * 16);
  pl.off_atom_start = off;  off = up(off + (size_t)pl.max_atoms * 8);
  pl.off_req_dec0 = off;    off = up(off + (size_t)num_seqs * 8);
  pl.off_req_declen = off;  off = up(off + (size_t)num_seqs * 4);
  pl.off_req_rows = off;    off = up(off + (size_t)num_seqs * 4);
  pl.off_items = off;       off = up(off + (size_t)pl.max_items * 32);
  pl.off_cta_begin = off;   off = up(off + (size_t)(pl.grid_max + 1) * 4);
  pl.off_seg_info = off;    off = up(off + (size_t)num_seqs * num_kv_heads * 8);
  pl.off_split = off;       off = up(off + (size_t)pl.max_slots * 16 + 16);
  pl.off_pref = off;        off = up(off + 16);
  // partial slots of up to kHgPartRows rows (head-group items: kHg heads x 8)
  pl.off_acc = off;
  off = up(off + (size_t)part_rows * head_dim * 4);
  pl.off_ml = off;
  off = up(off + (size_t)part_rows * 2 * 4);
  // a request's keys through the window start in the block holding key
  // L - n - window + 1: at most n + window - 1 + 15 keys from there
  pl.off_win_sl = pl.off_win_bt = off;
  if (pl.window > 0) {
    pl.win_max_seq_len =
        (int)std::min<int64_t>(max_seq_len, (int64_t)max_query_len + pl.window + 14);
    pl.win_blocks = (pl.win_max_seq_len + kBS - 1) / kBS;
    off = up(off + (size_t)num_seqs * 4);
    pl.off_win_bt = off;
    off = up(off + (size_t)num_seqs * pl.win_blocks * 4);
  }
  pl.total_bytes = off;
  return pl;
}

namespace {

struct WindowArgs {
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int64_t num_tokens;
  int num_seqs, max_query_len, max_seq_len, max_blocks_per_seq, window;
  int32_t* bt_out;
  int32_t* sl_out;
  int blocks_out;
};

// One warp per request.  A request whose metadata fails the checks gets a
// key count of -1, which every kernel of the step then flags and skips.
__global__ void __launch_bounds__(256) window_view_kernel(WindowArgs w) {
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= w.num_seqs) return;
  const ReqMeta m = load_req(w.qsl, w.seq_lens, r, w.num_tokens, w.max_query_len,
                             w.max_seq_len, w.max_blocks_per_seq);
  if (!m.ok) {
    if (lane == 0) w.sl_out[r] = -1;
    return;
  }
  const int lo = m.L - m.n - w.window + 1;  // first query's first key
  const int p0 = lo > 0 ? lo / kBS : 0;
  const int Lw = m.L - p0 * kBS;
  const int nbw = min((Lw + kBS - 1) / kBS, w.blocks_out);
  if (lane == 0) w.sl_out[r] = Lw;
  const int32_t* src = w.block_tables + (int64_t)r * w.max_blocks_per_seq + p0;
  int32_t* dst = w.bt_out + (int64_t)r * w.blocks_out;
  for (int k = lane; k < nbw; k += 32) dst[k] = __ldg(src + k);
}

}  // namespace

cudaError_t set_pipeline_hooks_fast(uint64_t wait_limit_ns, long long skip_copy) {
  cudaError_t e = cudaMemcpyToSymbol(g_wait_limit_ns, &wait_limit_ns,
                                     sizeof(wait_limit_ns));
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbol(g_skip_copy, &skip_copy, sizeof(skip_copy));
  return e;
}

cudaError_t launch_window_view(const AttnArgs& a, const AttnPlan& plan,
                               cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  WindowArgs w{};
  w.block_tables = a.block_tables;
  w.seq_lens = a.seq_lens;
  w.qsl = a.query_start_loc;
  w.num_tokens = a.num_tokens;
  w.num_seqs = a.num_seqs;
  w.max_query_len = a.max_query_len;
  w.max_seq_len = a.max_seq_len;
  w.max_blocks_per_seq = a.max_blocks_per_seq;
  w.window = plan.window;
  w.bt_out = reinterpret_cast<int32_t*>(ws + plan.off_win_bt);
  w.sl_out = reinterpret_cast<int32_t*>(ws + plan.off_win_sl);
  w.blocks_out = plan.win_blocks;
  const unsigned grid = (unsigned)((a.num_seqs + 7) / 8);
  window_view_kernel<<<grid, 256, 0, stream>>>(w);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

cudaError_t launch_attention_fast(const AttnArgs& a, const AttnPlan& plan,
                                  const CUtensorMap& tmap_k,
                                  const CUtensorMap& tmap_v, const TcMaps* tc,
                                  int num_sms, cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  FastParams fp{};
  fp.q = a.q;
  fp.out = a.out;
  fp.block_tables = a.block_tables;
  fp.seq_lens = a.seq_lens;
  fp.qsl = a.query_start_loc;
  fp.items = reinterpret_cast<const int4*>(ws + plan.off_items);
  fp.cta_begin = reinterpret_cast<const int*>(ws + plan.off_cta_begin);
  fp.split_list = reinterpret_cast<const int4*>(ws + plan.off_split + 16);
  fp.n_split = reinterpret_cast<const int*>(ws + plan.off_split);
  fp.max_slots = (int)plan.max_slots;
  fp.ws_acc = reinterpret_cast<float*>(ws + plan.off_acc);
  fp.ws_ml = reinterpret_cast<float*>(ws + plan.off_ml);
  fp.err = a.err;
  fp.num_tokens = a.num_tokens;
  fp.num_blocks = a.num_blocks;
  fp.max_blocks_per_seq = a.max_blocks_per_seq;
  fp.num_seqs = a.num_seqs;
  fp.num_q_heads = a.num_q_heads;
  fp.num_kv_heads = a.num_kv_heads;
  fp.group = plan.group;
  fp.max_query_len = a.max_query_len;
  fp.max_seq_len = a.max_seq_len;
  // FP8 and NVFP4 fold their per-tensor scales into the score and output
  // scales (INT4 has per-token scales only)
  const bool fp8 = a.cache_dtype == PA_FP8_E4M3 || a.cache_dtype == PA_NVFP4;
  fp.score_scale = a.scale * 1.4426950408889634f * (fp8 ? a.k_scale : 1.0f);
  fp.out_scale = fp8 ? a.v_scale : 1.0f;
  fp.k4 = static_cast<const uint8_t*>(a.k_cache);
  fp.v4 = static_cast<const uint8_t*>(a.v_cache);
  fp.head_dim = a.head_dim;
  fp.seg_heads = 1;
  fp.window = a.window > 0 ? a.window : kNoWindow;

  PlanArgs pa{};
  pa.qsl = a.query_start_loc;
  pa.seq_lens = a.seq_lens;
  pa.err = a.err;
  pa.num_tokens = a.num_tokens;
  pa.num_seqs = a.num_seqs;
  pa.max_query_len = a.max_query_len;
  pa.max_seq_len = a.max_seq_len;
  pa.max_blocks_per_seq = a.max_blocks_per_seq;
  pa.group = plan.group;
  pa.num_kv_heads = a.num_kv_heads;
  pa.prefill_weight = PA_PREFILL_WEIGHT;
  pa.prefill_tc = tc != nullptr;
  pa.tile_rows = tc ? tc_prefill_tile_rows(plan.group) : kPrefillTileRows;
  pa.n_atoms_out = reinterpret_cast<int*>(ws + plan.off_pref);
  pa.max_atoms = (int)plan.max_atoms;
  pa.max_items = (int)plan.max_items;
  pa.max_slots = (int)plan.max_slots;
  pa.atoms = reinterpret_cast<int4*>(ws + plan.off_atoms);
  pa.atom_start = reinterpret_cast<long long*>(ws + plan.off_atom_start);
  pa.req_dec0 = reinterpret_cast<long long*>(ws + plan.off_req_dec0);
  pa.req_declen = reinterpret_cast<int*>(ws + plan.off_req_declen);
  pa.items = reinterpret_cast<int4*>(ws + plan.off_items);
  pa.cta_begin = reinterpret_cast<int*>(ws + plan.off_cta_begin);
  pa.seg_cut = reinterpret_cast<int2*>(ws + plan.off_seg_info);
  pa.req_rows = reinterpret_cast<int*>(ws + plan.off_req_rows);
  pa.ws_ml = fp.ws_ml;
  pa.split_list = reinterpret_cast<int4*>(ws + plan.off_split + 16);
  pa.n_split = reinterpret_cast<int*>(ws + plan.off_split);
  if (use_head_groups(a, tc != nullptr)) {
    const TcMaps* t = plan.has_prefill || plan.cascade ? tc : nullptr;
    if (plan.cascade && t != nullptr && a.cascade_blocks > 0) {
      // shared-prefix step: the prefix tiles' rows and the uncut suffix
      // slots follow the split slots in the partial rows
      fp.cascade_blocks = a.cascade_blocks;
      fp.casc_splits = cascade_splits(plan, a.cascade_blocks);
      fp.casc_split_rows = plan.casc_split_rows;
      fp.unc_slot0 = plan.max_slots;
      fp.casc_row0 = plan.casc_row0;
    }
    const bool qb = a.q_dtype == PA_BF16;
    const bool d64 = a.head_dim == 64;
    switch (a.cache_dtype == PA_BF16   ? (d64 ? kKindBF16D64 : kKindBF16)
            : a.cache_dtype == PA_F16  ? (d64 ? kKindF16D64 : kKindF16)
            : a.cache_dtype == PA_INT4 ? (qb ? kKindI4BF16 : kKindI4F16)
            : a.cache_dtype == PA_NVFP4 ? (qb ? kKindN4BF16 : kKindN4F16)
            : qb                        ? kKindFp8BF16
                                        : kKindFp8F16) {
      case kKindBF16D64:
        return launch_hg<kKindBF16D64>(a, fp, plan, tmap_k, tmap_v, t, num_sms, stream);
      case kKindF16D64:
        return launch_hg<kKindF16D64>(a, fp, plan, tmap_k, tmap_v, t, num_sms, stream);
      case kKindI4BF16:
        return launch_hg<kKindI4BF16>(a, fp, plan, tmap_k, tmap_v, t, num_sms, stream);
      case kKindI4F16:
        return launch_hg<kKindI4F16>(a, fp, plan, tmap_k, tmap_v, t, num_sms, stream);
      case kKindN4BF16:
        return launch_hg<kKindN4BF16>(a, fp, plan, tmap_k, tmap_v, t, num_sms, stream);
      case kKindN4F16:
        return launch_hg<kKindN4F16>(a, fp, plan, tmap_k, tmap_v, t, num_sms, stream);
      case kKindBF16:
        return launch_hg<kKindBF16>(a, fp, plan, tmap_k, tmap_v, t, num_sms, stream);
      case kKindF16:
        return launch_hg<kKindF16>(a, fp, plan, tmap_k, tmap_v, t, num_sms, stream);
      case kKindFp8BF16:
        return launch_hg<kKindFp8BF16>(a, fp, plan, tmap_k, tmap_v, t, num_sms, stream);
      default:
        return launch_hg<kKindFp8F16>(a, fp, plan, tmap_k, tmap_v, t, num_sms, stream);
    }
  }
  if (a.cache_dtype == PA_BF16)
    return launch_kind<kKindBF16>(a, fp, pa, plan, tmap_k, tmap_v, tc, num_sms,
                                  stream);
  if (a.cache_dtype == PA_F16)
    return launch_kind<kKindF16>(a, fp, pa, plan, tmap_k, tmap_v, tc, num_sms,
                                 stream);
  if (a.q_dtype == PA_BF16)
    return launch_kind<kKindFp8BF16>(a, fp, pa, plan, tmap_k, tmap_v, tc,
                                     num_sms, stream);
  return launch_kind<kKindFp8F16>(a, fp, pa, plan, tmap_k, tmap_v, tc,
                                  num_sms, stream);
}

}  // namespace pa

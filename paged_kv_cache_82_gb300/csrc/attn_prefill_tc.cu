// attn_prefill_tc.cu -- the prefill tiles of a unified step on the
// 5th-generation tensor cores (tcgen05, sm_103a).
//
// What it computes ("vLLM engine anatomy": PagedAttention section and Figure
// 2 for the paging, Table 1 for GQA; "vLLM V1 engine architecture" for
// chunked prefill; "Boundaries: FlashAttention ..." for exact attention with
// an online softmax): for every query row of a prefill-class request (query
// token i of n, q head h of KV head g = h / G), softmax attention over the
// request's keys 0 .. L - n + i, read through the block table from 16-token
// pages.  Decode-class requests are left to the attention kernel of
// attn_fast.cu.
//
// How (one CTA per SM, persistent over the step's prefill tiles):
//  * A tile is 128 query rows of one (request, KV head): 128 / G consecutive
//    tokens times the G q heads of the group, row = token * G + head.  Keys
//    go in chunks of 128 (8 pages).  Warp 8 draws tiles (from a step-wide
//    counter, longest first, or in a fixed snake), decodes each and passes
//    it to the other warps through a two-slot ring in shared memory.
//  * warps 8 and 9 (TMA producers): the Q tile through a 3-D map over q
//    [token][head][dim] and, for every chunk, its pages of K (warp 8) and of
//    V (warp 9) through 2-D maps over the cache rows, each page as two
//    64-column halves under the 128-byte swizzle, into rings two (K) and
//    two (V) chunks deep.  The two rings advance independently, so K runs
//    ahead of the P.V that frees the V stages.  The same shared-memory
//    layout serves as the K-major B operand of Q.K^T and as the MN-major B
//    operand of P.V.  Block-table rows come a group of four chunks ahead.
//  * warps 10 and 11 (MMA): warp 10 allocates tensor memory (512 columns:
//    three S buffers and O) and issues S = Q.K^T (M 128, N = 16 x pages of
//    the chunk, K 128) into the S buffer of the chunk; warp 11 issues
//    O += P.V with P read from tensor memory, where the softmax wrote it over
//    that chunk's S.  Each warp issues its MMAs from one elected lane of the
//    converged warp, eight per asm block, so that the softmax warps sharing
//    its SM sub-partition do not slow the issue below the tensor rate.
//    P goes in two 16-bit parts, P = hi + lo, so that the rounding of the
//    probabilities to 16 bits costs no accuracy.  Completion is tracked with
//    tcgen05.commit on mbarriers;
//    with three buffers the softmax of one chunk overlaps the MMAs of its
//    neighbours.
//  * warps 0-7 (softmax): two threads per query row, one per half of the
//    key columns (warps w and w + 4 share lane quarter w % 4 of tensor
//    memory).  Each chunk: S from tensor memory, causal mask, online softmax
//    against a reference max that only moves when the row max has grown by
//    more than 2^8 (O is then rescaled in tensor memory; otherwise the
//    exponentials stay below 2^8), P into tensor memory; key pairs in packed
//    fp32x2 arithmetic.  At the end of the tile: O / l in the output type.
//  * V rows of the request's last page that lie past the sequence end are
//    cleared in shared memory before P.V (their P is 0, but 0 x NaN is not).
//
// Every wait is bounded; on a timeout the CTA records PA_DEV_ERR_TIMEOUT,
// lets its copies and MMAs in flight finish, frees its tensor memory and
// returns.
#include <float.h>

#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "tcgen05.cuh"

namespace pa {
namespace {

constexpr int kTcRows = 128;               // query rows of a tile (MMA M)
constexpr int kTcKeys = 128;               // keys of a chunk
constexpr int kTcPages = kTcKeys / kBS;    // pages of a chunk
#ifndef PA_TC_SOFTMAX_WARPS
#define PA_TC_SOFTMAX_WARPS 8
#endif
constexpr int kSoftmaxWarps = PA_TC_SOFTMAX_WARPS;  // 8 or 16: 2 or 4 per row quarter
constexpr int kParts = kSoftmaxWarps / 4;           // warps sharing a row
constexpr int kPartCols = 128 / kParts;             // a part's columns of a chunk
static_assert(kParts == 2 || kParts == 4, "two or four softmax warps per row quarter");
constexpr int kKWarp = kSoftmaxWarps;      // tiles, Q and K
constexpr int kVWarp = kSoftmaxWarps + 1;  // V
constexpr int kQkWarp = kSoftmaxWarps + 2; // S = Q.K^T MMAs (owns TMEM)
constexpr int kPvWarp = kSoftmaxWarps + 3; // O += P.V MMAs
constexpr int kTcThreads = (kSoftmaxWarps + 4) * 32;
constexpr int kHalf = 128 * 128;           // 128 rows x 128 B: one column half
constexpr int kTileBytes = 2 * kHalf;      // 128 rows x 128 columns, 16-bit
constexpr int kPageHalf = kBS * 128;       // one page, one column half
constexpr float kRescaleLog2 = 8.f;        // lazy rescale threshold (log2)
constexpr int kTcMaxSeqs = 1024;           // requests of a step it plans itself
#ifndef PA_TC_K_STAGES
#define PA_TC_K_STAGES 2
#endif
#ifndef PA_TC_V_STAGES
#define PA_TC_V_STAGES 2
#endif
#ifndef PA_TC_Q_STAGES
#define PA_TC_Q_STAGES 1
#endif
constexpr int kKStages = PA_TC_K_STAGES;  // ring depth in chunks, K
constexpr int kVStages = PA_TC_V_STAGES;  // ring depth in chunks, V
constexpr int kQStages = PA_TC_Q_STAGES;  // Q tiles in shared memory
constexpr int kSBufs = 3;                   // S / P buffers in tensor memory

// Tensor memory: three S buffers of 128 columns; the softmax overwrites each
// with its P (per 16-key MMA step, 8 columns of hi parts then 8 of lo parts),
// which the P.V of the chunk then reads; O after them.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 384;

// barriers
enum : int {
  kQFull = 0,
  kQEmpty = kQFull + kQStages,
  kKFull = kQEmpty + kQStages,
  kKEmpty = kKFull + kKStages,
  kVFull = kKEmpty + kKStages,
  kVEmpty = kVFull + kVStages,
  kSFull = kVEmpty + kVStages,       // S of the buffer written
  kPFull = kSFull + kSBufs,          // P of the buffer written (128 threads)
  kPvDone = kPFull + kSBufs,         // P.V of the buffer done: free, O updated
  kTileFull = kPvDone + kSBufs,      // tile slot filled (index and metadata)
  kTileEmpty = kTileFull + 2,        // slot read by the other 11 warps
  kXchg = kTileEmpty + 2,            // row parts exchanged, per quarter
  kQkDone = kXchg + 4,               // every S MMA has completed
  kPvDone2 = kQkDone + 1,            // every P.V MMA has completed
  // FP8 caches: the bf16 Q tile has landed (before its widening); the two
  // half-chunk staging buffers of E4M3 K pages, then of V pages, have landed
  kQRaw = kPvDone2 + 1,
  kK8Full = kQRaw + 1,
  kV8Full = kK8Full + 2,
  kNumBars = kV8Full + 2
};

constexpr int kSlotInts = 13;  // a tile slot: its index, then the TcTile fields

// FP8 caches: E4M3 pages are staged half a chunk (4 pages) at a time, two
// buffers per cache, and widened to f16 into the K / V stages
constexpr int kHalfChunk8 = 4 * kBS * 128;  // 4 pages of 128 E4M3 bytes a row

template <bool kFp8>
struct TcLayoutT {
  static constexpr int kK = 0;                               // K stages
  static constexpr int kV = kK + kKStages * kTileBytes;      // V stages
  static constexpr int kQ = kV + kVStages * kTileBytes;      // Q tiles
  static constexpr int kBars = kQ + kQStages * kTileBytes;
  static constexpr int kTmemSlot = kBars + 8 * kNumBars;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kTileSlot = kAbort + 4;               // int[2][kSlotInts]
  static constexpr int kXchgSlot = kTileSlot + 2 * kSlotInts * 4;  // float[2][kParts][128]
  // the step's tile list when the kernel plans it: per request, the first
  // tile (x heads) and the tile count; block-scan scratch
  static constexpr int kPlan = kXchgSlot + 2 * kParts * 128 * 4;  // int[2][kTcMaxSeqs]
  static constexpr int kScan = kPlan + 2 * kTcMaxSeqs * 4;   // int[36]
  // FP8: staging (1024-aligned for the swizzled TMA boxes), then the Q rows'
  // power-of-two shifts of the two tile slots (float[2][128])
  static constexpr int kK8 = (kScan + 36 * 4 + 1023) & ~1023;
  static constexpr int kV8 = kK8 + (kFp8 ? 2 * kHalfChunk8 : 0);
  static constexpr int kShift = kV8 + (kFp8 ? 2 * kHalfChunk8 : 0);
  static constexpr int kBytes = kShift + (kFp8 ? 2 * 128 * 4 : 0);
  static constexpr int kSmemBytes = kBytes + 1024;   // + alignment slack
};
using TcLayout = TcLayoutT<false>;
static_assert(TcLayoutT<true>::kSmemBytes <= 227 * 1024, "shared memory budget");
// Each CTA allocates all 512 tensor-memory columns: a second CTA of this
// kernel on the same SM would wait in its allocation.  Its shared memory
// keeps it off (228 KB per SM).
static_assert(2 * TcLayout::kSmemBytes > 228 * 1024, "one CTA per SM");
// the MMA groups move descriptor start addresses by plain adds: the largest
// operand address plus the largest step stays inside the 14-bit field
static_assert(((TcLayout::kQ + kQStages * kTileBytes + 1024) >> 4) + (kHalf >> 4) < (1 << 14),
              "descriptor start-address field");

struct TcParams {
  void* out;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int self_plan;         // 1: list the step's tiles here; 0: the planner's
  const int4* atoms;     // planner's tiles {r, g, tile, pages}, request order
  const int* n_atoms;
  int max_atoms;
  int dec_rows_max;      // requests with more query rows are prefill-class
  int* tile_ctr;         // non-null: tiles drawn from this step-wide counter
                         // (zeroed before the launch), else a fixed order
  int no_dep_wait;       // 1: start without waiting for the grid before (it
                         // produces nothing this kernel reads)
  unsigned* err;
  int64_t num_tokens;
  int64_t num_blocks;
  int max_blocks_per_seq, num_seqs;
  int num_q_heads, num_kv_heads, group;
  int max_query_len, max_seq_len;
  int tokens_per_tile;   // 128 / group
  float score_scale;     // softmax scale * log2(e) (* k_scale for FP8)
  float out_scale;       // 1, or v_scale for FP8
  int window;            // sliding window in keys (kNoWindow: none)
  // shared-prefix (cascade) steps: N > 0 leading block-table entries that
  // every request shares.  The prefix tiles (after the prefill tiles in the
  // list) take the tokens of the decode-class requests, all of whose keys
  // 0 .. 16 N - 1 they see, in casc_splits key ranges (blocks s N / S ..
  // (s + 1) N / S - 1), and write partial rows (O unscaled, m, l) at
  // casc_acc / casc_ml [s * casc_split_rows + token * num_q_heads + q head]
  int cascade_blocks;
  int casc_splits;
  int64_t casc_split_rows;
  float* casc_acc;
  float* casc_ml;
};

// one tile, as every role of the CTA sees it: its keys are the pages
// p0 .. p0 + pages - 1 of the request (p0 > 0 with a sliding window, or in a
// shared-prefix tile's key range).  A shared-prefix tile (casc) reads
// request 0's block-table row: tokens i0 .. i0 + ntok - 1 of the step, every
// one of them seeing all keys of the tile's range cs of the prefix 0 .. L - 1.
struct TcTile {
  int r, g, q0, n, L, i0, ntok, p0, pages, nc, cs;
  bool ok, casc;
};

// Tile li of the step's list, which runs request by request, tile index
// ascending (causal limits growing), KV head fastest: from the planner's
// list, or located in the kernel's own per-request prefix.  Past the n_real
// prefill tiles come the shared-prefix tiles of the first casc_tok tokens
// (key range, then tile index, then KV head fastest).
__device__ __forceinline__ TcTile tc_tile(const TcParams& p, const int* pre,
                                          const int* ntl, int li, int n_real,
                                          int casc_tok) {
  int r, g, tt;
  if (li >= n_real) {
    const int j = li - n_real;
    const int per_split =
        (casc_tok + p.tokens_per_tile - 1) / p.tokens_per_tile * p.num_kv_heads;
    TcTile t{};
    t.casc = true;
    t.cs = j / per_split;
    const int jj = j - t.cs * per_split;
    tt = jj / p.num_kv_heads;
    t.g = jj - tt * p.num_kv_heads;
    t.r = 0;
    t.q0 = 0;
    t.n = casc_tok;
    t.L = p.cascade_blocks * kBS;
    t.i0 = tt * p.tokens_per_tile;
    t.ntok = min(p.tokens_per_tile, casc_tok - t.i0);
    const int S = p.casc_splits;
    t.p0 = (int)((int64_t)t.cs * p.cascade_blocks / S);
    t.pages = (int)((int64_t)(t.cs + 1) * p.cascade_blocks / S) - t.p0;
    t.nc = (t.pages + kTcPages - 1) / kTcPages;
    t.ok = t.ntok > 0 && t.pages > 0 && t.cs < S && p.num_seqs > 0 &&
           p.cascade_blocks <= p.max_blocks_per_seq;
    return t;
  }
  if (p.self_plan) {
    int lo = 0, hi = p.num_seqs - 1;  // last request with pre[r] <= li
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= li) lo = mid; else hi = mid - 1;
    }
    r = lo;
    const int j = li - pre[r];
    tt = j / p.num_kv_heads;
    g = j - tt * p.num_kv_heads;
    if (tt >= ntl[r]) r = -1;  // (cannot happen for li < total)
  } else {
    const int4 at = __ldg(p.atoms + li);
    r = at.x;
    g = at.y;
    tt = at.z;
  }
  TcTile t{};
  t.r = r;
  t.g = g;
  t.ok = r >= 0 && r < p.num_seqs && g >= 0 && g < p.num_kv_heads;
  if (!t.ok) return t;
  const ReqMeta m = load_req(p.qsl, p.seq_lens, t.r, p.num_tokens,
                             p.max_query_len, p.max_seq_len,
                             p.max_blocks_per_seq);
  t.q0 = m.q0;
  t.n = m.n;
  t.L = m.L;
  t.i0 = tt * p.tokens_per_tile;
  t.ntok = min(p.tokens_per_tile, m.n - t.i0);
  t.ok = m.ok && tt >= 0 && t.ntok > 0;
  // keys up to the last token's limit L - n + i0 + ntok - 1, from the first
  // token's first key inside the window (L - n + i0 - window + 1)
  const int end = t.ok ? (t.L - t.n + t.i0 + t.ntok - 1) / kBS + 1 : 0;
  const int lo = t.L - t.n + t.i0 - p.window + 1;
  t.p0 = t.ok && lo > 0 ? lo / kBS : 0;
  t.pages = end - t.p0;
  t.nc = (t.pages + kTcPages - 1) / kTcPages;
  return t;
}

__device__ __forceinline__ bool aborted(volatile int* abort_flag) {
  return __any_sync(~0u, *abort_flag != 0);
}

// Bounded wait by a whole warp; false (and the CTA aborts) on a timeout.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity,
                                          volatile int* abort_flag,
                                          unsigned* err) {
  const bool ok = __all_sync(~0u, mbar_wait_bounded(bar, parity));
  if (!ok && (threadIdx.x & 31) == 0) {
    flag_error(err, PA_DEV_ERR_TIMEOUT);
    *abort_flag = 1;
  }
  return ok;
}

// The step's prefill tiles: per request (prefill-class: more than
// dec_rows_max query rows), ceil(rows / tile rows) tiles per KV head; the
// exclusive prefix of tiles x heads into pre[], the tile counts into ntl[].
// scan[33]: the tokens the shared-prefix tiles take (up to the last token of
// the last decode-class request; 0 without a shared prefix).  All threads
// of the block take part; returns the prefill tiles' total.
__device__ int plan_tiles(const TcParams& p, int* pre, int* ntl, int* scan) {
  const int rows_per_tile = p.tokens_per_tile * p.group;
  int run = 0;
  if (threadIdx.x == 0) scan[33] = 0;
  __syncthreads();
  for (int base = 0; base < p.num_seqs; base += blockDim.x) {
    const int r = base + threadIdx.x;
    int tiles = 0;
    if (r < p.num_seqs) {
      const ReqMeta m = load_req(p.qsl, p.seq_lens, r, p.num_tokens,
                                 p.max_query_len, p.max_seq_len,
                                 p.max_blocks_per_seq);
      if (m.ok && m.n * p.group > p.dec_rows_max)
        tiles = (m.n * p.group + rows_per_tile - 1) / rows_per_tile;
      else if (m.ok && m.n > 0 && p.cascade_blocks > 0)
        atomicMax(scan + 33, m.q0 + m.n);
    }
    const int ex = block_scan_excl<int>(tiles * p.num_kv_heads, scan + 32, scan);
    const int tot = scan[32];
    __syncthreads();
    if (r < p.num_seqs) {
      pre[r] = run + ex;
      ntl[r] = tiles;
    }
    run += tot;
  }
  __syncthreads();
  return run;
}

// k-th tile of CTA b of K: a snake over the list from its end (longest
// tiles first): b, 2K-1-b, 2K+b, ...; -1 past the end
__device__ __forceinline__ int snake_tile(int k, int total) {
  const int K = gridDim.x, b = blockIdx.x;
  const int idx = k * K + ((k & 1) ? K - 1 - b : b);
  return idx < total ? total - 1 - idx : -1;
}

// Tile slots: the warp that draws the tiles decodes each one (its metadata
// takes global reads whose latency would otherwise hit every warp at every
// tile start) and hands it to the other warps through slot k % 2.
__device__ __forceinline__ void put_tile(volatile int* slot, int li, const TcTile& t) {
  slot[0] = li;
  slot[1] = t.r;
  slot[2] = t.g;
  slot[3] = t.q0;
  slot[4] = t.n;
  slot[5] = t.L;
  slot[6] = t.i0;
  slot[7] = t.ntok;
  slot[8] = t.pages;
  slot[9] = t.nc;
  slot[10] = t.ok ? 1 : 0;
  slot[11] = t.p0;
  slot[12] = t.casc ? 1 + t.cs : 0;
}

// The k-th tile of a warp that does not draw tiles, from slot k % 2; the
// index is -1 when there are no more (or on a timeout).  shifts (FP8
// caches, softmax warps): the slot's per-row Q shifts, of which row's is
// copied to *shift before the slot is released.
__device__ __forceinline__ int follow_tile(const TcParams& p, uint32_t bars,
                                           volatile int* slots, int k,
                                           volatile int* abort_flag, TcTile& t,
                                           const volatile float* shifts = nullptr,
                                           int row = 0, float* shift = nullptr) {
  const int s = k & 1;
  if (!warp_wait(bars + 8 * (kTileFull + s), (k >> 1) & 1, abort_flag, p.err))
    return -1;
  volatile int* sl = slots + s * kSlotInts;
  const int li = sl[0];
  t.r = sl[1];
  t.g = sl[2];
  t.q0 = sl[3];
  t.n = sl[4];
  t.L = sl[5];
  t.i0 = sl[6];
  t.ntok = sl[7];
  t.pages = sl[8];
  t.nc = sl[9];
  t.ok = sl[10] != 0;
  t.p0 = sl[11];
  t.casc = sl[12] != 0;
  t.cs = t.casc ? sl[12] - 1 : 0;
  if (shifts != nullptr) *shift = shifts[s * 128 + row];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bars + 8 * (kTileEmpty + s));
  return li;
}

// Probabilities as two 16-bit parts each, p = hi + lo + O(2^-14 p): for bf16
// hi keeps the top half of the fp32 bits and lo the top half of the
// remainder p - hi (which is exact), both by truncation, so the split takes
// no conversion instructions; for f16 both parts are rounded to nearest.
template <bool kBF16>
__device__ __forceinline__ void split_pair(float2 pr, uint32_t& hi, uint32_t& lo) {
  const float a = pr.x, b = pr.y;
  if constexpr (kBF16) {
    const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
    hi = __byte_perm(ua, ub, 0x7632);
    // remainder p - hi, exact, as one packed fma
    const float2 r = __ffma2_rn(make_float2(__uint_as_float(ua & 0xFFFF0000u),
                                            __uint_as_float(ub & 0xFFFF0000u)),
                                make_float2(-1.f, -1.f), pr);
    lo = __byte_perm(__float_as_uint(r.x), __float_as_uint(r.y), 0x7632);
  } else {
    hi = pack2<false>(a, b);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hi));
    lo = pack2<false>(a - f.x, b - f.y);
  }
}

// 32 bytes (eight words from r[first]) to a 32-byte aligned global address
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t (&r)[16],
                                             int first) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst),
               "r"(r[first]), "r"(r[first + 1]), "r"(r[first + 2]), "r"(r[first + 3]),
               "r"(r[first + 4]), "r"(r[first + 5]), "r"(r[first + 6]), "r"(r[first + 7])
               : "memory");
}

// max of three (one instruction)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 2^x by the hardware approximation (relative error about 2^-22; results
// below 2^-126 flush to zero, which a softmax weight next to l >= 1 is)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// FP8 caches: widen np (<= 4) staged E4M3 pages -- 16 rows of 128 bytes
// each, 16-byte chunk k of row t at chunk k ^ (t & 7) as the TMA wrote it --
// to f16 rows p0 * 16 .. of a K / V stage (two 64-column halves of 128-byte
// rows under the same swizzle), exactly.  One warp, 16-byte units.
__device__ __forceinline__ void widen_pages(const uint8_t* src, uint8_t* stage,
                                            int p0, int np, int lane) {
  // lane: 16-byte chunk k = lane & 7 of rows t = t0 + 4 i of each page;
  // the chunk's column half and its f16 chunks are the same in every row.
  // The upper-half lanes take row t ^ 1: the two halves lie 16 KB apart (the
  // same banks), and the swizzle of the neighbouring row puts the 8 lanes of
  // each quarter-warp on 8 different bank groups, for the loads and for both
  // stores (otherwise every store costs two wavefronts per quarter-warp)
  const int k = lane & 7;
  const int hh = k >> 2, j0 = 2 * (k & 3);
  const int t0 = (lane >> 3) ^ hh;
  const uint8_t* s0 = src + t0 * 128;
  uint8_t* d0 = stage + hh * kHalf + (p0 * kBS + t0) * 128;
  for (int pg = 0; pg < np; ++pg) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = t0 + 4 * i;  // row in the page; (p0 + pg) * 16 + t in the stage
      const uint4 v = *reinterpret_cast<const uint4*>(s0 + pg * (kBS * 128) + i * 512 +
                                                       ((k ^ (t & 7)) << 4));
      uint32_t f[8];
      e4m3x4_to_f16x2x2(v.x, f[0], f[1]);
      e4m3x4_to_f16x2x2(v.y, f[2], f[3]);
      e4m3x4_to_f16x2x2(v.z, f[4], f[5]);
      e4m3x4_to_f16x2x2(v.w, f[6], f[7]);
      uint8_t* row = d0 + pg * (kBS * 128) + i * 512;
      *reinterpret_cast<uint4*>(row + ((j0 ^ (t & 7)) << 4)) =
          make_uint4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<uint4*>(row + (((j0 + 1) ^ (t & 7)) << 4)) =
          make_uint4(f[4], f[5], f[6], f[7]);
    }
  }
}

// FP8 caches, bf16 q: widen the Q tile (128 rows of two 64-column halves)
// to f16 in place, each row scaled by 2^-e so that its largest |q| stays
// inside the f16 range (e = 0 unless it exceeds 2^14); 2^e goes to
// shifts[row], for the softmax to undo on the scores.  One warp.
__device__ __forceinline__ void widen_q(uint8_t* q, float* shifts, int lane) {
  for (int R = lane; R < 128; R += 32) {
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint4 v = *reinterpret_cast<const uint4*>(q + (j >> 3) * kHalf + R * 128 +
                                                      (((j & 7) ^ (R & 7)) << 4));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
      }
    }
    int e = 0;
    if (amax > 16384.f) e = ilogbf(amax) - 13;
    const float down = exp2f((float)-e);
    shifts[R] = exp2f((float)e);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      uint4* a = reinterpret_cast<uint4*>(q + (j >> 3) * kHalf + R * 128 +
                                          (((j & 7) ^ (R & 7)) << 4));
      const uint4 v = *a;
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        o[i] = pack2<false>(__uint_as_float(w[i] << 16) * down,
                            __uint_as_float(w[i] & 0xFFFF0000u) * down);
      *a = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// kBF16: q and out are bf16 (else f16).  kFp8: the caches hold E4M3, which
// the producer warps widen to f16; the MMAs then run in f16 (Q widened too).
template <bool kBF16, bool kFp8>
__global__ void __launch_bounds__(kTcThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ TcParams p) {
  using TOut = typename std::conditional<kBF16, __nv_bfloat16, __half>::type;
  using Ly = TcLayoutT<kFp8>;
  constexpr bool kMma = kBF16 && !kFp8;  // bf16 MMA operands (else f16)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const sp = smem_raw + (base - raw);
  const uint32_t bars = base + TcLayout::kBars;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sp + TcLayout::kAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t count = 1;
      if (i >= kPFull && i < kPFull + kSBufs) count = kSoftmaxWarps * 32;
      if (i >= kXchg && i < kXchg + 4) count = kParts * 32;
      if (i == kTileEmpty || i == kTileEmpty + 1) count = kSoftmaxWarps + 3;
      mbar_init(bars + 8 * i, count);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kQkWarp) tc_alloc<kTmemCols>(base + TcLayout::kTmemSlot);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem =
      *reinterpret_cast<volatile uint32_t*>(sp + TcLayout::kTmemSlot);
  // The step's inputs (and the planner's list) are complete.  When this grid
  // follows the decode kernel of the step it need not wait for it: that
  // kernel let it start only after everything before it was complete.  The
  // grid behind this one may start once every CTA is past this wait.
  if (!p.no_dep_wait) pdl_wait();
  pdl_launch_dependents();
  volatile int* slots = reinterpret_cast<volatile int*>(sp + TcLayout::kTileSlot);
  int* const pre = reinterpret_cast<int*>(sp + TcLayout::kPlan);
  int* const ntl = pre + kTcMaxSeqs;
  const int n_real =
      p.self_plan ? plan_tiles(p, pre, ntl, reinterpret_cast<int*>(sp + TcLayout::kScan))
                  : min(*p.n_atoms, p.max_atoms);
  // shared-prefix tiles after the prefill tiles (self-planned steps only)
  const int casc_tok =
      p.self_plan ? reinterpret_cast<const int*>(sp + TcLayout::kScan)[33] : 0;
  const int n_tiles =
      n_real + (casc_tok > 0 ? (casc_tok + p.tokens_per_tile - 1) / p.tokens_per_tile *
                                   p.num_kv_heads * p.casc_splits
                             : 0);

  // Cache rows of the tile's pages 32 G .. 32 G + 31 (four chunks), one
  // page per lane, checked against the pool.  The producers fetch the next
  // group while they issue the current one: under the step's L2 traffic a
  // block-table read fetched at its own chunk would hold the producer for
  // about a chunk's time.
  static_assert(kTcPages * 4 == 32, "four chunks per group of rows");
  auto group_rows = [&](const TcTile& t, int grp) -> int {
    int row = 0;
    const int pg = grp * 32 + lane;
    if (pg < t.pages) {
      int blk = __ldg(p.block_tables + (int64_t)t.r * p.max_blocks_per_seq + t.p0 + pg);
      if (blk < 0 || blk >= p.num_blocks) {
        flag_error(p.err, PA_DEV_ERR_BLOCK_ID);
        blk = 0;
      }
      row = (blk * p.num_kv_heads + t.g) * kBS;
    }
    return row;
  };
  // lanes < pages of chunk c: their page's row, from the group held in cur
  auto chunk_rows = [&](int cur, int c) -> int {
    return __shfl_sync(~0u, cur, ((c & 3) << 3) | (lane & 7));
  };
  // one chunk of K or V: np pages, two 64-column halves each
  auto load_chunk = [&](const CUtensorMap* map, uint32_t dst, uint32_t full,
                        int np, int row) {
    if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)np * 2u * kPageHalf);
    __syncwarp();
    if (lane < np) {
      tma_load_2d(dst + lane * kPageHalf, map, full, 0, row);
      tma_load_2d(dst + kHalf + lane * kPageHalf, map, full, 64, row);
    }
  };

  // FP8 caches: stream a tile's chunks of E4M3 pages through the two
  // half-chunk staging buffers (8-byte barriers at bar8, bar8 + 8): the next
  // chunk's half is in flight while this half is widened into the f16 stage.
  // n8i / n8c: loads issued into / consumed from each buffer so far.
  // Returns false on a timeout.
  auto stream_fp8 = [&](const TcTile& t, const CUtensorMap* map, uint32_t stage0,
                        int nstages, uint32_t full0, uint32_t empty0,
                        uint8_t* stg8, uint32_t bar8, uint32_t& u, uint32_t* used,
                        uint32_t (&n8i)[2], uint32_t (&n8c)[2]) -> bool {
    auto half_pages = [&](int c, int h) {
      return max(0, min(4, t.pages - c * kTcPages - 4 * h));
    };
    auto issue = [&](int c, int h, int rows) {
      const int np = half_pages(c, h);
      if (np == 0) return;
      if (lane == 0) mbar_arrive_expect_tx(bar8 + 8 * h, (uint32_t)np * kBS * 128u);
      __syncwarp();
      const int pg = lane & 7;
      if (lane < 8 && pg >= 4 * h && pg < 4 * h + np)
        tma_load_2d(smem_u32(stg8 + h * kHalfChunk8 + (pg - 4 * h) * (kBS * 128)), map,
                    bar8 + 8 * h, 0, rows);
      ++n8i[h];
    };
    int cur = group_rows(t, 0), nxt = t.nc > 4 ? group_rows(t, 1) : 0;
    {
      const int r0 = chunk_rows(cur, 0);
      issue(0, 0, r0);
      issue(0, 1, r0);
    }
    for (int c = 0; c < t.nc; ++c, ++u) {
      if (c > 0 && (c & 3) == 0) {
        cur = nxt;
        nxt = c + 4 < t.nc ? group_rows(t, (c >> 2) + 1) : 0;
      }
      const int st = u % nstages;
      if (u >= (uint32_t)nstages &&
          !warp_wait(empty0 + 8 * st, ((u / nstages) & 1) ^ 1, abort_flag, p.err))
        return false;
      const int rows_next =
          c + 1 < t.nc ? chunk_rows(((c + 1) & 3) == 0 ? nxt : cur, c + 1) : 0;
      uint8_t* stage = sp + (stage0 - base) + st * kTileBytes;
      for (int h = 0; h < 2; ++h) {
        const int np = half_pages(c, h);
        if (np == 0) continue;
        if (!warp_wait(bar8 + 8 * h, n8c[h] & 1, abort_flag, p.err)) return false;
        ++n8c[h];
        widen_pages(stg8 + h * kHalfChunk8, stage, 4 * h, np, lane);
        __syncwarp();  // the buffer is read: the next half may land in it
        if (c + 1 < t.nc) issue(c + 1, h, rows_next);
      }
      fence_proxy_async_smem();  // the stage is read by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(full0 + 8 * st);
      ++used[st];
    }
    return true;
  };
  // copies still in flight in the staging buffers (after a timeout)
  auto drain_fp8 = [&](uint32_t bar8, const uint32_t (&n8i)[2], const uint32_t (&n8c)[2]) {
    if (lane == 0)
      for (int h = 0; h < 2; ++h)
        if (n8i[h] > n8c[h]) mbar_wait_bounded(bar8 + 8 * h, (n8i[h] - 1) & 1);
  };

  if (warp == kKWarp) {
    // ------------------------- producer: tiles, Q, K -------------------------
    if (lane == 0) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
    }
    const uint32_t q_bytes = 2u * 64u * (uint32_t)G * p.tokens_per_tile * 2u;
    uint32_t u = 0, qt = 0, nq_raw = 0;
    uint32_t used[kKStages] = {};  // loads issued into each stage
    uint32_t n8i[2] = {0u, 0u}, n8c[2] = {0u, 0u};
    const long long skip = skipped_copy();
    bool go = true;
    for (int k = 0; go; ++k) {
      // draw the next tile (longest first: from the step-wide counter, else
      // the fixed snake), decode it and hand it to the other warps through
      // slot k % 2
      const int s = k & 1;
      if (k >= 2 &&
          !warp_wait(bars + 8 * (kTileEmpty + s), ((k >> 1) - 1) & 1, abort_flag, p.err))
        break;
      int li;
      if (p.tile_ctr != nullptr) {
        li = -1;
        if (lane == 0) {
          const int ticket = *abort_flag ? n_tiles : atomicAdd(p.tile_ctr, 1);
          li = ticket < n_tiles ? n_tiles - 1 - ticket : -1;
        }
        li = __shfl_sync(~0u, li, 0);
      } else {
        li = snake_tile(k, n_tiles);
      }
      TcTile t{};
      if (li >= 0) t = tc_tile(p, pre, ntl, li, n_real, casc_tok);
      const uint32_t qb = qt % kQStages;
      bool q_ready = false;
      if constexpr (kFp8) {
        // Q first, widened to f16 (with its rows' shifts, handed over in the
        // tile slot) before the tile is published
        if (li >= 0 && t.ok && !aborted(abort_flag)) {
          if (qt >= (uint32_t)kQStages &&
              !warp_wait(bars + 8 * (kQEmpty + qb), ((qt / kQStages) - 1) & 1, abort_flag,
                         p.err))
            break;
          const uint32_t qd = base + TcLayout::kQ + qb * kTileBytes;
          if (lane == 0) {
            mbar_arrive_expect_tx(bars + 8 * kQRaw, q_bytes);
            tma_load_3d(qd, &tmap_q, bars + 8 * kQRaw, 0, t.g * G, t.q0 + t.i0);
            tma_load_3d(qd + kHalf, &tmap_q, bars + 8 * kQRaw, 64, t.g * G, t.q0 + t.i0);
          }
          ++nq_raw;
          if (!warp_wait(bars + 8 * kQRaw, (nq_raw - 1) & 1, abort_flag, p.err)) break;
          float* shifts = reinterpret_cast<float*>(sp + Ly::kShift) + s * 128;
          if constexpr (kBF16) {
            widen_q(sp + TcLayout::kQ + qb * kTileBytes, shifts, lane);
          } else {
            for (int R = lane; R < 128; R += 32) shifts[R] = 1.f;
          }
          fence_proxy_async_smem();
          __syncwarp();
          q_ready = true;
        }
      }
      if (lane == 0) {
        put_tile(slots + s * kSlotInts, li, t);
        mbar_arrive(bars + 8 * (kTileFull + s));
        if (q_ready) mbar_arrive(bars + 8 * (kQFull + qb));
      }
      __syncwarp();
      if (li < 0 || aborted(abort_flag)) break;
      if (!t.ok) continue;
      if constexpr (kFp8) {
        ++qt;
        if (!stream_fp8(t, &tmap_k, base + TcLayout::kK, kKStages, bars + 8 * kKFull,
                        bars + 8 * kKEmpty, sp + Ly::kK8, bars + 8 * kK8Full, u, used, n8i,
                        n8c)) {
          go = false;
          break;
        }
        continue;
      }
      // Q of this CTA's tile qt into buffer qt % kQStages, once the S MMAs of
      // the tile that last used it have completed
      if (qt >= (uint32_t)kQStages &&
          !warp_wait(bars + 8 * (kQEmpty + qb), ((qt / kQStages) - 1) & 1, abort_flag,
                     p.err))
        break;
      if (lane == 0) {
        const uint32_t fb = bars + 8 * (kQFull + qb);
        const uint32_t qd = base + TcLayout::kQ + qb * kTileBytes;
        mbar_arrive_expect_tx(fb, q_bytes);
        tma_load_3d(qd, &tmap_q, fb, 0, t.g * G, t.q0 + t.i0);
        tma_load_3d(qd + kHalf, &tmap_q, fb, 64, t.g * G,
                    t.q0 + t.i0);
      }
      ++qt;
      int cur = group_rows(t, 0), nxt = t.nc > 4 ? group_rows(t, 1) : 0;
      for (int c = 0; c < t.nc; ++c, ++u) {
        if (c > 0 && (c & 3) == 0) {
          cur = nxt;
          nxt = c + 4 < t.nc ? group_rows(t, (c >> 2) + 1) : 0;
        }
        const int st = u % kKStages;
        const int np = min(kTcPages, t.pages - c * kTcPages);
        const int row = chunk_rows(cur, c);
        if (u >= kKStages &&
            !warp_wait(bars + 8 * (kKEmpty + st), ((u / kKStages) & 1) ^ 1,
                       abort_flag, p.err)) {
          go = false;
          break;
        }
        if ((long long)u == skip) continue;  // testing hook: never issued
        load_chunk(&tmap_k, base + TcLayout::kK + st * kTileBytes,
                   bars + 8 * (kKFull + st), np, row);
        ++used[st];
      }
    }
    // let every copy this warp issued land before the CTA may exit
    if constexpr (kFp8) {
      drain_fp8(bars + 8 * kK8Full, n8i, n8c);
      if (lane == 0 && nq_raw > 0) mbar_wait_bounded(bars + 8 * kQRaw, (nq_raw - 1) & 1);
    } else {
      for (int st = 0; st < kKStages; ++st)
        if (used[st] > 0)
          mbar_wait_bounded(bars + 8 * (kKFull + st), (used[st] - 1) & 1);
      for (uint32_t qb = 0; qb < (uint32_t)kQStages; ++qb) {
        const uint32_t n = qt > qb ? (qt - qb + kQStages - 1) / kQStages : 0;  // loads into qb
        if (n > 0) mbar_wait_bounded(bars + 8 * (kQFull + qb), (n - 1) & 1);
      }
    }
  } else if (warp == kVWarp) {
    // ----------------------------- producer: V ------------------------------
    if (lane == 0) tma_prefetch_desc(&tmap_v);
    uint32_t u = 0;
    uint32_t used[kVStages] = {};
    uint32_t n8i[2] = {0u, 0u}, n8c[2] = {0u, 0u};
    bool go = true;
    for (int k = 0; go; ++k) {
      TcTile t;
      const int li = follow_tile(p, bars, slots, k, abort_flag, t);
      if (li < 0 || aborted(abort_flag)) break;
      if (!t.ok) continue;
      if constexpr (kFp8) {
        if (!stream_fp8(t, &tmap_v, base + TcLayout::kV, kVStages, bars + 8 * kVFull,
                        bars + 8 * kVEmpty, sp + Ly::kV8, bars + 8 * kV8Full, u, used, n8i,
                        n8c))
          go = false;
        continue;
      }
      int cur = group_rows(t, 0), nxt = t.nc > 4 ? group_rows(t, 1) : 0;
      for (int c = 0; c < t.nc; ++c, ++u) {
        if (c > 0 && (c & 3) == 0) {
          cur = nxt;
          nxt = c + 4 < t.nc ? group_rows(t, (c >> 2) + 1) : 0;
        }
        const int st = u % kVStages;
        const int np = min(kTcPages, t.pages - c * kTcPages);
        const int row = chunk_rows(cur, c);
        if (u >= kVStages &&
            !warp_wait(bars + 8 * (kVEmpty + st), ((u / kVStages) & 1) ^ 1,
                       abort_flag, p.err)) {
          go = false;
          break;
        }
        load_chunk(&tmap_v, base + TcLayout::kV + st * kTileBytes,
                   bars + 8 * (kVFull + st), np, row);
        ++used[st];
      }
    }
    if constexpr (kFp8) {
      drain_fp8(bars + 8 * kV8Full, n8i, n8c);
    } else {
      for (int st = 0; st < kVStages; ++st)
        if (used[st] > 0)
          mbar_wait_bounded(bars + 8 * (kVFull + st), (used[st] - 1) & 1);
    }
  } else if (warp == kQkWarp) {
    // ----------------------------- S = Q.K^T ------------------------------
    // The two MMA streams are issued by two warps: a tcgen05.mma keeps its
    // issuing thread busy for about twice the time the tensor core needs
    // for an N = 128 MMA, so one issuer could keep it only half busy.
    uint32_t u = 0, qt = 0;
    for (int k = 0;; ++k) {
      TcTile t;
      const int li = follow_tile(p, bars, slots, k, abort_flag, t);
      if (li < 0 || aborted(abort_flag)) break;
      if (!t.ok) continue;
      const uint32_t qb = qt % kQStages;
      if (!warp_wait(bars + 8 * (kQFull + qb), (qt / kQStages) & 1, abort_flag, p.err))
        break;
      const uint32_t q_s = base + TcLayout::kQ + qb * kTileBytes;
      ++qt;
      bool go = true;
      for (int c = 0; c < t.nc; ++c) {
        // S of chunk uu into buffer uu % 3, once the P.V that last read
        // that buffer has completed
        const uint32_t uu = u + c;
        const int st = uu % kKStages;
        const int b = uu % kSBufs;
        if (!warp_wait(bars + 8 * (kKFull + st), (uu / kKStages) & 1, abort_flag, p.err) ||
            (uu >= kSBufs &&
             !warp_wait(bars + 8 * (kPvDone + b), ((uu / kSBufs) - 1) & 1, abort_flag,
                        p.err))) {
          go = false;
          break;
        }
        tc_fence_after();
        {
          // the whole warp: one elected lane issues the group
          const int np = min(kTcPages, t.pages - c * kTcPages);
          const uint32_t idesc = tc_idesc_f16(kMma, false, kTcRows, np * kBS);
          const uint32_t k_s = base + TcLayout::kK + st * kTileBytes;
          tc_mma_ss_k128<kHalf>(tmem + b * 128, tc_desc_sw128(q_s, 16, 1024),
                                tc_desc_sw128(k_s, 16, 1024), idesc);
          tc_commit_elect(bars + 8 * (kSFull + b));
          tc_commit_elect(bars + 8 * (kKEmpty + st));
          if (c + 1 == t.nc) tc_commit_elect(bars + 8 * (kQEmpty + qb));  // Q is free then
        }
        __syncwarp();
      }
      if (!go) break;
      u += t.nc;
    }
    // every MMA issued has completed before tensor memory is freed
    __syncwarp();
    tc_commit_elect(bars + 8 * kQkDone);
    mbar_wait_bounded(bars + 8 * kQkDone, 0);
  } else if (warp == kPvWarp) {
    // ------------------------------ O += P.V ------------------------------
    const uint32_t idesc_pv = tc_idesc_f16(kMma, true, kTcRows, 128);
    uint32_t u = 0;
    for (int k = 0;; ++k) {
      TcTile t;
      const int li = follow_tile(p, bars, slots, k, abort_flag, t);
      if (li < 0 || aborted(abort_flag)) break;
      if (!t.ok) continue;
      const int last = (t.L - 1) / kBS - t.p0;  // tile page holding the last key
      const int tail = t.L % kBS;               // its keys (0: a full page)
      bool go = true;
      for (int c = 0; c < t.nc; ++c) {
        const uint32_t uu = u + c;
        const int sv = uu % kVStages;
        const int b = uu % kSBufs;
        if (!warp_wait(bars + 8 * (kPFull + b), (uu / kSBufs) & 1, abort_flag, p.err) ||
            !warp_wait(bars + 8 * (kVFull + sv), (uu / kVStages) & 1, abort_flag, p.err)) {
          go = false;
          break;
        }
        tc_fence_after();
        const int pg0 = c * kTcPages;
        const int np = min(kTcPages, t.pages - pg0);
        if (tail != 0 && last >= pg0 && last < pg0 + np) {
          // V rows past the sequence end (whatever the cache holds there)
          uint8_t* vp = sp + TcLayout::kV + sv * kTileBytes + (last - pg0) * kPageHalf;
          const int nrow = kBS - tail;
          for (int i = lane; i < nrow * 16; i += 32) {
            const int rr = tail + (i >> 4), ch = i & 15;
            *reinterpret_cast<uint4*>(vp + (ch >> 3) * kHalf + rr * 128 +
                                      (ch & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        {
          // the whole warp: one elected lane issues four pages (8 MMAs) per
          // group, single pages for the rest of a short chunk
          const uint64_t bv =
              tc_desc_sw128(base + TcLayout::kV + sv * kTileBytes, kHalf, 1024);
          const uint32_t t_p = tmem + b * 128;
          int pp = 0;
          for (; pp + 4 <= np; pp += 4)
            tc_mma_ts_pair4<kPageHalf>(tmem + kColO, t_p + pp * 16,
                                       bv + (uint64_t)(pp * (kPageHalf >> 4)), idesc_pv,
                                       (c > 0 || pp > 0) ? 1u : 0u);
          for (; pp < np; ++pp)
            tc_mma_ts_pair1(tmem + kColO, t_p + pp * 16,
                            bv + (uint64_t)(pp * (kPageHalf >> 4)), idesc_pv,
                            (c > 0 || pp > 0) ? 1u : 0u);
          tc_commit_elect(bars + 8 * (kVEmpty + sv));
          tc_commit_elect(bars + 8 * (kPvDone + b));
        }
        __syncwarp();
      }
      if (!go) break;
      u += t.nc;
    }
    __syncwarp();
    tc_commit_elect(bars + 8 * kPvDone2);
    mbar_wait_bounded(bars + 8 * kPvDone2, 0);
  } else {
    // ------------------------------ softmax -------------------------------
    // Warps w, w + 4, ... share the rows of lane quarter w % 4: warp w + 4 k
    // takes key columns kPartCols k .. kPartCols (k + 1) - 1 of every chunk.
    // The parts of a row trade their partial max every chunk (and their
    // partial sums at the end of the tile) through shared memory, on a
    // per-quarter mbarrier.
    constexpr int kJ = kPartCols / 32;  // 32-column groups of a part
    const int quarter = warp & 3, part = warp >> 2;
    const int row = quarter * 32 + lane;  // tensor-memory lane
    const uint32_t lrow = (uint32_t)(quarter * 32) << 16;
    const uint32_t t_o = tmem + lrow + kColO + part * kPartCols;
    const uint32_t xbar = bars + 8 * (kXchg + quarter);
    float* xslot = reinterpret_cast<float*>(sp + TcLayout::kXchgSlot);
    const int it = row / G, jh = row - it * G;
    uint32_t u = 0, xk = 0;  // chunks done, exchanges done
    // every part's value of this exchange (bounded wait); false on a timeout
    auto exchange = [&](float mine, float (&all)[kParts]) -> bool {
      float* sl = xslot + (xk & 1) * (kParts * 128);
      sl[part * 128 + row] = mine;
      mbar_arrive(xbar);
      const bool ok = warp_wait(xbar, xk & 1, abort_flag, p.err);
#pragma unroll
      for (int q = 0; q < kParts; ++q) all[q] = sl[q * 128 + row];
      ++xk;
      return ok;
    };
    const volatile float* qshifts =
        kFp8 ? reinterpret_cast<const volatile float*>(sp + Ly::kShift) : nullptr;
    for (int k = 0;; ++k) {
      TcTile t;
      float qshift = 1.f;  // FP8 caches: 2^e of this row's Q widening
      const int li = follow_tile(p, bars, slots, k, abort_flag, t, qshifts, row, &qshift);
      if (li < 0 || aborted(abort_flag)) break;
      if (!t.ok) continue;
      const float sscale = p.score_scale * qshift;
      // rows past the tile's tokens compute on the tile's last limit and are
      // never stored
      const bool valid = it < t.ntok;
      // (a shared-prefix tile: every row sees all keys of its range, which
      // also masks the columns of its last chunk past the range)
      const int lim =
          t.casc ? (t.p0 + t.pages) * kBS - 1 : t.L - t.n + t.i0 + (valid ? it : t.ntok - 1);
      float m_ref = -INFINITY, l = 0.f;
      bool go = true;
      for (int c = 0; c < t.nc; ++c) {
        const uint32_t uu = u + c;
        const int b = uu % kSBufs;
        const uint32_t t_b = tmem + lrow + b * 128 + part * kPartCols;
        if (!warp_wait(bars + 8 * (kSFull + b), (uu / kSBufs) & 1, abort_flag, p.err)) {
          go = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[kJ][32];
#pragma unroll
        for (int j = 0; j < kJ; ++j) tc_ld32(t_b + j * 32, sr[j]);
        tc_wait_ld_dep(sr);
        // partial row max of the raw scores (the scale is positive); keys
        // past the row's limit (only in chunks that reach the diagonal) and
        // keys at or before lim - window (only in chunks that reach the
        // window's edge) become -inf
        const int vis = lim - t.p0 * kBS - c * kTcKeys - part * kPartCols;  // columns .. vis
        const int wlo = vis - p.window;  // columns .. wlo out
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (__any_sync(~0u, vis < kPartCols - 1 || wlo >= 0)) {
#pragma unroll
          for (int j = 0; j < kPartCols; ++j)
            if (j > vis || j <= wlo) sr[j >> 5][j & 31] = __float_as_uint(-INFINITY);
        }
#pragma unroll
        for (int j = 0; j < kPartCols; j += 2)
          mx4[(j >> 1) & 3] = fmax3(mx4[(j >> 1) & 3], __uint_as_float(sr[j >> 5][j & 31]),
                                    __uint_as_float(sr[j >> 5][(j & 31) + 1]));
        float mx = fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]);
        float mx_all[kParts];
        if (!exchange(mx, mx_all)) {
          go = false;
          break;
        }
#pragma unroll
        for (int q = 0; q < kParts; ++q) mx = fmaxf(mx, mx_all[q]);  // the same in every part
        const float m_new = fmaxf(m_ref, mx * sscale);
        const bool grow = m_new > m_ref + kRescaleLog2;
        const float alpha = grow ? exp2f(m_ref - m_new) : 1.f;
        if (c > 0 && __any_sync(~0u, grow)) {
          // O is stable once the previous chunk's P.V has completed
          const uint32_t up = uu - 1;
          if (!warp_wait(bars + 8 * (kPvDone + up % kSBufs), (up / kSBufs) & 1,
                         abort_flag, p.err)) {
            go = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int j = 0; j < kJ; ++j) {
            uint32_t o[32];
            tc_ld32(t_o + j * 32, o);
            tc_wait_ld_dep(o);
#pragma unroll
            for (int k = 0; k < 32; ++k)
              o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tc_st32(t_o + j * 32, o);
          }
          tc_wait_st();
        }
        if (grow) {
          l *= alpha;
          m_ref = m_new;
        }
        // P = 2^(s * scale - m_ref) over the S just read, in place: the 16
        // keys of MMA step k take columns 16k .. 16k+7 (hi parts) and
        // 16k+8 .. 16k+15 (lo parts), key pairs packed low key first
        // (key pairs in packed fp32x2 arithmetic)
        const float2 scale2 = make_float2(sscale, sscale);
        // a row that has seen no key yet (a chunk wholly before its window)
        // keeps m_ref = -inf: its scores are all -inf and give P = 0
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        const float2 neg_m2 = make_float2(-m_use, -m_use);
        float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
          uint32_t w[32];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[j][2 * k]),
                                                    __uint_as_float(sr[j][2 * k + 1])),
                                        scale2, neg_m2);
            const float2 pr = make_float2(fast_exp2(x.x), fast_exp2(x.y));
            l2[k & 1] = __fadd2_rn(l2[k & 1], pr);
            const int slot = (k >> 3) * 16 + (k & 7);  // hi at slot, lo at slot + 8
            split_pair<kMma>(pr, w[slot], w[slot + 8]);
          }
          tc_st32(t_b + j * 32, w);
        }
        const float2 lsum = __fadd2_rn(l2[0], l2[1]);
        l += lsum.x + lsum.y;
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(bars + 8 * (kPFull + b));
      }
      if (!go) break;
      // the row sum: every part adds the partial sums in part order
      float l_all[kParts];
      if (!exchange(l, l_all)) break;
      float l_tot = l_all[0];
#pragma unroll
      for (int q = 1; q < kParts; ++q) l_tot += l_all[q];
      const uint32_t ul = u + t.nc - 1;
      if (!warp_wait(bars + 8 * (kPvDone + ul % kSBufs), (ul / kSBufs) & 1,
                     abort_flag, p.err))
        break;
      tc_fence_after();
      const float inv = p.out_scale / l_tot;
      // each thread writes kPartCols contiguous columns of its row: 32-byte
      // stores when the output allows them (row starts are 256 bytes apart)
      const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;
      TOut* o = static_cast<TOut*>(p.out) +
                ((int64_t)(t.q0 + t.i0 + it) * p.num_q_heads + t.g * G + jh) * 128 +
                part * kPartCols;
      // a shared-prefix tile leaves its rows unnormalised, for the merge
      const int64_t crow = (int64_t)t.cs * p.casc_split_rows +
                           (int64_t)(t.q0 + t.i0 + it) * p.num_q_heads + t.g * G + jh;
      if (t.casc && valid && part == 0) {
        p.casc_ml[crow * 2] = m_ref;
        p.casc_ml[crow * 2 + 1] = l_tot;
      }
#pragma unroll 1
      for (int j = 0; j < kJ; ++j) {
        uint32_t v[32];
        tc_ld32(t_o + j * 32, v);
        tc_wait_ld_dep(v);
        if (t.casc) {
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(p.casc_acc + crow * 128 +
                                                    part * kPartCols + j * 32);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              dst[k] = make_float4(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                                   __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]));
          }
        } else if (valid) {
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            pk[k] = pack2<kBF16>(__uint_as_float(v[2 * k]) * inv,
                                 __uint_as_float(v[2 * k + 1]) * inv);
          if (out32) {
            // whole 32-byte sectors, two per 32 columns
            st_global_v8(o + j * 32, pk, 0);
            st_global_v8(o + j * 32 + 16, pk, 8);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(o + j * 32);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
          }
        }
      }
      tc_fence_before();
      u += t.nc;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kQkWarp) {
    tc_fence_after();
    tc_dealloc<kTmemCols>(tmem);
  }
}

template <bool kBF16, bool kFp8>
cudaError_t launch_tc(const TcParams& p, const TcMaps& m, int grid,
                      cudaStream_t stream);

}  // namespace

cudaError_t set_pipeline_hooks_tc(uint64_t wait_limit_ns, long long skip_copy) {
  cudaError_t e = cudaMemcpyToSymbol(g_wait_limit_ns, &wait_limit_ns,
                                     sizeof(wait_limit_ns));
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbol(g_skip_copy, &skip_copy, sizeof(skip_copy));
  return e;
}

namespace {

template <bool kBF16, bool kFp8>
cudaError_t launch_tc(const TcParams& p, const TcMaps& m, int grid,
                      cudaStream_t stream) {
  static bool configured[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(prefill_tc_kernel<kBF16, kFp8>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TcLayoutT<kFp8>::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = TcLayoutT<kFp8>::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, prefill_tc_kernel<kBF16, kFp8>, m.q, m.k, m.v, p);
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace

bool tc_prefill_supported(const AttnArgs& a) {
  const int G = a.num_q_heads / a.num_kv_heads;
  // (the row max is taken on raw scores: the scale must be positive)
  if (!(a.head_dim == 128 && G >= 1 && G <= kTcRows && a.scale > 0.f)) return false;
  if (a.cache_dtype == PA_FP8_E4M3)  // widened to f16 in shared memory
    return a.q_dtype == PA_BF16 || a.q_dtype == PA_F16;
  return (a.cache_dtype == PA_BF16 || a.cache_dtype == PA_F16) &&
         a.q_dtype == a.cache_dtype;
}

int tc_prefill_tile_rows(int group) { return (kTcRows / group) * group; }

cudaError_t launch_prefill_tc(const AttnArgs& a, const TcMaps& maps,
                              bool self_plan, const int4* atoms,
                              const int* n_atoms, int max_atoms,
                              int dec_rows_max, int* tile_ctr, bool after_decode,
                              int num_sms, cudaStream_t stream, float* casc_acc,
                              float* casc_ml, int casc_splits,
                              int64_t casc_split_rows) {
  TcParams p{};
  p.casc_splits = 1;
  if (self_plan && a.cascade_blocks > 0 && casc_acc && casc_ml && casc_splits >= 1) {
    p.cascade_blocks = a.cascade_blocks;
    p.casc_splits = casc_splits;
    p.casc_split_rows = casc_split_rows;
    p.casc_acc = casc_acc;
    p.casc_ml = casc_ml;
  }
  p.out = a.out;
  p.block_tables = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.qsl = a.query_start_loc;
  p.self_plan = self_plan ? 1 : 0;
  p.atoms = atoms;
  p.n_atoms = n_atoms;
  p.max_atoms = max_atoms;
  p.dec_rows_max = dec_rows_max;
  p.tile_ctr = tile_ctr;
  p.no_dep_wait = after_decode ? 1 : 0;
  p.err = a.err;
  p.num_tokens = a.num_tokens;
  p.num_blocks = a.num_blocks;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.max_query_len = a.max_query_len;
  p.max_seq_len = a.max_seq_len;
  p.tokens_per_tile = kTcRows / p.group;
  const bool fp8 = a.cache_dtype == PA_FP8_E4M3;
  p.score_scale = a.scale * 1.4426950408889634f * (fp8 ? a.k_scale : 1.0f);
  p.out_scale = fp8 ? a.v_scale : 1.0f;
  p.window = a.window > 0 ? a.window : kNoWindow;
  int grid = max_atoms < num_sms ? max_atoms : num_sms;
  if (grid < 1) grid = 1;
  const bool qb = a.q_dtype == PA_BF16;
  if (fp8)
    return qb ? launch_tc<true, true>(p, maps, grid, stream)
              : launch_tc<false, true>(p, maps, grid, stream);
  return qb ? launch_tc<true, false>(p, maps, grid, stream)
            : launch_tc<false, false>(p, maps, grid, stream);
}

}  // namespace pa

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
//  * A plan kernel turns (query_start_loc, seq_lens) into a work list on the
//    device: decode-class requests (q_len * group <= 16 rows) are cut into
//    splits of `blocks_per_split` pages along the context (split-K), long
//    prompts into 64-row tiles.  Big items first.
//  * The main kernel runs one work item per CTA: a producer warp walks the
//    block table and streams each (block, KV head) page of K and V into a
//    shared-memory ring with TMA (cp.async.bulk.tensor, 128-byte swizzle),
//    completing on mbarriers; four consumer warps run Q.K^T and P.V on the
//    warp-level tensor-core MMA straight from the swizzled pages, with an
//    fp32 online softmax in registers.  A decode item spreads its pages over
//    the four warps and merges them in shared memory; a prefill tile gives
//    each warp 16 rows and all pages.
//  * A merge kernel combines the splits of a request in a fixed order
//    (deterministic): M = max m_s, out = sum e^{m_s-M} acc_s / sum e^{m_s-M} l_s.
//
// Decode is HBM-bound: every page is read from HBM exactly once per step and
// the MMA only keeps the ALU work (group x 128 MACs per key) off the CUDA
// cores.
#include <float.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

#ifndef PA_NARROW_MIN_BLOCKS
#define PA_NARROW_MIN_BLOCKS 3  // resident CTAs per SM, <= 8-row kernel
#endif
#ifndef PA_SPLIT_MIN_BLOCKS
#define PA_SPLIT_MIN_BLOCKS 16  // smallest decode split, in blocks
#endif
#ifndef PA_SPLIT_WAVES
#define PA_SPLIT_WAVES 16       // target decode items per SM
#endif
#ifndef PA_L2_PREFETCH_PAGES
#define PA_L2_PREFETCH_PAGES 0  // pages prefetched into L2 ahead of the ring (0: off)
#endif
#ifndef PA_STAGES_16BIT
#define PA_STAGES_16BIT 8       // ring depth in pages, bf16 / fp16 caches
#endif

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kPlanThreads = 1024;

// ---------------------------------------------------------------------------
// compile-time traits of the four supported (cache, q) type pairs
// ---------------------------------------------------------------------------
enum : int { kKindBF16 = 0, kKindF16 = 1, kKindFp8BF16 = 2, kKindFp8F16 = 3 };

template <int kKind>
struct Traits {
  static constexpr bool kFp8 = kKind >= kKindFp8BF16;
  static constexpr bool kMmaBF16 = kKind == kKindBF16;  // else f16 MMA
  static constexpr bool kQBF16 = kKind == kKindBF16 || kKind == kKindFp8BF16;
  static constexpr int kRowBytes = kFp8 ? 128 : 256;    // head_dim 128
  static constexpr int kPageBytes = kBS * kRowBytes;    // one (block, head)
  static constexpr int kStageBytes = 2 * kPageBytes;    // K page + V page
  static constexpr int kStages = kFp8 ? 2 * PA_STAGES_16BIT : PA_STAGES_16BIT;
  static constexpr int kRingBytes = kStages * kStageBytes;  // 64 KiB
  // Token order inside an 8-token MMA tile (row n of the tile holds token
  // perm(n)).  Chosen so that the fragment reads of both K and V from the
  // 128-byte-swizzled pages are free of shared-memory bank conflicts.
  static constexpr uint32_t kPerm = kFp8 ? 0x36147250u : 0x57463120u;
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
  const int4* items;
  const int* num_items;
  int* work_counter;     // next unclaimed work item (zeroed by the planner)
  const int* req_nsplit;
  float* ws_acc;
  float* ws_ml;
  unsigned* err;
  int64_t num_tokens;
  int64_t num_blocks;
  int max_blocks_per_seq;
  int num_seqs;
  int num_q_heads, num_kv_heads, group;
  int max_query_len, max_seq_len;
  int blocks_per_split, max_splits;
  int64_t max_items;
  float score_scale;  // softmax scale * log2(e) (* k_scale for FP8)
  float out_scale;    // 1, or v_scale for FP8
};

// ---------------------------------------------------------------------------
// plan kernel: one CTA builds the work list
// ---------------------------------------------------------------------------
struct Counts {
  int pre, full, last;
};

__device__ __forceinline__ Counts block_exclusive_scan(Counts v, Counts* total,
                                                       Counts* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  Counts inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int a = __shfl_up_sync(~0u, inc.pre, d);
    int b = __shfl_up_sync(~0u, inc.full, d);
    int c = __shfl_up_sync(~0u, inc.last, d);
    if (lane >= d) {
      inc.pre += a;
      inc.full += b;
      inc.last += c;
    }
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    Counts w = lane < nw ? warp_sums[lane] : Counts{0, 0, 0};
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int a = __shfl_up_sync(~0u, w.pre, d);
      int b = __shfl_up_sync(~0u, w.full, d);
      int c = __shfl_up_sync(~0u, w.last, d);
      if (lane >= d) {
        w.pre += a;
        w.full += b;
        w.last += c;
      }
    }
    if (lane < nw) warp_sums[lane] = w;  // inclusive warp prefix
    if (lane == nw - 1) *total = w;
  }
  __syncthreads();
  Counts base = warp == 0 ? Counts{0, 0, 0} : warp_sums[warp - 1];
  Counts ex;
  ex.pre = base.pre + inc.pre - v.pre;
  ex.full = base.full + inc.full - v.full;
  ex.last = base.last + inc.last - v.last;
  __syncthreads();  // warp_sums / total reused by the next chunk
  return ex;
}

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(FastParams p, int4* items, int* num_items, int* req_nsplit) {
  __shared__ Counts warp_sums[32];
  __shared__ Counts chunk_total;
  const int G = p.group, H = p.num_kv_heads;
  // pass 1: totals of the three item classes (prefill tiles, full decode
  // splits, last decode splits)
  Counts run{0, 0, 0};
  int total_pre = 0, total_full = 0;
  for (int pass = 0; pass < 2; ++pass) {
    run = Counts{0, 0, 0};
    for (int base = 0; base < p.num_seqs; base += blockDim.x) {
      const int r = base + threadIdx.x;
      Counts c{0, 0, 0};
      int tiles = 0, splits = 0;
      ReqMeta m{0, 0, 0, 0, false};
      if (r < p.num_seqs) {
        m = load_req(p.qsl, p.seq_lens, r, p.num_tokens, p.max_query_len,
                     p.max_seq_len, p.max_blocks_per_seq);
        if (!m.ok) {
          if (pass == 0) flag_error(p.err, PA_DEV_ERR_METADATA);
        } else if (m.n > 0) {
          if (m.n * G <= kDecodeMaxRows) {
            splits = (m.nb + p.blocks_per_split - 1) / p.blocks_per_split;
            c.full = (splits - 1) * H;
            c.last = H;
          } else {
            tiles = (m.n * G + kPrefillTileRows - 1) / kPrefillTileRows;
            c.pre = tiles * H;
          }
        }
        if (pass == 0) req_nsplit[r] = splits;
      }
      Counts ex = block_exclusive_scan(c, &chunk_total, warp_sums);
      if (pass == 1 && r < p.num_seqs) {
        // prefill tiles, last tile (most keys) first
        int o = run.pre + ex.pre;
        for (int tt = tiles - 1; tt >= 0; --tt)
          for (int g = 0; g < H; ++g)
            if (o < p.max_items) items[o++] = make_int4(r, g, kItemPrefill, tt);
        o = total_pre + run.full + ex.full;
        for (int s = 0; s < splits - 1; ++s)
          for (int g = 0; g < H; ++g)
            if (o < p.max_items) items[o++] = make_int4(r, g, kItemDecode, s);
        o = total_pre + total_full + run.last + ex.last;
        if (splits > 0)
          for (int g = 0; g < H; ++g)
            if (o < p.max_items)
              items[o++] = make_int4(r, g, kItemDecode, splits - 1);
      }
      run.pre += chunk_total.pre;
      run.full += chunk_total.full;
      run.last += chunk_total.last;
      __syncthreads();
    }
    total_pre = run.pre;
    total_full = run.full;
  }
  if (threadIdx.x == 0) {
    int64_t n = (int64_t)run.pre + run.full + run.last;
    if (n > p.max_items) {
      flag_error(p.err, PA_DEV_ERR_METADATA);
      n = p.max_items;
    }
    *num_items = (int)n;
    *p.work_counter = 0;
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
          ((int64_t)(q0 + i) * Hq + h) * 128);
    }
    uint4 ch[4];
    if constexpr (!Tr::kFp8) {
      // 16-bit cache: chunk 4j + c of the row (8 elements) feeds k-steps
      // 2j and 2j+1
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ch[j] = valid ? __ldg(src + 4 * j + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
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

// Process one page (16 keys) held in shared memory at k_base / v_base.
template <int kKind, bool kRows16>
__device__ __forceinline__ void process_page(uint32_t k_base, uint32_t v_base,
                                             const uint32_t (&qa)[8][4],
                                             WarpState& st, int key0,
                                             int valid_keys, bool need_mask,
                                             int lim0, int lim1,
                                             float sscale0, float sscale1,
                                             int lane) {
  using Tr = Traits<kKind>;
  constexpr bool kB = Tr::kMmaBF16;
  constexpr uint32_t P = Tr::kPerm;
  const int r = lane >> 2, c = lane & 3;
  // Q.K^T: two accumulators per 8-key tile (even / odd k-steps) so that four
  // independent MMA chains are in flight
  float s[2][4], s2[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) s[nt][e] = s2[nt][e] = 0.f;
    const int t = nt * 8 + perm_of(P, r);
    if constexpr (!Tr::kFp8) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int dhi = j >> 1;
        const int u = ((j & 1) << 2) | c;
        const int phys = u ^ (((t << 1) | dhi) & 7);
        const uint4 kv = lds128(k_base + t * 256 + dhi * 128 + phys * 16);
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
          const uint32_t b0 = e4m3x2_to_f16x2(wv[tt]);
          const uint32_t b1 = e4m3x2_to_f16x2(wv[tt] >> 16);
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
  // scale, mask
  const int tA = perm_of(P, 2 * c), tB = perm_of(P, 2 * c + 1);
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v = s[nt][e] * (e < 2 ? sscale0 : sscale1);
      if (need_mask) {
        const int key = key0 + nt * 8 + ((e & 1) ? tB : tA);
        if (key > (e < 2 ? lim0 : lim1)) v = -INFINITY;
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
        const int phys = r ^ (((t << 1) | h) & 7);
        v[k] = lds128(v_base + t * 256 + h * 128 + phys * 16);
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
      mma_acc<false, kRows16>(st.o[T], pa, e4m3x2_to_f16x2(ab01),
                              e4m3x2_to_f16x2(cd01));
      mma_acc<false, kRows16>(st.o[T + 1], pa, e4m3x2_to_f16x2(ab01 >> 16),
                              e4m3x2_to_f16x2(cd01 >> 16));
      mma_acc<false, kRows16>(st.o[T + 2], pa, e4m3x2_to_f16x2(ab23),
                              e4m3x2_to_f16x2(cd23));
      mma_acc<false, kRows16>(st.o[T + 3], pa, e4m3x2_to_f16x2(ab23 >> 16),
                              e4m3x2_to_f16x2(cd23 >> 16));
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

constexpr int kItemQueue = 4;  // work items the producer may run ahead

// Shared-memory carve-up of one CTA (offsets from a 1024-aligned base).
template <int kKind, bool kWide>
struct Layout {
  using Tr = Traits<kKind>;
  static constexpr int kE = kWide ? 4 : 2;  // accumulator rows kept per lane
  static constexpr int kRing = 0;
  static constexpr int kScratch = Tr::kRingBytes;                 // partial O
  static constexpr int kScratchBytes = kConsumerWarps * 16 * kE * 32 * 4;
  static constexpr int kML = kScratch + kScratchBytes;            // m, l
  static constexpr int kMLBytes = kConsumerWarps * 16 * 2 * 4;
  static constexpr int kBars = kML + kMLBytes;                    // 8 B each
  static constexpr int kNumBars = 2 * Tr::kStages + 2 * kItemQueue;
  static constexpr int kItems = kBars + 8 * kNumBars;             // int4 each
  static constexpr int kAbort = kItems + 16 * kItemQueue;
  static constexpr int kBytes = kAbort + 16;
  static constexpr int kSmemBytes = 1024 + kBytes;  // + alignment slack
};

struct Smem {
  uint32_t base;          // shared address, 1024-aligned
  uint8_t* ptr;           // generic pointer to the same byte
  int stages;
  __device__ uint32_t full(int s) const { return bars + 8 * s; }
  __device__ uint32_t empty(int s) const { return bars + 8 * (stages + s); }
  __device__ uint32_t item_full(int q) const { return bars + 8 * (2 * stages + q); }
  __device__ uint32_t item_empty(int q) const {
    return bars + 8 * (2 * stages + kItemQueue + q);
  }
  uint32_t bars;
  int4* items;
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

__device__ __forceinline__ ItemGeom item_geom(const FastParams& p, int kind,
                                              int x, const ReqMeta& rm) {
  ItemGeom ig;
  if (kind == kItemDecode) {
    ig.page0 = x * p.blocks_per_split;
    ig.npages = min(p.blocks_per_split, rm.nb - ig.page0);
    ig.row0 = 0;
    ig.rows = rm.n * p.group;
  } else {
    ig.row0 = x * kPrefillTileRows;
    ig.rows = min(kPrefillTileRows, rm.n * p.group - ig.row0);
    const int lim_last = rm.L - rm.n + (ig.row0 + ig.rows - 1) / p.group;
    ig.page0 = 0;
    ig.npages = lim_last / kBS + 1;
  }
  return ig;
}

// One consumer warp's share of one work item.  Pages are numbered by the
// CTA-wide counter c0 + j; in a decode item page c goes to warp c % 4 (the
// same warp for a given ring slot, since the ring depth is a multiple of 4),
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
  int my_min = INT_MAX;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int rr = rq + 8 * half;
    lim[half] = rm.L - 1;
    if (rr < wrows) {
      lim[half] = rm.L - rm.n + (wrow0 + rr) / G;
      my_min = min(my_min, lim[half]);
    }
  }
#pragma unroll
  for (int d = 1; d < 32; d <<= 1)
    my_min = min(my_min, __shfl_xor_sync(~0u, my_min, d));
  const int min_lim = min(my_min, rm.L - 1);
  const float ss0 = p.score_scale * rscale[0];
  const float ss1 = p.score_scale * rscale[1];

  WarpState st;
#pragma unroll
  for (int T = 0; T < 16; ++T)
    st.o[T][0] = st.o[T][1] = st.o[T][2] = st.o[T][3] = 0.f;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.f;

  const int first = decode ? (int)((warp - (int)(c0 & 3u)) & 3) : 0;
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
    const bool need_mask = key0 + kBS - 1 > min_lim;
    const uint32_t kb = sm.base + Ly::kRing + slot * Tr::kStageBytes;
    process_page<kKind, kRows16>(kb, kb + Tr::kPageBytes, qa, st, key0, valid,
                                 need_mask, lim[0], lim[1], ss0, ss1, lane);
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
  const int nsplit = __ldg(p.req_nsplit + r);
#pragma unroll
  for (int Tq = 0; Tq < 4; ++Tq) {
    const int T = warp * 4 + Tq;
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
      if (nsplit <= 1) {
        store_out<OutT<kKind>>(p.out, row * 128 + col, num / den * p.out_scale);
      } else {
        const int64_t slotp = row * p.max_splits + x;
        p.ws_acc[slotp * 128 + col] = num;
        if (T == 0 && (e & 1) == 0 && c == 0) {
          p.ws_ml[slotp * 2 + 0] = M;
          p.ws_ml[slotp * 2 + 1] = den;
        }
      }
    }
  }
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
__global__ void __launch_bounds__(kThreads, 2)
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
  sm.items = reinterpret_cast<int4*>(sm.ptr + Ly::kItems);
  sm.abort_flag = reinterpret_cast<volatile int*>(sm.ptr + Ly::kAbort);
  sm.scratch = reinterpret_cast<float*>(sm.ptr + Ly::kScratch);
  sm.ml = reinterpret_cast<float*>(sm.ptr + Ly::kML);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(sm.full(i), 1);
      mbar_init(sm.empty(i), kConsumerWarps);
    }
    for (int q = 0; q < kItemQueue; ++q) {
      mbar_init(sm.item_full(q), 1);
      mbar_init(sm.item_empty(q), kConsumerWarps);
    }
    *sm.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int num_items = __ldg(p.num_items);

  if (warp == kConsumerWarps) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
    }
    uint32_t c = 0;     // pages issued
    for (int k = 0;; ++k) {
      const int q = k % kItemQueue;
      int4 it = make_int4(-1, 0, 0, 0);
      if (lane == 0) {
        bool ok = k < kItemQueue ||
                  mbar_wait_bounded(sm.item_empty(q), ((k / kItemQueue) - 1) & 1);
        if (!ok) {
          flag_error(p.err, PA_DEV_ERR_TIMEOUT);
          *sm.abort_flag = 1;
        }
        if (ok && *sm.abort_flag == 0) {
          const int idx = atomicAdd(p.work_counter, 1);
          if (idx < num_items) it = __ldg(p.items + idx);
        }
        if (ok) {
          sm.items[q] = it;
          mbar_arrive(sm.item_full(q));
        }
      }
      it.x = __shfl_sync(~0u, it.x, 0);
      it.y = __shfl_sync(~0u, it.y, 0);
      it.z = __shfl_sync(~0u, it.z, 0);
      it.w = __shfl_sync(~0u, it.w, 0);
      if (it.x < 0) break;
      const ReqMeta rm = load_req(p.qsl, p.seq_lens, it.x, p.num_tokens,
                                  p.max_query_len, p.max_seq_len,
                                  p.max_blocks_per_seq);
      const ItemGeom ig = item_geom(p, it.z, it.w, rm);
      if (!kWide && (it.z == kItemPrefill || ig.rows > 8)) continue;
      const int32_t* bt =
          p.block_tables + (int64_t)it.x * p.max_blocks_per_seq + ig.page0;
      // block ids of this item, 32 per register, loaded two chunks ahead
      const int n = ig.npages;
      int ids0 = lane < n ? __ldg(bt + lane) : 0;
      int ids1 = 32 + lane < n ? __ldg(bt + 32 + lane) : 0;
      int ids2 = 64 + lane < n ? __ldg(bt + 64 + lane) : 0;
      constexpr int PF = PA_L2_PREFETCH_PAGES;
      static_assert(PF >= 0 && PF <= 32, "prefetch window must fit one id chunk");
      auto page_row = [&](int blk) {
        if (blk < 0 || (int64_t)blk >= p.num_blocks) {
          flag_error(p.err, PA_DEV_ERR_BLOCK_ID);
          blk = 0;
        }
        return (blk * p.num_kv_heads + it.y) * kBS;
      };
      auto prefetch = [&](int row) {
        if constexpr (Tr::kFp8) {
          tma_prefetch_2d(&tmap_k, 0, row);
          tma_prefetch_2d(&tmap_v, 0, row);
        } else {
          tma_prefetch_3d(&tmap_k, 0, 0, row);
          tma_prefetch_3d(&tmap_v, 0, 0, row);
        }
      };
      // the first window goes to L2 at once
      if (PF > 0 && lane < min(PF, n)) prefetch(page_row(ids0));
      int go = 1;
      for (int j = 0; j < n && go; ++j, ++c) {
        if (j > 0 && (j & 31) == 0) {
          ids0 = ids1;
          ids1 = ids2;
          const int idx = j + 64 + lane;
          ids2 = idx < n ? __ldg(bt + idx) : 0;
        }
        int blk = __shfl_sync(~0u, ids0, j & 31);
        const int jp = j + PF;
        const int blk_pf = __shfl_sync(~0u, (jp >> 5) == (j >> 5) ? ids0 : ids1,
                                       jp & 31);
        if (lane == 0) {
          if (PF > 0 && jp < n) prefetch(page_row(blk_pf));
          const int slot = c % S;
          if (c >= (uint32_t)S &&
              !mbar_wait_bounded(sm.empty(slot), ((c / S) - 1) & 1)) {
            flag_error(p.err, PA_DEV_ERR_TIMEOUT);
            *sm.abort_flag = 1;
          }
          if (*sm.abort_flag) {
            go = 0;
          } else {
            const int row = page_row(blk);
            const uint32_t dst = sm.base + Ly::kRing + slot * Tr::kStageBytes;
            mbar_arrive_expect_tx(sm.full(slot), Tr::kStageBytes);
            if constexpr (Tr::kFp8) {
              tma_load_2d(dst, &tmap_k, sm.full(slot), 0, row);
              tma_load_2d(dst + Tr::kPageBytes, &tmap_v, sm.full(slot), 0, row);
            } else {
              tma_load_3d(dst, &tmap_k, sm.full(slot), 0, 0, row);
              tma_load_3d(dst + Tr::kPageBytes, &tmap_v, sm.full(slot), 0, 0, row);
            }
          }
        }
        go = __shfl_sync(~0u, go, 0);
      }
      if (!go) {
        // stop claiming; hand the consumers an end marker if a queue slot
        // frees up, then let the copies already in flight land
        if (lane == 0) {
          const int q2 = (k + 1) % kItemQueue;
          if (k + 1 < kItemQueue ||
              mbar_wait_bounded(sm.item_empty(q2), (((k + 1) / kItemQueue) - 1) & 1)) {
            sm.items[q2] = make_int4(-1, 0, 0, 0);
            mbar_arrive(sm.item_full(q2));
          }
          const uint32_t from = c > (uint32_t)S ? c - S : 0;
          for (uint32_t i = from; i < c; ++i)
            mbar_wait_bounded(sm.full(i % S), (i / S) & 1);
        }
        break;
      }
    }
    return;
  }

  // ------------------------------ consumers -------------------------------
  uint32_t c = 0;  // pages consumed (CTA-wide numbering, as issued)
  for (int k = 0;; ++k) {
    const int q = k % kItemQueue;
    const bool got =
        __all_sync(~0u, mbar_wait_bounded(sm.item_full(q), (k / kItemQueue) & 1));
    int4 it = make_int4(-1, 0, 0, 0);
    if (got) {
      it = sm.items[q];
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.item_empty(q));
    } else if (lane == 0) {
      flag_error(p.err, PA_DEV_ERR_TIMEOUT);
      *sm.abort_flag = 1;
    }
    // every consumer warp meets here once per item: decisions below are
    // uniform, the previous item's shared scratch is no longer read, and all
    // earlier pages have been consumed by their owners
    if (consumers_sync_any(it.x < 0 || *sm.abort_flag != 0)) break;
    const ReqMeta rm = load_req(p.qsl, p.seq_lens, it.x, p.num_tokens,
                                p.max_query_len, p.max_seq_len,
                                p.max_blocks_per_seq);
    const ItemGeom ig = item_geom(p, it.z, it.w, rm);
    if constexpr (kWide) {
      if (it.z == kItemPrefill || ig.rows > 8)
        consume_item<kKind, true, true>(p, sm, rm, it.x, it.y, it.z, it.w, ig,
                                        c, warp, lane);
      else
        consume_item<kKind, false, true>(p, sm, rm, it.x, it.y, it.z, it.w, ig,
                                         c, warp, lane);
    } else {
      if (it.z == kItemPrefill || ig.rows > 8) {
        // the host never sends such an item to the narrow kernel
        if (threadIdx.x == 0) flag_error(p.err, PA_DEV_ERR_METADATA);
        continue;
      }
      consume_item<kKind, false, false>(p, sm, rm, it.x, it.y, it.z, it.w, ig,
                                        c, warp, lane);
    }
    c += ig.npages;
  }
}

// ---------------------------------------------------------------------------
// split-K merge: one warp per (token, q head) row of a split decode request
// ---------------------------------------------------------------------------
template <typename TOut>
__global__ void __launch_bounds__(128)
merge_kernel(FastParams p) {
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.num_tokens * p.num_q_heads) return;
  const int64_t t = row / p.num_q_heads;
  // request owning token t: last r with qsl[r] <= t
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.qsl + mid) <= t) lo = mid; else hi = mid - 1;
  }
  const int r = lo;
  const ReqMeta rm = load_req(p.qsl, p.seq_lens, r, p.num_tokens, p.max_query_len,
                              p.max_seq_len, p.max_blocks_per_seq);
  if (!rm.ok || t < rm.q0 || t >= rm.q0 + rm.n) return;
  if (rm.n * p.group > kDecodeMaxRows) return;
  const int ns = __ldg(p.req_nsplit + r);
  if (ns <= 1) return;
  const float* ml = p.ws_ml + row * p.max_splits * 2;
  float M = -INFINITY;
  for (int s = lane; s < ns; s += 32) M = fmaxf(M, ml[2 * s]);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) M = fmaxf(M, __shfl_xor_sync(~0u, M, d));
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float den = 0.f;
  const float* a = p.ws_acc + row * p.max_splits * 128;
  for (int s = 0; s < ns; ++s) {
    const float ms = ml[2 * s];
    const float w = ms == -INFINITY ? 0.f : exp2f(ms - M);
    den += w * ml[2 * s + 1];
    const float4 v = *reinterpret_cast<const float4*>(a + s * 128 + 4 * lane);
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
cudaError_t launch_kind(const FastParams& fp, const AttnPlan& plan,
                        const CUtensorMap& tk, const CUtensorMap& tv,
                        int4* items, int* count, int* nsplit,
                        cudaStream_t stream) {
  using Tr = Traits<kKind>;
  (void)Tr::kStages;
  // the narrow kernel covers steps whose every item has <= 8 rows
  const bool wide = (int64_t)fp.max_query_len * fp.group > 8;
  int grid = 0;
  cudaError_t e = wide ? prepare_kernel<kKind, true>(&grid)
                       : prepare_kernel<kKind, false>(&grid);
  if (e != cudaSuccess) return e;
  if ((int64_t)grid > plan.max_items) grid = (int)plan.max_items;
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(fp, items, count, nsplit);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const ProfileEvents& pe = profile_events();
  if (pe.start) cudaEventRecord(pe.start, stream);
  if (wide)
    attn_fast_kernel<kKind, true>
        <<<grid, kThreads, Layout<kKind, true>::kSmemBytes, stream>>>(tk, tv, fp);
  else
    attn_fast_kernel<kKind, false>
        <<<grid, kThreads, Layout<kKind, false>::kSmemBytes, stream>>>(tk, tv, fp);
  e = cudaGetLastError();
  if (pe.stop) cudaEventRecord(pe.stop, stream);
  if (e != cudaSuccess) return e;
  if (plan.max_splits > 1) {
    const int64_t rows = fp.num_tokens * fp.num_q_heads;
    const unsigned mgrid = (unsigned)((rows + 3) / 4);
    merge_kernel<OutT<kKind>><<<mgrid, 128, 0, stream>>>(fp);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

bool fast_path_supported(const AttnArgs& a) {
  if (a.head_dim != 128) return false;
  if (a.num_q_heads / a.num_kv_heads > kDecodeMaxRows && false) return false;
  if (a.cache_dtype == PA_BF16 && a.q_dtype == PA_BF16) return true;
  if (a.cache_dtype == PA_F16 && a.q_dtype == PA_F16) return true;
  if (a.cache_dtype == PA_FP8_E4M3 && (a.q_dtype == PA_BF16 || a.q_dtype == PA_F16))
    return true;
  return false;
}

AttnPlan make_plan(int64_t num_tokens, int num_q_heads, int num_kv_heads,
                   int head_dim, int num_seqs, int max_query_len,
                   int max_seq_len, int num_sms) {
  AttnPlan pl{};
  pl.group = num_q_heads / num_kv_heads;
  const int64_t mb = ((int64_t)max_seq_len + kBS - 1) / kBS;
  // Split size: aim for several waves of CTAs (two resident per SM) so that
  // the tail of the step is short, but keep every split long enough to hide
  // its pipeline start-up and bound the number of partial results.
  const int64_t target = (int64_t)num_sms * PA_SPLIT_WAVES;
  const int64_t units = (int64_t)num_seqs * num_kv_heads;
  int64_t bps = mb;
  if (units > 0) {
    const int64_t want_splits = (target + units - 1) / units;
    bps = (mb + want_splits - 1) / want_splits;
  }
  if (bps < PA_SPLIT_MIN_BLOCKS) bps = PA_SPLIT_MIN_BLOCKS;
  if (bps > mb) bps = mb;
  if (bps < 1) bps = 1;
  int64_t ms = (mb + bps - 1) / bps;
  if (ms > 64) {  // bound the partial-result storage
    bps = (mb + 63) / 64;
    ms = (mb + bps - 1) / bps;
  }
  pl.blocks_per_split = (int)bps;
  pl.max_splits = (int)(ms < 1 ? 1 : ms);
  pl.has_prefill = (int64_t)max_query_len * pl.group > kDecodeMaxRows;
  int64_t items = 0;
  if (pl.group <= kDecodeMaxRows)
    items += (int64_t)num_seqs * num_kv_heads * pl.max_splits;
  if (pl.has_prefill)
    items += (int64_t)num_kv_heads *
             ((num_tokens * pl.group + kPrefillTileRows - 1) / kPrefillTileRows +
              num_seqs);
  pl.max_items = items;
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  size_t off = 0;
  pl.off_items = off;
  off = up(off + (size_t)items * 16);
  pl.off_count = off;
  off = up(off + 16);
  pl.off_nsplit = off;
  off = up(off + (size_t)num_seqs * 4);
  pl.off_acc = off;
  const size_t rows = (size_t)num_tokens * num_q_heads;
  if (pl.max_splits > 1) off = up(off + rows * pl.max_splits * head_dim * 4);
  pl.off_ml = off;
  if (pl.max_splits > 1) off = up(off + rows * pl.max_splits * 2 * 4);
  pl.total_bytes = off;
  return pl;
}

cudaError_t launch_attention_fast(const AttnArgs& a, const AttnPlan& plan,
                                  const CUtensorMap& tmap_k,
                                  const CUtensorMap& tmap_v,
                                  cudaStream_t stream) {
  if (plan.max_items == 0) return cudaSuccess;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  FastParams fp{};
  fp.q = a.q;
  fp.out = a.out;
  fp.block_tables = a.block_tables;
  fp.seq_lens = a.seq_lens;
  fp.qsl = a.query_start_loc;
  fp.items = reinterpret_cast<const int4*>(ws + plan.off_items);
  fp.num_items = reinterpret_cast<const int*>(ws + plan.off_count);
  fp.work_counter = reinterpret_cast<int*>(ws + plan.off_count + 4);
  fp.req_nsplit = reinterpret_cast<const int*>(ws + plan.off_nsplit);
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
  fp.blocks_per_split = plan.blocks_per_split;
  fp.max_splits = plan.max_splits;
  fp.max_items = plan.max_items;
  const bool fp8 = a.cache_dtype == PA_FP8_E4M3;
  fp.score_scale = a.scale * 1.4426950408889634f * (fp8 ? a.k_scale : 1.0f);
  fp.out_scale = fp8 ? a.v_scale : 1.0f;
  int4* items = reinterpret_cast<int4*>(ws + plan.off_items);
  int* count = reinterpret_cast<int*>(ws + plan.off_count);
  int* nsplit = reinterpret_cast<int*>(ws + plan.off_nsplit);
  if (a.cache_dtype == PA_BF16)
    return launch_kind<kKindBF16>(fp, plan, tmap_k, tmap_v, items, count, nsplit, stream);
  if (a.cache_dtype == PA_F16)
    return launch_kind<kKindF16>(fp, plan, tmap_k, tmap_v, items, count, nsplit, stream);
  if (a.q_dtype == PA_BF16)
    return launch_kind<kKindFp8BF16>(fp, plan, tmap_k, tmap_v, items, count, nsplit, stream);
  return launch_kind<kKindFp8F16>(fp, plan, tmap_k, tmap_v, items, count, nsplit, stream);
}

}  // namespace pa

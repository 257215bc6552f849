// attn_generic.cu -- paged attention for the shapes the tensor-core kernel
// does not take (fp32 caches, head_dim 64): one warp per (token, query head),
// keys visited in logical order with an fp32 online softmax.
//
// Same definition as the fast path ("vLLM engine anatomy": paging through the
// block table, Figure 2; GQA, Table 1; exact softmax attention computed
// online, "Boundaries: FlashAttention ..."): query i of request r sees keys
// 0 .. L - n + i (with a sliding window of W keys only L - n + i - W + 1 ..
// L - n + i), query head h reads KV head h / group.
#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

struct GenericParams {
  const void* q;
  void* out;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;
  unsigned* err;
  int64_t num_tokens;
  int64_t num_blocks;
  int max_blocks_per_seq, num_seqs;
  int num_q_heads, num_kv_heads, group;
  int max_query_len, max_seq_len;
  float scale, k_scale, v_scale;
  int window;  // sliding window in keys (kNoWindow: none)
};

// Element d of the token at offset o of the page of (blk, g); the 4-bit
// formats decode from their pages (pa.h), without the per-tensor scale.
struct Int4Page {};
struct Nvfp4Page {};

template <typename TC, int kD>
__device__ __forceinline__ float load_cache(const void* base, int64_t page,
                                            int o, int d) {
  if constexpr (std::is_same<TC, uint8_t>::value) {
    return e4m3_to_f32(static_cast<const uint8_t*>(base)[(page * kBS + o) * kD + d]);
  } else if constexpr (std::is_same<TC, Int4Page>::value) {
    const uint8_t* pg = static_cast<const uint8_t*>(base) + page * (8 * kD + 64);
    const uint32_t byte = pg[o * (kD / 2) + d / 2];
    const int nib = (int)((d & 1) ? (byte >> 4) : (byte & 15u));
    const float sc = *reinterpret_cast<const float*>(pg + kBS * (kD / 2) + 4 * o);
    return sc * (float)(nib >= 8 ? nib - 16 : nib);
  } else if constexpr (std::is_same<TC, Nvfp4Page>::value) {
    const uint8_t* pg = static_cast<const uint8_t*>(base) + page * (9 * kD);
    const uint32_t byte = pg[o * (kD / 2) + d / 2];
    const uint32_t nib = (d & 1) ? (byte >> 4) : (byte & 15u);
    return e4m3_to_f32(pg[kBS * (kD / 2) + o * (kD / 16) + d / 16]) * e2m1_to_f32(nib);
  } else {
    return to_f32(static_cast<const TC*>(base)[(page * kBS + o) * kD + d]);
  }
}

template <typename TQ, typename TC, int kD>
__global__ void __launch_bounds__(128)
attn_generic_kernel(GenericParams p) {
  constexpr int kPer = kD / 32;
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.num_tokens * p.num_q_heads) return;
  const int64_t t = row / p.num_q_heads;
  const int h = (int)(row - t * p.num_q_heads);
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.qsl + mid) <= t) lo = mid; else hi = mid - 1;
  }
  const int r = lo;
  const ReqMeta rm = load_req(p.qsl, p.seq_lens, r, p.num_tokens,
                              p.max_query_len, p.max_seq_len,
                              p.max_blocks_per_seq);
  if (t < rm.q0 || t >= rm.q0 + rm.n) return;  // token of no request
  if (!rm.ok) {
    if (lane == 0) flag_error(p.err, PA_DEV_ERR_METADATA);
    return;
  }
  const int i = (int)(t - rm.q0);
  const int lim = rm.L - rm.n + i;
  const int first = max(0, lim - p.window + 1);  // keys first .. lim
  const int g = h / p.group;
  const TQ* qp = static_cast<const TQ*>(p.q) + row * kD;
  float qv[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) qv[k] = to_f32(qp[lane + 32 * k]) * p.scale * p.k_scale;
  float m = -INFINITY, l = 0.f, acc[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
  const int32_t* bt = p.block_tables + (int64_t)r * p.max_blocks_per_seq;
  for (int j = first; j <= lim; ++j) {
    int blk = __ldg(bt + j / kBS);
    if (blk < 0 || (int64_t)blk >= p.num_blocks) {
      if (lane == 0) flag_error(p.err, PA_DEV_ERR_BLOCK_ID);
      blk = 0;
    }
    const int64_t page = (int64_t)blk * p.num_kv_heads + g;
    const int o = j % kBS;
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      dot += qv[k] * load_cache<TC, kD>(p.k_cache, page, o, lane + 32 * k);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) dot += __shfl_xor_sync(~0u, dot, d);
    const float mnew = fmaxf(m, dot);
    const float alpha = expf(m - mnew);
    const float pj = expf(dot - mnew);
    l = l * alpha + pj;
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      acc[k] = acc[k] * alpha + pj * load_cache<TC, kD>(p.v_cache, page, o, lane + 32 * k);
    m = mnew;
  }
  TQ* op = static_cast<TQ*>(p.out) + row * kD;
  const float inv = p.v_scale / l;
#pragma unroll
  for (int k = 0; k < kPer; ++k) op[lane + 32 * k] = from_f32<TQ>(acc[k] * inv);
}

template <typename TQ, typename TC>
cudaError_t launch_t(const GenericParams& gp, int head_dim, cudaStream_t stream) {
  const int64_t rows = gp.num_tokens * gp.num_q_heads;
  const unsigned grid = (unsigned)((rows + 3) / 4);
  if (head_dim == 128)
    attn_generic_kernel<TQ, TC, 128><<<grid, 128, 0, stream>>>(gp);
  else
    attn_generic_kernel<TQ, TC, 64><<<grid, 128, 0, stream>>>(gp);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace

cudaError_t launch_attention_generic(const AttnArgs& a, cudaStream_t stream) {
  GenericParams gp{};
  gp.q = a.q;
  gp.out = a.out;
  gp.k_cache = a.k_cache;
  gp.v_cache = a.v_cache;
  gp.block_tables = a.block_tables;
  gp.seq_lens = a.seq_lens;
  gp.qsl = a.query_start_loc;
  gp.err = a.err;
  gp.num_tokens = a.num_tokens;
  gp.num_blocks = a.num_blocks;
  gp.max_blocks_per_seq = a.max_blocks_per_seq;
  gp.num_seqs = a.num_seqs;
  gp.num_q_heads = a.num_q_heads;
  gp.num_kv_heads = a.num_kv_heads;
  gp.group = a.num_q_heads / a.num_kv_heads;
  gp.max_query_len = a.max_query_len;
  gp.max_seq_len = a.max_seq_len;
  const bool fp8 = a.cache_dtype == PA_FP8_E4M3 || a.cache_dtype == PA_NVFP4;
  gp.scale = a.scale;
  gp.k_scale = fp8 ? a.k_scale : 1.0f;
  gp.v_scale = fp8 ? a.v_scale : 1.0f;
  gp.window = a.window > 0 ? a.window : kNoWindow;
  switch (a.cache_dtype) {
    case PA_F32:
      return launch_t<float, float>(gp, a.head_dim, stream);
    case PA_F16:
      return launch_t<__half, __half>(gp, a.head_dim, stream);
    case PA_BF16:
      return launch_t<__nv_bfloat16, __nv_bfloat16>(gp, a.head_dim, stream);
    case PA_FP8_E4M3:
      if (a.q_dtype == PA_BF16)
        return launch_t<__nv_bfloat16, uint8_t>(gp, a.head_dim, stream);
      return launch_t<__half, uint8_t>(gp, a.head_dim, stream);
    case PA_INT4:
      if (a.q_dtype == PA_BF16)
        return launch_t<__nv_bfloat16, Int4Page>(gp, a.head_dim, stream);
      return launch_t<__half, Int4Page>(gp, a.head_dim, stream);
    case PA_NVFP4:
      if (a.q_dtype == PA_BF16)
        return launch_t<__nv_bfloat16, Nvfp4Page>(gp, a.head_dim, stream);
      return launch_t<__half, Nvfp4Page>(gp, a.head_dim, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa

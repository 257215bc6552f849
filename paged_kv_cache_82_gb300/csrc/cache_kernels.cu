// cache_kernels.cu -- writes into the paged KV cache.
//
//  * reshape_and_cache: every token processed in a step has its K and V
//    written into its slot (block = slot / 16, offset = slot % 16), as
//    "vLLM engine anatomy" describes under "Prefill, decode ..." and in
//    Figure 2; an FP8 cache ("01. vLLM", --kv-cache-dtype fp8) stores the
//    E4M3 code nearest to fl32(x / scale); the 4-bit caches of the same
//    table (nvfp4, int4_per_token_head) quantise each (token, KV head).
//  * copy_blocks: block-granular copy-on-write of shared blocks ("vLLM
//    engine anatomy", PagedAttention section; V0's blocks_to_copy in "vLLM
//    V0 vs V1").
//
// Both are HBM-bound streaming copies: 16-byte vector loads/stores, one
// thread per 8-element chunk of a (token, head) row.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kThreads = 256;

template <typename Tin, int kN>
struct alignas(sizeof(Tin) * kN) Vec {
  Tin v[kN];
};

// One thread = 8 consecutive elements of one (token, head) row of K or V.
template <typename Tin, bool kFp8>
__global__ void __launch_bounds__(kThreads)
reshape_vec_kernel(const Tin* __restrict__ key, const Tin* __restrict__ value,
                   int64_t num_tokens, int64_t key_stride, int64_t value_stride,
                   void* __restrict__ k_cache, void* __restrict__ v_cache,
                   int64_t num_slots, int num_kv_heads, int head_dim,
                   const int64_t* __restrict__ slot_mapping, float k_scale,
                   float v_scale, unsigned* err) {
  const int chunks = head_dim >> 3;
  const int64_t per_token = 2ll * num_kv_heads * chunks;
  const int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (id >= num_tokens * per_token) return;
  const int64_t t = id / per_token;
  const int rem = (int)(id - t * per_token);
  const int which = rem / (num_kv_heads * chunks);  // 0 = K, 1 = V
  const int rem2 = rem - which * num_kv_heads * chunks;
  const int h = rem2 / chunks;
  const int c = rem2 - h * chunks;
  // the row does not depend on the slot: both loads go out together
  const Tin* src = (which ? value + t * value_stride : key + t * key_stride) +
                   (int64_t)h * head_dim + c * 8;
  const Vec<Tin, 8> in = *reinterpret_cast<const Vec<Tin, 8>*>(src);
  const int64_t slot = __ldg(slot_mapping + t);
  if (slot < 0) return;  // padding token
  if (slot >= num_slots) {
    if (rem == 0) flag_error(err, PA_DEV_ERR_SLOT);
    return;
  }
  const int64_t b = slot / kBS, o = slot - (slot / kBS) * kBS;
  const int64_t dst = ((b * num_kv_heads + h) * kBS + o) * head_dim + c * 8;
  if constexpr (!kFp8) {
    Tin* cache = static_cast<Tin*>(which ? v_cache : k_cache);
    *reinterpret_cast<Vec<Tin, 8>*>(cache + dst) = in;
  } else {
    const float scale = which ? v_scale : k_scale;
    uint8_t* cache = static_cast<uint8_t*>(which ? v_cache : k_cache);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float y = __fdiv_rn(to_f32(in.v[e]), scale);
      const uint32_t code =
          __nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3);
      if (e < 4)
        lo |= code << (8 * e);
      else
        hi |= code << (8 * (e - 4));
    }
    *reinterpret_cast<uint2*>(cache + dst) = make_uint2(lo, hi);
  }
}

// One thread = one element (any alignment / stride).
template <typename Tin, bool kFp8>
__global__ void __launch_bounds__(kThreads)
reshape_scalar_kernel(const Tin* __restrict__ key, const Tin* __restrict__ value,
                      int64_t num_tokens, int64_t key_stride,
                      int64_t value_stride, void* __restrict__ k_cache,
                      void* __restrict__ v_cache, int64_t num_slots,
                      int num_kv_heads, int head_dim,
                      const int64_t* __restrict__ slot_mapping, float k_scale,
                      float v_scale, unsigned* err) {
  const int64_t per_token = 2ll * num_kv_heads * head_dim;
  const int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (id >= num_tokens * per_token) return;
  const int64_t t = id / per_token;
  const int rem = (int)(id - t * per_token);
  const int which = rem / (num_kv_heads * head_dim);
  const int rem2 = rem - which * num_kv_heads * head_dim;
  const int h = rem2 / head_dim;
  const int d = rem2 - h * head_dim;
  const int64_t slot = __ldg(slot_mapping + t);
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (rem == 0) flag_error(err, PA_DEV_ERR_SLOT);
    return;
  }
  const int64_t b = slot / kBS, o = slot - (slot / kBS) * kBS;
  const Tin x = (which ? value + t * value_stride : key + t * key_stride)
      [(int64_t)h * head_dim + d];
  const int64_t dst = ((b * num_kv_heads + h) * kBS + o) * head_dim + d;
  if constexpr (!kFp8) {
    static_cast<Tin*>(which ? v_cache : k_cache)[dst] = x;
  } else {
    const float y = __fdiv_rn(to_f32(x), which ? v_scale : k_scale);
    static_cast<uint8_t*>(which ? v_cache : k_cache)[dst] =
        static_cast<uint8_t>(__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3));
  }
}

template <typename Tin, bool kFp8>
cudaError_t launch_reshape_t(const void* key, const void* value,
                             int64_t num_tokens, int64_t key_stride,
                             int64_t value_stride, void* k_cache,
                             void* v_cache, int64_t num_blocks,
                             int num_kv_heads, int head_dim,
                             const int64_t* slot_mapping, float k_scale,
                             float v_scale, bool vector_ok, unsigned* err,
                             cudaStream_t stream) {
  const int64_t per_token =
      2ll * num_kv_heads * (vector_ok ? head_dim / 8 : head_dim);
  const int64_t threads = num_tokens * per_token;
  const int64_t blocks = (threads + kThreads - 1) / kThreads;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  if (vector_ok) {
    reshape_vec_kernel<Tin, kFp8><<<(unsigned)blocks, kThreads, 0, stream>>>(
        static_cast<const Tin*>(key), static_cast<const Tin*>(value),
        num_tokens, key_stride, value_stride, k_cache, v_cache,
        num_blocks * kBS, num_kv_heads, head_dim, slot_mapping, k_scale,
        v_scale, err);
  } else {
    reshape_scalar_kernel<Tin, kFp8><<<(unsigned)blocks, kThreads, 0, stream>>>(
        static_cast<const Tin*>(key), static_cast<const Tin*>(value),
        num_tokens, key_stride, value_stride, k_cache, v_cache,
        num_blocks * kBS, num_kv_heads, head_dim, slot_mapping, k_scale,
        v_scale, err);
  }
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

// 4-bit caches: one warp per (token, KV head, K or V).  Lane l holds the
// kE = head_dim / 32 consecutive elements l*kE ..; a 16-element NVFP4 block
// is the 16 / kE lanes of one aligned group.  Quantisation follows the
// page format of pa.h: INT4, s = fl32(max|x| / 7), code = nearest integer
// to fl32(x / s) in [-7, 7]; NVFP4 per block, b = E4M3(fl32(fl32(max|x| / 6)
// / scale)), r = fl32(e4m3(b) * scale), code = E2M1(fl32(x / r)).
template <typename Tin, bool kNvfp4, int kD>
__global__ void __launch_bounds__(kThreads)
reshape_4bit_kernel(const Tin* __restrict__ key, const Tin* __restrict__ value,
                    int64_t num_tokens, int64_t key_stride,
                    int64_t value_stride, uint8_t* __restrict__ k_cache,
                    uint8_t* __restrict__ v_cache, int64_t num_slots,
                    int num_kv_heads, const int64_t* __restrict__ slot_mapping,
                    float k_scale, float v_scale, unsigned* err) {
  constexpr int kE = kD / 32;
  constexpr int kPage = kNvfp4 ? 9 * kD : 8 * kD + 64;
  const int lane = threadIdx.x & 31;
  const int64_t w = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  if (w >= num_tokens * 2 * num_kv_heads) return;
  const int64_t t = w / (2 * num_kv_heads);
  const int rem = (int)(w - t * 2 * num_kv_heads);
  const int which = rem / num_kv_heads, h = rem - which * num_kv_heads;
  const int64_t slot = __ldg(slot_mapping + t);
  if (slot < 0) return;  // padding token
  if (slot >= num_slots) {
    if (rem == 0 && lane == 0) flag_error(err, PA_DEV_ERR_SLOT);
    return;
  }
  const Tin* src = (which ? value + t * value_stride : key + t * key_stride) +
                   (int64_t)h * kD + lane * kE;
  float x[kE];
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < kE; ++e) {
    x[e] = to_f32(src[e]);
    amax = fmaxf(amax, fabsf(x[e]));
  }
  const int64_t b = slot / kBS;
  const int o = (int)(slot - b * kBS);
  uint8_t* page = (which ? v_cache : k_cache) + (b * num_kv_heads + h) * kPage;
  uint32_t code[kE];
  if constexpr (!kNvfp4) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, d));
    const float sc = amax > 0.f ? __fdiv_rn(amax, 7.0f) : 0.f;
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      int c = sc > 0.f ? __float2int_rn(__fdiv_rn(x[e], sc)) : 0;
      c = max(-7, min(7, c));
      code[e] = (uint32_t)c & 0xFu;
    }
    if (lane == 0)
      *reinterpret_cast<float*>(page + kBS * (kD / 2) + 4 * o) = sc;
  } else {
    constexpr int kLanes = 16 / kE;  // lanes of one 16-element block
#pragma unroll
    for (int d = 1; d < kLanes; d <<= 1) amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, d));
    const float g = which ? v_scale : k_scale;
    const float u = __fdiv_rn(__fdiv_rn(amax, 6.0f), g);
    const uint8_t bs =
        static_cast<uint8_t>(__nv_cvt_float_to_fp8(u, __NV_SATFINITE, __NV_E4M3));
    const float r = __fmul_rn(e4m3_to_f32(bs), g);
#pragma unroll
    for (int e = 0; e < kE; ++e) code[e] = r > 0.f ? e2m1_encode(__fdiv_rn(x[e], r)) : 0u;
    if (lane % kLanes == 0)
      page[kBS * (kD / 2) + o * (kD / 16) + (lane * kE) / 16] = bs;
  }
  // kE / 2 bytes of codes: element 2i in the low nibble of byte i
  uint8_t* dst = page + o * (kD / 2) + lane * (kE / 2);
#pragma unroll
  for (int i = 0; i < kE / 2; ++i)
    dst[i] = static_cast<uint8_t>(code[2 * i] | (code[2 * i + 1] << 4));
}

// Copy whole blocks: blockIdx.y walks the pairs, x-threads stripe the
// block's bytes in 16-byte units (K and V).
__global__ void __launch_bounds__(kThreads)
copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                   int64_t num_blocks, int64_t block_vecs,
                   const int64_t* __restrict__ block_mapping, int64_t num_pairs,
                   unsigned* err) {
  for (int64_t p = blockIdx.y; p < num_pairs; p += gridDim.y) {
    const int64_t src = __ldg(block_mapping + 2 * p);
    const int64_t dst = __ldg(block_mapping + 2 * p + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (blockIdx.x == 0 && threadIdx.x == 0)
        flag_error(err, PA_DEV_ERR_BLOCK_ID);
      continue;
    }
    const uint4* ks = k_cache + src * block_vecs;
    const uint4* vs = v_cache + src * block_vecs;
    uint4* kd = k_cache + dst * block_vecs;
    uint4* vd = v_cache + dst * block_vecs;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
         i < block_vecs; i += (int64_t)gridDim.x * blockDim.x) {
      const uint4 a = ks[i];
      const uint4 b = vs[i];
      kd[i] = a;
      vd[i] = b;
    }
  }
}

}  // namespace

cudaError_t launch_reshape_and_cache(const void* key, const void* value,
                                     pa_dtype kv_dtype, int64_t num_tokens,
                                     int64_t key_stride, int64_t value_stride,
                                     void* k_cache, void* v_cache,
                                     pa_dtype cache_dtype, int64_t num_blocks,
                                     int num_kv_heads, int head_dim,
                                     const int64_t* slot_mapping, float k_scale,
                                     float v_scale, bool vector_ok,
                                     unsigned* err, cudaStream_t stream) {
  const bool fp8 = cache_dtype == PA_FP8_E4M3;
#define PA_RESHAPE(T, F)                                                     \
  return launch_reshape_t<T, F>(key, value, num_tokens, key_stride,         \
                                value_stride, k_cache, v_cache, num_blocks, \
                                num_kv_heads, head_dim, slot_mapping,       \
                                k_scale, v_scale, vector_ok, err, stream)
  switch (kv_dtype) {
    case PA_F32:
      if (fp8) PA_RESHAPE(float, true);
      PA_RESHAPE(float, false);
    case PA_F16:
      if (fp8) PA_RESHAPE(__half, true);
      PA_RESHAPE(__half, false);
    case PA_BF16:
      if (fp8) PA_RESHAPE(__nv_bfloat16, true);
      PA_RESHAPE(__nv_bfloat16, false);
    default:
      return cudaErrorInvalidValue;
  }
#undef PA_RESHAPE
}

cudaError_t launch_reshape_4bit(const void* key, const void* value,
                                pa_dtype kv_dtype, int64_t num_tokens,
                                int64_t key_stride, int64_t value_stride,
                                void* k_cache, void* v_cache,
                                pa_dtype cache_dtype, int64_t num_blocks,
                                int num_kv_heads, int head_dim,
                                const int64_t* slot_mapping, float k_scale,
                                float v_scale, unsigned* err,
                                cudaStream_t stream) {
  const int64_t warps = num_tokens * 2 * num_kv_heads;
  const int64_t blocks = (warps * 32 + kThreads - 1) / kThreads;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  const bool nv = cache_dtype == PA_NVFP4;
  uint8_t* kc = static_cast<uint8_t*>(k_cache);
  uint8_t* vc = static_cast<uint8_t*>(v_cache);
  const int64_t slots = num_blocks * kBS;
#define PA_RESHAPE4(T, NV, D)                                                  \
  reshape_4bit_kernel<T, NV, D><<<(unsigned)blocks, kThreads, 0, stream>>>(    \
      static_cast<const T*>(key), static_cast<const T*>(value), num_tokens,    \
      key_stride, value_stride, kc, vc, slots, num_kv_heads, slot_mapping,     \
      k_scale, v_scale, err)
#define PA_RESHAPE4_D(T)                                                       \
  if (head_dim == 128) {                                                       \
    if (nv) PA_RESHAPE4(T, true, 128); else PA_RESHAPE4(T, false, 128);        \
  } else {                                                                     \
    if (nv) PA_RESHAPE4(T, true, 64); else PA_RESHAPE4(T, false, 64);          \
  }
  switch (kv_dtype) {
    case PA_F32: PA_RESHAPE4_D(float); break;
    case PA_F16: PA_RESHAPE4_D(__half); break;
    case PA_BF16: PA_RESHAPE4_D(__nv_bfloat16); break;
    default: return cudaErrorInvalidValue;
  }
#undef PA_RESHAPE4_D
#undef PA_RESHAPE4
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, int64_t num_blocks,
                               int64_t block_bytes,
                               const int64_t* block_mapping, int64_t num_pairs,
                               unsigned* err, cudaStream_t stream) {
  const int64_t vecs = block_bytes / 16;
  int64_t gx = (vecs + kThreads - 1) / kThreads;
  if (gx > 64) gx = 64;
  const int64_t gy = num_pairs < 65535 ? num_pairs : 65535;
  copy_blocks_kernel<<<dim3((unsigned)gx, (unsigned)gy), kThreads, 0, stream>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_blocks,
      vecs, block_mapping, num_pairs, err);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace pa

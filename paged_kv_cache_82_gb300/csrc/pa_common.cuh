// pa_common.cuh -- shared device helpers of libpa (sm_103a only).
//
// Inline-PTX wrappers for the Blackwell data movers used by the attention
// kernel (mbarrier, cp.async.bulk.tensor), the legacy warp-level MMA used for
// the bandwidth-bound decode contraction, and the metadata checks that every
// kernel applies to device-resident indices.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

constexpr int kBS = PA_BLOCK_SIZE;  // tokens per physical block

__host__ __device__ constexpr bool is_4bit(int t) {
  return t == PA_INT4 || t == PA_NVFP4;
}

// ----------------------------------------------------------------------------
// device error word (one per device, defined in pa_api.cu; kernels receive
// its address)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void flag_error(unsigned* err, unsigned bits) {
  atomicOr(err, bits);
}

// ----------------------------------------------------------------------------
// step metadata of one request, validated the same way by every kernel
// ----------------------------------------------------------------------------
struct ReqMeta {
  int q0;  // first query token
  int n;   // query tokens this step
  int L;   // keys in the cache, this step's included
  int nb;  // physical blocks holding the keys
  bool ok;
};

__device__ __forceinline__ ReqMeta load_req(const int32_t* __restrict__ qsl,
                                            const int32_t* __restrict__ seq_lens,
                                            int r, int64_t num_tokens,
                                            int max_query_len, int max_seq_len,
                                            int max_blocks_per_seq) {
  ReqMeta m;
  m.q0 = __ldg(qsl + r);
  int q1 = __ldg(qsl + r + 1);
  m.n = q1 - m.q0;
  m.L = __ldg(seq_lens + r);
  m.nb = (m.L + kBS - 1) / kBS;
  m.ok = m.q0 >= 0 && m.n >= 0 && (int64_t)q1 <= num_tokens &&
         m.n <= max_query_len && m.L >= m.n && m.L <= max_seq_len &&
         m.nb <= max_blocks_per_seq;
  return m;
}

// ----------------------------------------------------------------------------
// shared-memory address helpers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// ----------------------------------------------------------------------------
// mbarrier (CTA scope)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::
          "r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(
                   bar)
               : "memory");
}

// Test-and-wait on a phase: the thread may be suspended (up to the hint, in
// ns) until the phase completes, instead of spinning on the issue slots.
#ifndef PA_SUSPEND_HINT_NS
#define PA_SUSPEND_HINT_NS 0  // 0: the hardware's default time limit
#endif

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
#if PA_SUSPEND_HINT_NS > 0
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(PA_SUSPEND_HINT_NS)
      : "memory");
#else
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
#endif
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: gives up after g_wait_limit_ns of wall time (2 s unless
// pa_set_wait_limit_ns says otherwise).  A pipeline whose wait gives up
// records PA_DEV_ERR_TIMEOUT and unwinds; it never spins forever.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Per translation unit (static), per device; written by the unit's
// set_pipeline_hooks() on the host.
//  g_wait_limit_ns -- the longest one bounded wait spins, in ns;
//  g_skip_copy     -- testing hook: the pipeline stage whose copy CTA 0 of
//                     the unit's pipelined kernels never issues (-1: none),
//                     so that the waits on that stage can only run out.
static __device__ uint64_t g_wait_limit_ns = kWaitLimitNs;
static __device__ long long g_skip_copy = -1;

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar,
                                                  uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t limit = g_wait_limit_ns;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && global_timer_ns() - t0 > limit) return false;
  }
}

// The stage CTA 0 of this grid leaves out (testing hook), -1 elsewhere.
__device__ __forceinline__ long long skipped_copy() {
  return blockIdx.x == 0 ? g_skip_copy : -1;
}

// ----------------------------------------------------------------------------
// exclusive block-wide prefix sum of one value per thread (every thread of
// the block calls it); *total receives the block's sum.  warp_sums: 32
// elements of shared memory.
// ----------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ T block_scan_excl(T v, T* total, T* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const T o = __shfl_up_sync(~0u, inc, d);
    if (lane >= d) inc += o;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    T w = lane < nw ? warp_sums[lane] : T(0);
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const T o = __shfl_up_sync(~0u, w, d);
      if (lane >= d) w += o;
    }
    if (lane < nw) warp_sums[lane] = w;
    if (lane == nw - 1) *total = w;
  }
  __syncthreads();
  const T ex = (warp == 0 ? T(0) : warp_sums[warp - 1]) + inc - v;
  __syncthreads();
  return ex;
}

// ----------------------------------------------------------------------------
// programmatic dependent launch: let the next grid in the stream start its
// prologue; wait until the previous grid has completed and its writes are
// visible
// ----------------------------------------------------------------------------
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ----------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) loads into shared memory, completing on an
// mbarrier.  Coordinates are element indices, innermost first.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(
                   reinterpret_cast<uint64_t>(map))
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map,
                                            uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// L2 prefetch of the box that a load with the same coordinates copies: no
// shared memory, no completion; a later load of the box then hits L2
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y,
                                                   int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}
// the same for a contiguous range (16-byte aligned, a multiple of 16 bytes)
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map,
                                            uint32_t bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// untiled bulk copy global -> shared, completing on an mbarrier: both
// addresses 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src,
                                          uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// ----------------------------------------------------------------------------
// warp-level MMA m16n8k16, fp32 accumulate (A row-major, B column-major)
// ----------------------------------------------------------------------------
template <bool kBF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                         uint32_t b0, uint32_t b1) {
  if constexpr (kBF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// two fp32 -> packed 16-bit pair (lo = first), round to nearest even
template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kBF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// four E4M3 bytes (lowest byte first) -> two packed f16 pairs, exact: bytes
// 0, 1 into lo and 2, 3 into hi.  The two 16-bit halves of the word feed the
// conversions directly (no shift to bring the upper pair down).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four_bytes, uint32_t& lo,
                                                  uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(four_bytes));
}

// ----------------------------------------------------------------------------
// scalar conversions for the element types
// ----------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) {
  return __half2float(x);
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) {
  return __float2half_rn(x);
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// E2M1 (OCP Microscaling FP4: sign bit 3, exponent bits 2-1 with bias 1,
// mantissa bit 0; values 0, 0.5, 1, 1.5, 2, 3, 4, 6).
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  const float mag = e == 0 ? 0.5f * (float)m
                           : (1.0f + 0.5f * (float)m) * (float)(1u << (e - 1));
  return (c & 8u) ? -mag : mag;
}

// E2M1 code nearest to y: the magnitude code counts the midpoints between
// grid values that |y| has passed; a midpoint itself goes to the code with
// mantissa bit 0 (ties to even); beyond 6 it saturates.  The sign bit
// follows y's sign.
__device__ __forceinline__ uint32_t e2m1_encode(float y) {
  const float a = fabsf(y);
  const uint32_t mag = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) +
                       (uint32_t)(a > 1.25f) + (uint32_t)(a >= 1.75f) +
                       (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
                       (uint32_t)(a > 5.0f);
  return (signbit(y) ? 8u : 0u) | mag;
}

__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c),
                                         __NV_E4M3);
  return __half2float(__half(h));
}

}  // namespace pa

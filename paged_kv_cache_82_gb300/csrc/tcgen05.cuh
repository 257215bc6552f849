// tcgen05.cuh -- inline-PTX wrappers for the 5th-generation tensor cores of
// sm_103a: tensor-memory (TMEM) allocation, loads and stores, the MMA with
// shared-memory or TMEM operands, its completion tracking on an mbarrier, and
// the shared-memory matrix descriptor for 128-byte swizzled tiles.
#pragma once

#include <stdint.h>

namespace pa {

// ---------------------------------------------------------------------------
// ordering of tcgen05 operations against thread synchronisation
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// generic-proxy writes to shared memory made visible to the tensor core
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMEM allocation (one warp executes each of these)
// ---------------------------------------------------------------------------
template <uint32_t kCols>
__device__ __forceinline__ void tc_alloc(uint32_t slot_smem) {
  asm volatile(
      "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
          slot_smem),
      "n"(kCols)
      : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                   : "memory");
}
template <uint32_t kCols>
__device__ __forceinline__ void tc_dealloc(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(
                   taddr),
               "n"(kCols)
               : "memory");
}

// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 family format):
// start address, leading- and stride-dimension byte offsets (all >> 4), the
// descriptor version (1) and the swizzle mode (2 = 128 B).  The operand tile
// must sit on a 1024-byte boundary; the start address may step inside a
// swizzle atom along K (32 bytes per 16 elements of 16 bits).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t saddr, uint32_t lbo,
                                                  uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) |
         ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) |
         ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16 with fp32 accumulation: A and B both
// bf16 (else both f16), A K-major, B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t tc_idesc_f16(bool bf16, bool b_mn_major,
                                                    int m, int n) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

// ---------------------------------------------------------------------------
// MMA issue.  Each call is executed by a whole, converged warp: one lane,
// chosen by elect.sync, issues the whole group of MMAs from a single asm
// block.  (Issued one by one from a lone lane next to busy warps on the same
// SM sub-partition, each MMA took two to three times the tensor core's time
// for it; a group issued back to back keeps the tensor core fed.)
// Descriptor arithmetic: the start address field holds (byte address >> 4)
// in its low 14 bits; shared addresses stay below 2^18 bytes and every
// offset added here keeps the field below 2^14, so a plain 64-bit add moves
// the start address.
// ---------------------------------------------------------------------------

// S = A * B^T over K = 128: A (M rows) and B (N rows) K-major in 128-byte
// swizzled tiles of 64 columns, the two column halves kHalfBytes apart.
// Step kk reads columns 16kk .. 16kk + 15; the first step overwrites D.
template <uint32_t kHalfBytes>
__device__ __forceinline__ void tc_mma_ss_k128(uint32_t d_tmem, uint64_t a_desc,
                                               uint64_t b_desc, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b64 a1, a2, a3, a4, a5, a6, a7, b1, b2, b3, b4, b5, b6, b7;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"
      "add.s64 a4, %1, %4;\n\tadd.s64 a5, a4, 2;\n\tadd.s64 a6, a4, 4;\n\tadd.s64 a7, a4, 6;\n\t"
      "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"
      "add.s64 b4, %2, %4;\n\tadd.s64 b5, b4, 2;\n\tadd.s64 b6, b4, 4;\n\tadd.s64 b7, b4, 6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a4, b4, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a5, b5, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a6, b6, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a7, b7, %3, 1;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "n"(kHalfBytes >> 4)
      : "memory");
}

// O (+)= P * V for four 16-row steps of B: A (P) in tensor memory, each step
// as two 16-bit parts, hi in columns 16j .. 16j + 7 and lo in 16j + 8 ..
// 16j + 15 from a_tmem; B (V) in shared memory, step j at b_desc moved by
// j * kStepBytes.  acc = 0: the first MMA overwrites D.
template <uint32_t kStepBytes>
__device__ __forceinline__ void tc_mma_ts_pair4(uint32_t d_tmem, uint32_t a_tmem,
                                                uint64_t b_desc, uint32_t idesc,
                                                uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t"
      ".reg .b64 b1, b2, b3;\n\t"
      "elect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
      "add.u32 a4, %1, 32;\n\tadd.u32 a5, %1, 40;\n\tadd.u32 a6, %1, 48;\n\t"
      "add.u32 a7, %1, 56;\n\t"
      "add.s64 b1, %2, %5;\n\tadd.s64 b2, b1, %5;\n\tadd.s64 b3, b2, %5;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], %2, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b1, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b1, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b2, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b2, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b3, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], b3, %3, 1;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc),
      "n"(kStepBytes >> 4)
      : "memory");
}
// one step of the above (two MMAs)
__device__ __forceinline__ void tc_mma_ts_pair1(uint32_t d_tmem, uint32_t a_tmem,
                                                uint64_t b_desc, uint32_t idesc,
                                                uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 a1;\n\t"
      "elect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "add.u32 a1, %1, 8;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], %2, %3, 1;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}

// The mbarrier gets one arrival once every MMA this thread issued before it
// has completed.  tc_commit: the calling thread alone; tc_commit_elect: a
// whole converged warp, for the MMAs its elected lane issued (elect.sync
// picks the same lane every time in a fully active warp).
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];\n\t}" ::"r"(bar)
      : "memory");
}

// ---------------------------------------------------------------------------
// TMEM <-> registers, shape 32x32b: thread t of the warp moves lane
// (lane base + t), consecutive 32-bit columns from the given one.  The warp
// may only touch its own quarter of the lanes (32 * (warp id % 4)).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,"
      "%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,"
      "%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]),
        "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,"
      "%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,"
      "%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
      "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]),
      "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),
      "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,"
      "%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
      "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]),
      "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Wait for the loads, with the destination registers as operands: the
// compiler may not move their uses above the wait.
template <int N>
__device__ __forceinline__ void tc_wait_ld_dep(uint32_t (&r)[N]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}
template <int M, int N>
__device__ __forceinline__ void tc_wait_ld_dep(uint32_t (&r)[M][N]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < M; ++j)
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[j][i]));
}
__device__ __forceinline__ void tc_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace pa

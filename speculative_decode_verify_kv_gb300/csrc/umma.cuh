// umma.cuh -- 5th-generation tensor core (tcgen05) primitives for sm_103a:
// TMEM allocation, shared-memory operand descriptors, the single-thread
// UMMA issue, commit-to-mbarrier, and TMEM -> register loads.
#pragma once

#include "common.cuh"

namespace trtv {

// Shared-memory descriptor of a K-major bf16 operand stored as rows of
// 128 bytes (64 elements) with the 128-byte swizzle that TMA writes: eight-row
// core groups 1024 bytes apart.  `saddr` is the start of the tile (or the start
// plus 32 B per 16-element k-step inside the 128-byte row).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16 >> 4) << 16;     // leading byte offset (unused when swizzled)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;   // stride byte offset: next 8-row group
  d |= static_cast<uint64_t>(1) << 46;           // descriptor version
  d |= static_cast<uint64_t>(2) << 61;           // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (both K-major), f32 accumulator.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4 with E4M3 A and B (format code 0, both
// K-major), f32 accumulator.
__host__ __device__ constexpr uint32_t umma_idesc_e4m3(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}



// Shared-memory descriptor with explicit leading / stride byte offsets
// (128-byte swizzle).
__device__ __forceinline__ uint64_t umma_desc_sw128_lbo_sbo(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(lbo >> 4) << 16;
  d |= static_cast<uint64_t>(sbo >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one UMMA, issued by a single thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every UMMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 consecutive f32 columns of this thread's TMEM lane (32x32b shape: warp
// q of a warpgroup reads lanes 32q .. 32q + 31).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace trtv

namespace trtv {


// Store 16 consecutive 32-bit columns of this thread's TMEM lane (32x32b).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}


// Shared-memory descriptor of an MN-major bf16 operand in the same
// 128B-swizzled rows (here: V, one row of 64 head dims per token in each of
// the tile's two 64-column halves).  Along K (tokens) the 8-row groups are
// 1024 bytes apart (stride byte offset); along N the 64-column swizzle atoms
// are `atom_stride` bytes apart (leading byte offset), so one N = 128 UMMA
// covers both halves.
__device__ __forceinline__ uint64_t umma_desc_sw128_mn(uint32_t saddr, uint32_t atom_stride) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(atom_stride >> 4) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

}  // namespace trtv

namespace trtv {

// tcgen05.ld of 32 columns without waiting; pair with tmem_ld_wait_dep.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Wait for the outstanding tcgen05.ld; the registers pass through the wait so
// no use of them can be scheduled ahead of it.
__device__ __forceinline__ void tmem_ld_wait_dep(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

}  // namespace trtv

namespace trtv {

// tcgen05.ld of 8 / 16 consecutive 32-bit columns (32x32b shape), no wait;
// pair with tmem_ld_wait_dep of the same width.
__device__ __forceinline__ void tmem_ld_async(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait_dep(uint32_t (&r)[8]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_ld_wait_dep(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// Store 8 consecutive 32-bit columns of this thread's TMEM lane (32x32b).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

}  // namespace trtv

namespace trtv {



// umma_commit from one elected lane (the whole warp executes the call).
__device__ __forceinline__ void umma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n" ::"r"(smem_u32(bar))
      : "memory");
}

// A shared-memory descriptor moved by `bytes` (a multiple of 16): the start
// address is the low 14-bit field in units of 16 bytes.
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

}  // namespace trtv

namespace trtv {

// Four UMMAs into one accumulator from one elected lane of the warp (the
// whole warp executes the call): descriptors a[i], b[i]; the first
// accumulates only if `acc_first`, the others always.  One elect and one
// asm block for the burst keep the issuing thread's work between the
// instructions to the issue itself.
template <bool FP8>
__device__ __forceinline__ void umma4_elect(uint32_t d_tmem, const uint64_t (&a)[4], const uint64_t (&b)[4],
                                            uint32_t idesc, uint32_t acc_first) {
  if constexpr (FP8) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %10, 0;\n\t"
        "setp.eq.b32 t, 1, 1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %9, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %3, %4, %9, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %5, %6, %9, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %7, %8, %9, t;\n\t}\n" ::"r"(d_tmem),
        "l"(a[0]), "l"(b[0]), "l"(a[1]), "l"(b[1]), "l"(a[2]), "l"(b[2]), "l"(a[3]), "l"(b[3]), "r"(idesc),
        "r"(acc_first)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %10, 0;\n\t"
        "setp.eq.b32 t, 1, 1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %9, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %4, %9, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %9, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %9, t;\n\t}\n" ::"r"(d_tmem),
        "l"(a[0]), "l"(b[0]), "l"(a[1]), "l"(b[1]), "l"(a[2]), "l"(b[2]), "l"(a[3]), "l"(b[3]), "r"(idesc),
        "r"(acc_first)
        : "memory");
  }
}

}  // namespace trtv

namespace trtv {

// Four UMMAs into one accumulator with A read from tensor memory (columns
// a[i]) and B from shared memory (descriptors b[i]), issued by one elected
// lane of the warp (the whole warp executes the call); the first accumulates
// only if `acc_first`, the others always.
template <bool FP8>
__device__ __forceinline__ void umma4_tmem_a_elect(uint32_t d_tmem, const uint32_t (&a)[4], const uint64_t (&b)[4],
                                                   uint32_t idesc, uint32_t acc_first) {
  if constexpr (FP8) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %10, 0;\n\t"
        "setp.eq.b32 t, 1, 1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %9, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%3], %4, %9, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%5], %6, %9, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%7], %8, %9, t;\n\t}\n" ::"r"(d_tmem),
        "r"(a[0]), "l"(b[0]), "r"(a[1]), "l"(b[1]), "r"(a[2]), "l"(b[2]), "r"(a[3]), "l"(b[3]), "r"(idesc),
        "r"(acc_first)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %10, 0;\n\t"
        "setp.eq.b32 t, 1, 1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %9, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %4, %9, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %9, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %9, t;\n\t}\n" ::"r"(d_tmem),
        "r"(a[0]), "l"(b[0]), "r"(a[1]), "l"(b[1]), "r"(a[2]), "l"(b[2]), "r"(a[3]), "l"(b[3]), "r"(idesc),
        "r"(acc_first)
        : "memory");
  }
}

}  // namespace trtv

namespace trtv {

// 16-lane TMEM shapes (lanes base .. base + 15 of the warp's quadrant).
// .16x256b, repetition k (columns base + 8k .. + 7): thread t holds lane
// t / 4 columns 8k + 2 (t % 4) and + 1 in r[4k], r[4k + 1], and lane t / 4 + 8
// the same columns in r[4k + 2], r[4k + 3].  .16x128b, repetition k (columns
// base + 4k .. + 3): thread t holds lane t / 4 column 4k + t % 4 in r[2k] and
// lane t / 4 + 8 in r[2k + 1].  Loads do not wait; pair with tmem_ld_wait_dep.
__device__ __forceinline__ void tmem_ld16x256_x8(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16x256_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16x256_x4(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile("tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
               : "memory");
}

__device__ __forceinline__ void tmem_st16x128_x8(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile("tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
               : "memory");
}

}  // namespace trtv

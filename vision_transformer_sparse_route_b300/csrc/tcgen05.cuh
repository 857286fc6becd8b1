// tcgen05.cuh -- inline-PTX helpers for the 5th-generation tensor cores of
// sm_100-family GPUs (sm_103a here): tensor-memory (TMEM) allocation, the
// shared-memory matrix descriptor, the instruction descriptor of kind::f16
// MMAs (bf16 in, f32 accumulate), the MMA itself, its completion through an
// mbarrier, and loads from TMEM into registers.
//
// Layout conventions used by this library: every operand tile in shared
// memory has 128-byte rows (64 bf16) written with the 128-byte swizzle (the
// 16-byte chunk c of row r sits at chunk position c ^ (r % 8)), 8-row groups
// 1024 bytes apart, from a 1024-byte aligned base. Such a tile is
//   - "K-major" when its rows are the M (or N) index and the 64 elements of a
//     row run along K: one MMA of K = 16 reads a 32-byte column slice, so the
//     descriptor for K step s starts 32 s bytes into the row;
//   - "MN-major" when its rows run along K and the 64 elements of a row along
//     N: K step s (16 rows) starts 2048 s bytes further.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace bra {

// ------------------------------------------------------------------- TMEM
// Allocates ncols columns (a power of two, 32 .. 512) of tensor memory for
// this CTA; one whole warp executes it. The TMEM address is written to the
// shared-memory word at dst.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}

// Lets other CTAs on this SM allocate (after this CTA's only allocation).
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Frees an allocation; one whole warp executes it.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Orders tcgen05 operations before / after a thread synchronisation.
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor of a 128-byte-swizzled tile (see above):
// start address, leading byte offset (lbo; unused by these layouts, 0), stride
// byte offset (sbo: between 8-row groups, 1024), version 1, swizzle mode 2
// (128 bytes).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Descriptor of a 64-byte-swizzled K-major tile: rows of 64 bytes (32 bf16),
// the 16-byte chunk c of row r at chunk position c ^ ((r / 2) % 4), 8-row
// groups 512 bytes apart, from a 512-byte aligned base; swizzle mode 4.
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)(512 >> 4) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)4 << 61;  // 64-byte swizzle
  return d;
}

// The same with a leading byte offset: for an MN-major tile wider than 64
// elements along N, the distance from one 64-element atom to the next.
__device__ __forceinline__ uint64_t smem_desc_sw128_lbo(uint32_t addr, uint32_t lbo,
                                                        uint32_t sbo) {
  return smem_desc_sw128(addr, sbo) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16);
}

// Instruction descriptor of a kind::f16 MMA with bf16 A and B and an f32
// accumulator: M x N, A K-major, B K-major (b_mn_major = 0) or MN-major (1).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int b_mn_major) {
  return (1u << 4)                    // D format: f32
         | (1u << 7)                  // A format: bf16
         | (1u << 10)                 // B format: bf16
         | ((uint32_t)b_mn_major << 16)
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

// -------------------------------------------------------------------- MMA
// D[tmem] (+)= A[smem] * B[smem], issued by one thread. accumulate = 0
// overwrites D.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier at bar receives one arrival once every MMA this thread issued
// before has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// --------------------------------------------------------------- TMEM loads
// 32 consecutive columns of this warp's 32 TMEM lanes (32x32b shape: lane i
// of the warp gets TMEM lane (warp % 4) * 32 + i), one 32-bit value per
// column into r[0..31]. Complete after tmem_ld_wait().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// One column of this warp's 32 TMEM lanes.
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr) : "memory");
  return r;
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace bra

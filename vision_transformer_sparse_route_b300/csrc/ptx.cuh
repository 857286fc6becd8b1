// ptx.cuh -- inline-PTX helpers for sm_103a: shared-memory addresses,
// mbarriers with bounded waits, TMA tensor copies, ldmatrix and the bf16
// warp-level MMA. Included once, by bra.cu.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bra {

// Bits of the device status word (read by bra_device_status).
constexpr unsigned kStatusTimeout = 1u;  // an mbarrier wait gave up
constexpr unsigned kStatusBadIndex = 2u; // a routing index was out of range

// One status word per device; kernels OR bits into it, the host reads it.
__device__ unsigned g_status;

// A wait gives up after this long (nanoseconds of the global timer), far
// longer than any copy this library issues takes.
constexpr uint64_t kWaitLimitNs = 500000000ull;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(count)
               : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// One arrival on bar (no transaction bytes).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Parity to wait for on a "full" barrier at the n-th use of its ring slot,
// and on a "free" barrier (the first use of a slot does not wait: a fresh
// barrier's preceding phase counts as complete).
__device__ __forceinline__ uint32_t full_parity(int n) { return (uint32_t)(n & 1); }
__device__ __forceinline__ uint32_t free_parity(int n) { return (uint32_t)((n & 1) ^ 1); }

// Non-blocking test of phase `parity` of `bar` (try_wait may suspend the
// thread for a while; a thread that polls several barriers must not).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for phase `parity` of `bar` to complete, for at most limit_ns.
// On giving up it sets kStatusTimeout and returns false; the caller carries
// on (so that every thread still reaches every barrier of the block). Once
// the timeout bit is set (until the host clears it), waits that do not
// succeed at once return false immediately, so a launch that went wrong ends
// quickly instead of timing out wait by wait.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  // after one wait of this launch has given up, later ones do not wait again
  if (*reinterpret_cast<volatile unsigned *>(&g_status) & kStatusTimeout) return false;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit_ns) {
      atomicOr(&g_status, kStatusTimeout);
      return false;
    }
  return true;
}

// Waits for phase `parity` of `bar` for at most limit_ns even after a wait of
// this launch has given up: used before a CTA exits or frees memory, so that
// no copy or MMA it issued is still in flight. Sets kStatusTimeout on giving up.
__device__ __forceinline__ bool mbar_drain(uint64_t *bar, uint32_t parity,
                                           uint64_t limit_ns = kWaitLimitNs) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit_ns) {
      atomicOr(&g_status, kStatusTimeout);
      return false;
    }
  return true;
}

// Called by one thread at the very end of a kernel that issues TMA copies:
// after a wait of this launch has given up, the normal hand-offs no longer
// guarantee that every copy has landed, so the CTA stays alive a little
// longer (its shared memory must outlive its copies).
__device__ __forceinline__ void settle_after_timeout() {
  if (*reinterpret_cast<volatile unsigned *>(&g_status) & kStatusTimeout) {
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 200000ull) {
    }
  }
}

// -------------------------------------------------------------------- TMA
// 4-D tiled load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map,
                                            uint64_t *bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_"
      "tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar))
      : "memory");
}

// 4-D tiled store of one box from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map,
                                             const void *src, int c0, int c1,
                                             int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, "
      "%3, %4, %5}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

__device__ __forceinline__ void tma_store_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until every committed store has finished reading shared memory.
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map))
               : "memory");
}

// ------------------------------------------------------- ldmatrix and MMA
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0,
                                        uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0,
                                              uint32_t &r1, uint32_t &r2,
                                              uint32_t &r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr));
}

// Transpose of an 8x8 matrix of 16-bit values held one row pair per lane
// (lane l: row l / 4, columns 2 (l % 4) and 2 (l % 4) + 1, low half first).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// D = A * B + D, m16n8k16, bf16 inputs, f32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4],
                                               const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Packs two floats into bf16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) {
  return __uint_as_float(w << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t w) {
  return __uint_as_float(w & 0xffff0000u);
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a tile of 128-byte rows
// written by TMA with 128-byte swizzling into a 1024-byte-aligned buffer: the
// chunk index is XORed with the row index modulo 8.
__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

}  // namespace bra

namespace bra {

// One warp; its first thread waits on an mbarrier phase that expects 16
// bytes of copies none of which is ever issued, so the bounded wait gives up
// after limit_ns, sets kStatusTimeout and the kernel returns normally. It
// exercises the device-side failure path without a fault.
__global__ void bra_wait_timeout_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar, 16);
    mbar_wait(&bar, 0, limit_ns);
  }
  __syncwarp();
}

}  // namespace bra

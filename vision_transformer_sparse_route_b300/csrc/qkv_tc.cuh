// qkv_tc.cuh -- the Q/K/V projections in front of BRA on the 5th-generation
// tensor cores: q = x W_q^T + b_q, k = x W_k^T + b_k, v = x W_v^T + b_v for
// every token (page "CVPR2023：BiFormer中的双层路由注意力机制解析" §3,
// `q = self.q_proj(x)`, `k_proj`, `v_proj`), bf16 in, f32 accumulate, one
// rounding to bf16.
//
// x is [M][C] (the tokens of a channels-last map), W [3C][C] in the [out][in]
// layout of a linear layer (rows 0..C-1 give q, C..2C-1 k, 2C..3C-1 v), bias
// [3C] f32. A persistent CTA per SM walks 128-token tiles of x:
//   warp 0     TMA copies: the tile's x (C / 64 boxes of 128 tokens x 64
//              channels, 128-byte swizzled) into a ring, and the weight tiles
//              (64 output rows x 64 input channels): kept resident when the
//              whole W fits (C <= 128), else streamed through a ring;
//   warp 1     one thread issues, per group of output tiles (3 or 1
//              64-channel tiles), the C / 16 MMAs of D = x_tile W_group^T
//              (M = 128, N = 192 or 64, K = 16 each, both operands K-major)
//              into one of the tensor-memory accumulators;
//   warps 4-11, two epilogue warpgroups taking alternate accumulators,
//              each owning the 128 lanes (one token each): add the bias,
//              round to bf16 into a 128-byte-swizzled staging tile, and each
//              warp copies its own 32 rows out to q, k or v with 16-byte
//              stores, four whole rows (512 contiguous bytes) a warp
//              instruction. (The SM's TMA unit takes about the same time for
//              a box whatever its size; left to the x loads it keeps them
//              short.)
// With W resident (C <= 128) three 64-channel output tiles form one MMA
// group of N = 192 against W stored atom-major ([ka][nt][64 rows], so the
// group's 192 rows are contiguous): a third of the MMA instructions of
// N = 64, whose issue rate is what bounds short bursts.
// Token rows past M read zeros (the x copy's fill) and are not stored.
#pragma once

#include "attend_bf16.cuh"
#include "tcgen05.cuh"

namespace bra {

constexpr int kQkvEpi = 2;                // epilogue warpgroups
constexpr int kQkvThreads = 128 + 128 * kQkvEpi;
constexpr uint32_t kQkvTmemCols = 512;

struct QkvGeom {
  int M, K, N;      // x [M][K], W [N][K]; outputs N channels in all
  int ow;           // channels of each output tensor (N: one tensor; N / 3: q, k, v)
  int ka;           // 64-channel atoms along K, K / 64
  int nt;           // 64-channel output tiles, N / 64
  int tiles;        // 128-token tiles
  int nx, nw, ns;   // x ring (<= 4), weight ring (<= 12), staging tiles (1 to 3 for
                    // each epilogue warpgroup)
  int w_resident;   // the whole W stays in shared memory (nw == nt), stored atom-major
                    // ([ka][nt][64 rows]) so that 3 output tiles form one N = 192 operand
  int gw;           // output tiles per MMA group: 3 (N = 192) with W resident and nt a
                    // multiple of 3, else 1
  int nacc;         // tensor-memory accumulators: 2 of 256 columns (gw 3) or 4 of 64
  uint32_t off_w, off_st, off_b, off_bar;  // x ring at 0
};

enum QkvBar {
  kQbFx = 0,      // [4] x tile landed
  kQbXfree = 4,   // [4] x tile read (MMA commit)
  kQbFw = 8,      // [12] weight tile landed
  kQbWfree = 20,  // [12] weight tile read (MMA commit)
  kQbAfull = 32,  // [8] accumulator complete (MMA commit)
  kQbAfree = 40,  // [8] accumulator read (128 arrivals)
  kQbDone = 48,   // every MMA complete, before the tensor memory is freed
  kQbCount = 49
};

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void qkv_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// RES: a residual of the output's layout is added before the rounding.
template <bool RES>
__global__ void __launch_bounds__(kQkvThreads, 1)
    bra_qkv_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                      const __grid_constant__ CUtensorMap tm_w,
                      const float *__restrict__ bias, QkvGeom g,
                      __nv_bfloat16 *__restrict__ oq, __nv_bfloat16 *__restrict__ ok,
                      __nv_bfloat16 *__restrict__ ov, const __nv_bfloat16 *__restrict__ res) {
  extern __shared__ uint8_t qkv_smem_raw[];
  uint8_t *smem = qkv_smem_raw + ((1024u - (smem_u32(qkv_smem_raw) & 1023u)) & 1023u);
  float *sb = reinterpret_cast<float *>(smem + g.off_b);  // [N]
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + g.off_bar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kQbCount);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int my_tiles = g.tiles > (int)blockIdx.x
                           ? (g.tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1
                           : 0;
  const uint32_t x_stage = (uint32_t)g.ka * 16384u, w_stage = (uint32_t)g.ka * 8192u;

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars[kQbFx + i], 1);
      mbar_init(&bars[kQbXfree + i], 1);
    }
    for (int i = 0; i < 12; ++i) {
      mbar_init(&bars[kQbFw + i], 1);
      mbar_init(&bars[kQbWfree + i], 1);
    }
    for (int i = 0; i < 4; ++i) {  // up to four accumulators
      mbar_init(&bars[kQbAfull + i], 1);
      mbar_init(&bars[kQbAfree + i], 128);
    }
    mbar_init(&bars[kQbDone], 1);
    fence_mbar_init();
  }
  for (int e = tid; e < g.N; e += kQkvThreads) sb[e] = bias ? __ldg(bias + e) : 0.f;
  if (warp == 1) {
    tmem_alloc(tmem_slot, kQkvTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ================================================= TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tm_x);
      prefetch_tensormap(&tm_w);
      int j = 0;  // weight tiles issued
      for (int li = 0; li < my_tiles; ++li) {
        const int tile = blockIdx.x + li * gridDim.x;
        const int xs = li % g.nx;
        mbar_wait(&bars[kQbXfree + xs], (uint32_t)(((li / g.nx) & 1) ^ 1));
        mbar_arrive_expect_tx(&bars[kQbFx + xs], x_stage);
        for (int a = 0; a < g.ka; ++a)
          tma_load_2d(smem + xs * x_stage + a * 16384, &tm_x, &bars[kQbFx + xs], 64 * a,
                      128 * tile);
        if (g.w_resident && li > 0) continue;
        for (int n = 0; n < g.nt; ++n, ++j) {
          const int ws = j % g.nw;
          if (!g.w_resident) mbar_wait(&bars[kQbWfree + ws], (uint32_t)(((j / g.nw) & 1) ^ 1));
          mbar_arrive_expect_tx(&bars[kQbFw + ws], w_stage);
          for (int a = 0; a < g.ka; ++a)
            tma_load_2d(smem + g.off_w +
                            (g.w_resident ? (uint32_t)(a * g.nt + n) * 8192u
                                          : ws * w_stage + a * 8192u),
                        &tm_w, &bars[kQbFw + ws], 64 * a, 64 * n);
        }
      }
      // no copy still in flight at exit
      for (int li = (my_tiles > g.nx ? my_tiles - g.nx : 0); li < my_tiles; ++li)
        mbar_drain(&bars[kQbFx + li % g.nx], (uint32_t)((li / g.nx) & 1));
      for (int jj = (j > g.nw ? j - g.nw : 0); jj < j; ++jj)
        mbar_drain(&bars[kQbFw + jj % g.nw], (uint32_t)((jj / g.nw) & 1));
    }
    __syncwarp();
  } else if (warp == 1) {
    // ====================================================== MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 64 * g.gw, 0);
      const uint32_t acc_cols = g.gw == 3 ? 256u : 64u;
      int j = 0, acc = 0;
      for (int li = 0; li < my_tiles; ++li) {
        const int xs = li % g.nx;
        mbar_wait(&bars[kQbFx + xs], (uint32_t)((li / g.nx) & 1));
        const uint32_t x0 = smem_u32(smem + xs * x_stage);
        // output tiles n0 .. n0 + gw - 1 as one MMA group (N = 64 gw)
        for (int n0 = 0; n0 < g.nt; n0 += g.gw, ++acc) {
          const int ws = g.w_resident ? n0 : j % g.nw;
          for (int jj = 0; jj < g.gw; ++jj)
            mbar_wait(&bars[kQbFw + ws + jj], g.w_resident ? 0u : (uint32_t)((j / g.nw) & 1));
          const int as = acc % g.nacc;
          mbar_wait(&bars[kQbAfree + as], free_parity(acc / g.nacc));
          tc_fence_after();
          for (int a = 0; a < g.ka; ++a) {
            const uint32_t w0 = smem_u32(
                smem + g.off_w +
                (g.w_resident ? (uint32_t)(a * g.nt + n0) * 8192u : ws * w_stage + a * 8192u));
            for (int s = 0; s < 4; ++s)
              mma_bf16_ss(tmem + as * acc_cols, smem_desc_sw128(x0 + a * 16384 + 32 * s, 1024),
                          smem_desc_sw128(w0 + 32 * s, 1024), idesc,
                          (a > 0 || s > 0) ? 1u : 0u);
          }
          mma_commit(&bars[kQbAfull + as]);
          if (!g.w_resident) {
            mma_commit(&bars[kQbWfree + ws]);
            ++j;
          }
        }
        mma_commit(&bars[kQbXfree + xs]);
      }
      mma_commit(&bars[kQbDone]);
      mbar_drain(&bars[kQbDone], 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ============================================ epilogue (TMEM lanes)
    const int eg = (warp - 4) >> 2;  // epilogue warpgroup: accumulators acc with acc % kQkvEpi == eg
    const int r = (tid - 128) & 127;  // token row of the tile
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t acc_cols = g.gw == 3 ? 256u : 64u;
    const int nsg = g.ns / kQkvEpi;  // staging tiles of this warpgroup
    int acc = 0, cnt = 0;            // MMA groups seen; output tiles this warpgroup staged
    for (int li = 0; li < my_tiles; ++li) {
      const int tile = blockIdx.x + li * gridDim.x;
      for (int n0 = 0; n0 < g.nt; n0 += g.gw, ++acc) {
        if (acc % kQkvEpi != eg) continue;
        const int as = acc % g.nacc;
        mbar_wait(&bars[kQbAfull + as], full_parity(acc / g.nacc));
        tc_fence_after();
        for (int jj = 0; jj < g.gw; ++jj, ++cnt) {
        const int n = n0 + jj, ss = eg * nsg + cnt % nsg;
        uint32_t v0[32], v1[32];
        tmem_ld32(lane_base + as * acc_cols + jj * 64, v0);
        tmem_ld32(lane_base + as * acc_cols + jj * 64 + 32, v1);
        tmem_ld_wait();
        if (jj == g.gw - 1) {  // the accumulator is read
          tc_fence_before();
          qkv_arrive(&bars[kQbAfree + as]);
        }
        // a warp stages and copies out only its own 32 rows: its previous
        // copy from this staging tile is complete
        __syncwarp();
        uint8_t *row = smem + g.off_st + ss * 16384 + r * 128;
        const float *bn = sb + n * 64;
        const int otiles = g.ow / 64;
        const int t = n / otiles, cc = n % otiles;  // output tensor; its 64-channel chunk
        const long long mr = 128ll * tile + r;       // this thread's token
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 16-byte chunk c: output channels 8c .. 8c+7
          const uint32_t *src = c < 4 ? v0 + 8 * c : v1 + 8 * (c - 4);
          const float4 b0 = *reinterpret_cast<const float4 *>(bn + 8 * c);
          const float4 b1 = *reinterpret_cast<const float4 *>(bn + 8 * c + 4);
          float f[8] = {__uint_as_float(src[0]) + b0.x, __uint_as_float(src[1]) + b0.y,
                        __uint_as_float(src[2]) + b0.z, __uint_as_float(src[3]) + b0.w,
                        __uint_as_float(src[4]) + b1.x, __uint_as_float(src[5]) + b1.y,
                        __uint_as_float(src[6]) + b1.z, __uint_as_float(src[7]) + b1.w};
          if (RES && mr < g.M) {  // the residual, added before the one rounding
            const uint4 rv = __ldg(reinterpret_cast<const uint4 *>(
                res + mr * g.ow + 64 * cc + 8 * c));
            const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              f[2 * e] += __uint_as_float(rw[e] << 16);
              f[2 * e + 1] += __uint_as_float(rw[e] & 0xffff0000u);
            }
          }
          const uint4 packed = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                          pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
          *reinterpret_cast<uint4 *>(row + ((c ^ (r & 7)) << 4)) = packed;
        }
        __syncwarp();
        // copy the staged rows out with the load/store units (the SM's TMA
        // unit is left to the x loads): 4 whole rows, 512 contiguous bytes,
        // per instruction
        {
          __nv_bfloat16 *dst = t == 0 ? oq : (t == 1 ? ok : ov);
          const uint8_t *tile_st = smem + g.off_st + ss * 16384;
          const int w4 = warp & 3, ch = lane & 7;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = 32 * w4 + 4 * i + (lane >> 3);
            const long long m = 128ll * tile + rr;
            const uint4 val =
                *reinterpret_cast<const uint4 *>(tile_st + rr * 128 + ((ch ^ (rr & 7)) << 4));
            if (m < g.M) *reinterpret_cast<uint4 *>(dst + m * g.ow + 64 * cc + 8 * ch) = val;
          }
        }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kQkvTmemCols);
  if (tid == 0) settle_after_timeout();
}

}  // namespace bra

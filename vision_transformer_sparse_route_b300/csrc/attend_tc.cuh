// attend_tc.cuh -- fused routed attention + LePE on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory) for bf16 maps with 8 x 8
// regions (64 tokens), 64 channels (2 heads of 32) and up to 4 routed regions
// per query region: the BiFormer stage-1 shape and the 512 x 512 dense-
// prediction shape.
//
// Same operation as attend_bf16.cuh (page "CVPR2023：BiFormer中的双层路由
// 注意力机制解析" §3: k_g = gather(k, I_r), attn = softmax(q k_g^T * scale),
// out = attn v_g, out += lce(v); LePE of page "从静态到动态：BRA双层路由注意力
// 如何革新视觉Transformer的计算范式" §4; page "BiFormer: Vision Transformer mit
// Bi-Level-Routing-Attention": attention over the union of the routed
// regions, with dense matrix products only).
//
// One persistent CTA of 20 warps per SM walks the query regions ("units")
// blockIdx.x, blockIdx.x + gridDim.x, ... . The warps have roles:
//   warp 0     copies each unit's Q straight into a block-diagonal 128 x 64
//              operand in a Q ring: two TMA boxes of one head's 32 channels
//              (64-byte swizzled rows) land as [Q_h0][zeros][Q_h1], so that
//              rows 0-63 hold head 0's queries with channels 32-63 zero and
//              rows 64-127 head 1's with channels 0-31 zero (the two K atoms
//              share the zero block), and one M = 128 MMA computes both
//              heads' logits against one K tile; and each unit's V halo
//              (region plus ks/2 border, zero filled outside the image) into
//              a halo ring;
//   warp 1     one thread issues S = Q_bd K^T (M = 128, N = 64 topk, K = 64)
//              into a tensor-memory slot and O = P V block by block (M = 128,
//              N = 64, K = 64 keys per block) into the slot's first 64
//              columns, whichever has its inputs first (it polls without
//              blocking);
//   warps 2, 3 read the routing (one unit ahead) and copy the routed
//              regions' K tiles (warp 2) and V tiles (warp 3) by index into a
//              K ring and a V ring, each as soon as its own ring has room;
//   warps 4-7  own the 128 tensor-memory lanes (row r: head r / 64, query
//              r % 64): the row maximum of S, P = 2^(S d^-1/2 log2 e - max) as
//              bf16 (the operand of P V) into shared memory 64 keys at a time,
//              the row sum of that bf16 P in f32 (or the MMA forms it); then
//              O / sum plus the LePE from the O tile, rounded once to bf16
//              into a staging tile that the warpgroup copies out with
//              coalesced 16-byte stores. Two
//              such warpgroups take alternate units, so that one computes
//              while the other waits for its P V;
//   warps 12-19 the LePE stencil of each unit from the halo, ahead of the
//              tensor cores, into an f32 O tile: two groups of four warps on
//              alternate units (a thread: one channel pair, two columns,
//              eight rows).
// Only warps 2 and 3 read the routing index, so when the kernel is launched right
// after the routing grid (programmatic dependent launch) everything else --
// Q tiles, halos, LePE -- starts before that grid has finished. Every ring,
// slot and tile hand-off is an mbarrier, every wait bounded. The operand
// layouts are those of tcgen05.cuh (128-byte swizzled rows).
#pragma once

#include "attend_bf16.cuh"
#include "tcgen05.cuh"

namespace bra {

constexpr int kTcWarps = 20;
constexpr int kTcThreads = 32 * kTcWarps;
constexpr int kTcLepeThreads = 256;   // warps 12-19, two groups of 128 on alternate units
constexpr int kTcLepeWarp0 = 12;
constexpr uint32_t kTcTmemCols = 512;

struct TcGeom {
  int H, W, S, topk, R, units;
  int nq, nh, nk, nv;       // Q, halo, K and V ring stages (each <= 4)
  int nslot;                // tensor-memory slots (<= 4)
  uint32_t slot_cols;       // columns of a slot (>= 64 topk, a power of two)
  int halo_w, halo_h;
  uint32_t off_h, off_k, off_v, off_ones, off_p, off_o, off_st, off_w, off_bar;  // Q ring at 0
                            // (stages of 12 KB: Q_h0, zeros, Q_h1)
  int sum_mma;              // row sums from the P V MMA (one key block): N = 80, the
                            // 16 extra columns against a tile of ones
  uint32_t h_bytes;         // bytes of one halo stage
  float scale_log2;         // d^-1/2 * log2(e)
};

// Barrier slots (uint64 each) from off_bar; rings of up to four.
enum TcBar {
  kBarFq = 0,       // [4] Q operand landed (TMA)
  kBarQfree = 4,    // [4] Q operand read (MMA commit)
  kBarFh = 8,       // [4] halo landed (TMA)
  kBarHfree = 12,   // [4] halo read (128 LePE arrivals)
  kBarFk = 16,      // [4] K tiles landed (TMA)
  kBarKfree = 20,   // [4] K tiles read (MMA commit)
  kBarFv = 24,      // [4] V tiles landed (TMA)
  kBarVfree = 28,   // [4] V tiles read (MMA commit)
  kBarSfull = 32,   // [4] S in a tensor-memory slot (MMA commit)
  kBarOfull = 36,   // [4] O in a tensor-memory slot (MMA commit)
  kBarTfree = 40,   // [4] slot read (128 arrivals)
  kBarPfull = 44,   // [2] P block of softmax warpgroup g written (128 arrivals)
  kBarPfree = 46,   // [2] P block of softmax warpgroup g read (MMA commit)
  kBarOfill = 48,   // [2] LePE written into the O tile (128 arrivals)
  kBarOfree = 50,   // [2] O tile consumed and stored (128 arrivals)
  kBarDone = 52,    // every MMA complete (MMA commit), before the tensor memory is freed
  kBarCount = 53
};

template <int KS>
__global__ void __launch_bounds__(kTcThreads, 1)
    bra_attend_tc_kernel(const __grid_constant__ CUtensorMap tm_q,  // boxes of 32 channels
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_vh,
                         const int32_t *__restrict__ idx, const float *__restrict__ lepe_w,
                         const float *__restrict__ lepe_b, TcGeom g,
                         __nv_bfloat16 *__restrict__ out) {
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t *smem = tc_smem_raw + ((1024u - (smem_u32(tc_smem_raw) & 1023u)) & 1023u);
  float *sw = reinterpret_cast<float *>(smem + g.off_w);  // [KS*KS][64], bias [64]
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + g.off_bar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kBarCount);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int PAD = KS / 2;
  const int topk = g.topk;
  const int n_units = g.units > (int)blockIdx.x
                          ? (g.units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1
                          : 0;

  // ---- set-up: barriers, weights, the permanent zeros of the Q operands
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kBarPfull + i], 128);
      mbar_init(&bars[kBarPfree + i], 1);
      mbar_init(&bars[kBarOfill + i], kTcLepeThreads / 2);
      mbar_init(&bars[kBarOfree + i], 128);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars[kBarFq + i], 1);
      mbar_init(&bars[kBarQfree + i], 1);
      mbar_init(&bars[kBarFh + i], 1);
      mbar_init(&bars[kBarHfree + i], kTcLepeThreads / 2);
      mbar_init(&bars[kBarFk + i], 1);
      mbar_init(&bars[kBarKfree + i], 1);
      mbar_init(&bars[kBarFv + i], 1);
      mbar_init(&bars[kBarVfree + i], 1);
      mbar_init(&bars[kBarSfull + i], 1);
      mbar_init(&bars[kBarOfull + i], 1);
      mbar_init(&bars[kBarTfree + i], 128);
    }
    mbar_init(&bars[kBarDone], 1);
    fence_mbar_init();
  }
  for (int e = tid; e < 64 * KS * KS; e += kTcThreads) {
    const int tap = e / 64, c = e % 64;
    sw[e] = __ldg(lepe_w + (size_t)c * KS * KS + tap);
  }
  if (tid < 64) sw[KS * KS * 64 + tid] = lepe_b ? __ldg(lepe_b + tid) : 0.f;
  // the ones tile (bf16 1.0), the extra N columns of P V that give row sums
  if (g.sum_mma)
    for (int e = tid; e < 8192 / 16; e += kTcThreads)
      *reinterpret_cast<uint4 *>(smem + g.off_ones + e * 16) =
          make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
  // the zero block between Q_h0 and Q_h1 of every Q stage stays zero
  for (int e = tid; e < g.nq * 256; e += kTcThreads)
    *reinterpret_cast<uint4 *>(smem + (e >> 8) * 12288 + 4096 + (e & 255) * 16) =
        make_uint4(0, 0, 0, 0);
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTcTmemCols);
    tmem_relinquish();
  }
  fence_async_shared();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto unit_at = [&](int k, int &b, int &y0, int &x0) {
    const int u = blockIdx.x + k * gridDim.x;
    const int i = u % g.R;
    b = u / g.R;
    y0 = (i / g.S) * 8;
    x0 = (i % g.S) * 8;
  };

  if (warp == 0) {
    // ============================================ Q and halo producer
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_vh);
      for (int k = 0; k < n_units; ++k) {
        int b, y0, x0;
        unit_at(k, b, y0, x0);
        const int st = k % g.nq;
        mbar_wait(&bars[kBarQfree + st], free_parity(k / g.nq));
        mbar_arrive_expect_tx(&bars[kBarFq + st], 8192);
        uint8_t *qs = smem + st * 12288;
        tma_load_4d(qs, &tm_q, &bars[kBarFq + st], 0, x0, y0, b);          // head 0
        tma_load_4d(qs + 8192, &tm_q, &bars[kBarFq + st], 32, x0, y0, b);  // head 1
        const int hs = k % g.nh;
        mbar_wait(&bars[kBarHfree + hs], free_parity(k / g.nh));
        mbar_arrive_expect_tx(&bars[kBarFh + hs], g.h_bytes);
        tma_load_4d(smem + g.off_h + hs * g.h_bytes, &tm_vh, &bars[kBarFh + hs], 0, x0 - PAD,
                    y0 - PAD, b);
      }
      // no Q or halo copy still in flight at exit
      for (int k = (n_units > g.nq ? n_units - g.nq : 0); k < n_units; ++k)
        mbar_drain(&bars[kBarFq + k % g.nq], full_parity(k / g.nq));
      for (int k = (n_units > g.nh ? n_units - g.nh : 0); k < n_units; ++k)
        mbar_drain(&bars[kBarFh + k % g.nh], full_parity(k / g.nh));
    }
    __syncwarp();
  } else if (warp == 1) {
    // ====================================================== MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, 64 * topk, 0);
      const uint32_t idesc_o = idesc_bf16_f32(128, g.sum_mma ? 80 : 64, 1);
      int next1 = 0;           // next unit for S = Q_bd K^T
      int next2 = 0, blk = 0;  // next unit and key block for O = P V
      int pcnt0 = 0, pcnt1 = 0;  // P blocks consumed so far from each warpgroup's buffer
      uint64_t t_idle = 0;
      unsigned n_idle = 0;
      while (next2 < n_units) {
        bool progressed = false;
        // S of the next unit, as soon as its Q operand, K tiles and slot are ready
        if (next1 < n_units) {
          const int k = next1, qs = k % g.nq, ks_ = k % g.nk, sl = k % g.nslot;
          if (mbar_test_wait(&bars[kBarFq + qs], full_parity(k / g.nq)) &&
              mbar_test_wait(&bars[kBarFk + ks_], full_parity(k / g.nk)) &&
              mbar_test_wait(&bars[kBarTfree + sl], free_parity(k / g.nslot))) {
            tc_fence_after();
            const uint32_t d = tmem + sl * g.slot_cols;
            const uint32_t a0 = smem_u32(smem + qs * 12288);
            const uint32_t k0 = smem_u32(smem + g.off_k + ks_ * topk * 8192);
            // K steps 0-1: channels 0-31 (rows 0-63 Q_h0, 64-127 zeros);
            // K steps 2-3: channels 32-63 (rows 0-63 zeros, 64-127 Q_h1)
            for (int s = 0; s < 4; ++s)
              mma_bf16_ss(d, smem_desc_sw64(a0 + (s < 2 ? 32 * s : 4096 + 32 * (s - 2))),
                          smem_desc_sw128(k0 + 32 * s, 1024), idesc_s, s > 0);
            mma_commit(&bars[kBarSfull + sl]);
            mma_commit(&bars[kBarQfree + qs]);
            mma_commit(&bars[kBarKfree + ks_]);
            ++next1;
            progressed = true;
          }
        }
        // the next P block of the oldest unit whose S is out, once written
        if (next2 < next1) {
          const int k = next2, pb = k & 1, vs = k % g.nv, sl = k % g.nslot;
          if (mbar_test_wait(&bars[kBarPfull + pb], full_parity(pb ? pcnt1 : pcnt0)) &&
              (blk > 0 || mbar_test_wait(&bars[kBarFv + vs], full_parity(k / g.nv)))) {
            tc_fence_after();
            const uint32_t d = tmem + sl * g.slot_cols;
            const uint32_t p0 = smem_u32(smem + g.off_p + pb * 16384);
            const uint32_t v0 = smem_u32(smem + g.off_v + vs * topk * 8192) + blk * 8192;
            const uint32_t lbo = smem_u32(smem + g.off_ones) - v0;  // V atom -> ones atom
            for (int s = 0; s < 4; ++s)
              mma_bf16_ss(d, smem_desc_sw128(p0 + 32 * s, 1024),
                          smem_desc_sw128_lbo(v0 + s * 2048, g.sum_mma ? lbo : 0u, 1024),
                          idesc_o, (blk > 0 || s > 0) ? 1u : 0u);
            mma_commit(&bars[kBarPfree + pb]);
            if (pb) ++pcnt1; else ++pcnt0;
            if (++blk == topk) {
              mma_commit(&bars[kBarOfull + sl]);
              mma_commit(&bars[kBarVfree + vs]);
              blk = 0;
              ++next2;
            }
            progressed = true;
          }
        }
        // give up (and flag it) if nothing moves for as long as a bounded
        // wait; the clock is read once every 1024 idle polls
        if (progressed) {
          t_idle = 0;
          n_idle = 0;
        } else if ((++n_idle & 1023) == 0) {
          if (t_idle == 0) {
            t_idle = global_ns();
          } else if (global_ns() - t_idle > kWaitLimitNs ||
                     (*reinterpret_cast<volatile unsigned *>(&g_status) & kStatusTimeout)) {
            atomicOr(&g_status, kStatusTimeout);
            break;
          }
        }
      }
      mma_commit(&bars[kBarDone]);
      mbar_drain(&bars[kBarDone], 0);  // every MMA complete before the memory is freed
    }
    __syncwarp();
  } else if (warp == 2 || warp == 3) {
    // ================================ K (warp 2) and V (warp 3) producers
    const bool is_v = warp == 3;
    const CUtensorMap *tm = is_v ? &tm_v : &tm_k;
    const int nr = is_v ? g.nv : g.nk;
    uint64_t *full = &bars[is_v ? kBarFv : kBarFk];
    uint64_t *freed = &bars[is_v ? kBarVfree : kBarKfree];
    uint8_t *ring = smem + (is_v ? g.off_v : g.off_k);
    if (lane == 0) prefetch_tensormap(tm);
    grid_dependency_wait();  // the routing index comes from the previous grid
    // lane m < topk copies routed region m; its index is read one unit ahead
    int j_next = n_units > 0 && lane < topk ? __ldg(idx + (size_t)blockIdx.x * topk + lane) : 0;
    for (int k = 0; k < n_units; ++k) {
      const int u = blockIdx.x + k * gridDim.x;
      const int b = u / g.R, st = k % nr;
      const int j = j_next;
      if (k + 1 < n_units && lane < topk)
        j_next = __ldg(idx + (size_t)(u + gridDim.x) * topk + lane);
      int xj = 0, yj = g.H;  // a box wholly below the image is all fill (zeros)
      if (j < 0 || j >= g.R) {
        if (lane < topk && !is_v) atomicOr(&g_status, kStatusBadIndex);
      } else {
        xj = (j % g.S) * 8;
        yj = (j / g.S) * 8;
      }
      mbar_wait(&freed[st], free_parity(k / nr));
      if (lane == 0) mbar_arrive_expect_tx(&full[st], topk * 8192);
      __syncwarp();
      if (lane < topk) tma_load_4d(ring + (st * topk + lane) * 8192, tm, &full[st], 0, xj, yj, b);
    }
    // no K or V copy still in flight at exit
    for (int k = (n_units > nr ? n_units - nr : 0); k < n_units; ++k)
      mbar_drain(&full[k % nr], full_parity(k / nr));
  } else if (warp < kTcLepeWarp0) {
    // ========================== softmax and O epilogue (TMEM lanes), two
    // warpgroups taking alternate units
    const int wg = (warp - 4) >> 2;  // 0: warps 4-7, 1: warps 8-11
    const int r = (tid - 128) & 127;  // tensor-memory lane = operand row
    const int h = r >> 6, tq = r & 63;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float2 sc2 = make_float2(g.scale_log2, g.scale_log2);
    int pcnt = 0;  // P blocks this warpgroup has written (into its own buffer)
    // O of unit k (in its slot, once out) / row sum, plus the LePE that the
    // LePE warps left in the O tile, rounded once to bf16 into the staging
    // tile, which one thread stores with a TMA copy
    auto epilogue = [&](int k, float inv) {
      const int sl = k % g.nslot, ot = k & 1;
      mbar_wait(&bars[kBarOfull + sl], full_parity(k / g.nslot));
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(lane_base + sl * g.slot_cols + h * 32, v);
      if (g.sum_mma) inv = __uint_as_float(tmem_ld1(lane_base + sl * g.slot_cols + 64));
      tmem_ld_wait();
      if (g.sum_mma) inv = 1.f / inv;
      tc_fence_before();
      mbar_arrive(&bars[kBarTfree + sl]);
      mbar_wait(&bars[kBarOfill + ot], full_parity(k >> 1));
      // this warpgroup is done copying its previous unit out of the staging tile
      named_sync(3 + wg, 128);
      // O tile [64 tokens][16 chunks of 4 floats]: chunk c of token t sits at
      // chunk position c ^ (t % 8); staging tile [64 tokens][8 chunks of 8
      // bf16], 128-byte swizzled (chunk c at c ^ (t % 8)), as the store's
      // tensor map expects
      const float *orow =
          reinterpret_cast<const float *>(smem + g.off_o + ot * 16384) + tq * 64 + h * 32;
      uint8_t *srow_st = smem + g.off_st + ot * 8192 + tq * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 8 channels a step: O chunks 2c, 2c + 1
        const float4 l0 = *reinterpret_cast<const float4 *>(orow + (((2 * c) ^ (tq & 7)) << 2));
        const float4 l1 =
            *reinterpret_cast<const float4 *>(orow + (((2 * c + 1) ^ (tq & 7)) << 2));
        const uint4 packed = make_uint4(
            pack_bf16x2(fmaf(__uint_as_float(v[8 * c]), inv, l0.x),
                        fmaf(__uint_as_float(v[8 * c + 1]), inv, l0.y)),
            pack_bf16x2(fmaf(__uint_as_float(v[8 * c + 2]), inv, l0.z),
                        fmaf(__uint_as_float(v[8 * c + 3]), inv, l0.w)),
            pack_bf16x2(fmaf(__uint_as_float(v[8 * c + 4]), inv, l1.x),
                        fmaf(__uint_as_float(v[8 * c + 5]), inv, l1.y)),
            pack_bf16x2(fmaf(__uint_as_float(v[8 * c + 6]), inv, l1.z),
                        fmaf(__uint_as_float(v[8 * c + 7]), inv, l1.w)));
        *reinterpret_cast<uint4 *>(srow_st + (((h * 4 + c) ^ (tq & 7)) << 4)) = packed;
      }
      named_sync(3 + wg, 128);
      // copy the staged unit out with the load/store units: 8 threads a
      // token (its 128 bytes), four whole tokens a warp instruction (a TMA
      // store would hold up its issuing thread, and with it this warpgroup's
      // next P, for about half a microsecond)
      {
        int b, y0, x0;
        unit_at(k, b, y0, x0);
        const uint8_t *st = smem + g.off_st + ot * 8192;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int e = it * 128 + r, t = e >> 3, ch = e & 7;
          const uint4 val = *reinterpret_cast<const uint4 *>(st + t * 128 + ((ch ^ (t & 7)) << 4));
          *reinterpret_cast<uint4 *>(
              out + (((size_t)b * g.H + y0 + (t >> 3)) * g.W + x0 + (t & 7)) * 64 + 8 * ch) = val;
        }
      }
      mbar_arrive(&bars[kBarOfree + ot]);
    };
    for (int k = wg; k < n_units; k += 2) {
      const int sl = k % g.nslot;
      const uint32_t srow = lane_base + sl * g.slot_cols;
      mbar_wait(&bars[kBarSfull + sl], full_parity(k / g.nslot));
      tc_fence_after();
      // the row maximum of the raw logits (four independent chains), 32
      // columns at a time
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      for (int c0 = 0; c0 < 64 * topk; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(srow + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          m4[0] = max3(m4[0], __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
          m4[1] = max3(m4[1], __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
          m4[2] = max3(m4[2], __uint_as_float(v[j + 4]), __uint_as_float(v[j + 5]));
          m4[3] = max3(m4[3], __uint_as_float(v[j + 6]), __uint_as_float(v[j + 7]));
        }
      }
      const float base = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * g.scale_log2;
      const float2 nb = make_float2(-base, -base);
      // P (bf16) 64 keys at a time into this warpgroup's P buffer, and its
      // row sum (four chains) unless the MMA forms it
      float l4[4] = {0.f, 0.f, 0.f, 0.f};
      uint8_t *prow = smem + g.off_p + wg * 16384 + r * 128;
      // 32 keys (16-byte chunks 4 half .. 4 half + 3) of P from the logits in v
      auto emit = [&](const uint32_t(&v)[32], int half) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // 8 keys
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 8 * c + 2 * e;
            const float2 x = __ffma2_rn(
                make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), sc2, nb);
            pk[e] = exp2_bf16x2(x.x, x.y);
            if (!g.sum_mma) l4[e] += bf16_lo(pk[e]) + bf16_hi(pk[e]);
          }
          *reinterpret_cast<uint4 *>(prow + (((half * 4 + c) ^ (r & 7)) << 4)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      };
      for (int blk = 0; blk < topk; ++blk, ++pcnt) {
        mbar_wait(&bars[kBarPfree + wg], free_parity(pcnt));
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t v[32];
          tmem_ld32(srow + blk * 64 + half * 32, v);
          tmem_ld_wait();
          emit(v, half);
        }
        fence_async_shared();
        tc_fence_before();
        mbar_arrive(&bars[kBarPfull + wg]);
      }
      // this unit's O, as soon as its P V is out: while this warpgroup waits
      // for it the other one computes its softmax
      epilogue(k, 1.f / ((l4[0] + l4[1]) + (l4[2] + l4[3])));
    }
  } else {
    // ================================================ LePE into the O tile
    // two groups of four warps take alternate units; a thread: channel pair
    // cp, region columns 2 xp and 2 xp + 1, all 8 rows (each halo value it
    // loads feeds both columns)
    const int lg = (warp - kTcLepeWarp0) >> 2;           // LePE group: units k % 2 == lg
    const int lt = (tid - 32 * kTcLepeWarp0) & 127;      // 0..127
    const int cp = lt & 31, xp = lt >> 5;
    const int c = 2 * cp;
    float2 wgt[KS * KS];
#pragma unroll
    for (int e = 0; e < KS * KS; ++e) wgt[e] = *reinterpret_cast<const float2 *>(sw + e * 64 + c);
    const float2 bias = *reinterpret_cast<const float2 *>(sw + KS * KS * 64 + c);
    for (int k = lg; k < n_units; k += 2) {
      const int hs = k % g.nh, ot = k & 1;
      mbar_wait(&bars[kBarFh + hs], full_parity(k / g.nh));
      const uint8_t *hb = smem + g.off_h + hs * g.h_bytes;
      float2 acc[2][8];
#pragma unroll
      for (int dx = 0; dx < 2; ++dx)
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) acc[dx][rr] = bias;
      // halo rows yy, halo columns 2 xp .. 2 xp + KS: each value feeds both
      // output columns (taps w and w - 1) and up to KS output rows
      const uint8_t *col = hb + 2 * xp * 128 + c * 2;
#pragma unroll
      for (int yy = 0; yy < 8 + KS - 1; ++yy) {
        const uint8_t *rp = col + yy * (8 + KS - 1) * 128;
#pragma unroll
        for (int w = 0; w < KS + 1; ++w) {
          const uint32_t t2 = *reinterpret_cast<const uint32_t *>(rp + w * 128);
          const float2 vv = make_float2(__uint_as_float(t2 << 16),
                                        __uint_as_float(t2 & 0xffff0000u));
#pragma unroll
          for (int dx = 0; dx < 2; ++dx) {
            const int tw = w - dx;  // tap column for output column 2 xp + dx
            if (tw < 0 || tw >= KS) continue;
#pragma unroll
            for (int uu = 0; uu < KS; ++uu) {
              const int rr = yy - uu;
              if (rr >= 0 && rr < 8) acc[dx][rr] = __ffma2_rn(wgt[uu * KS + tw], vv, acc[dx][rr]);
            }
          }
        }
      }
      mbar_arrive(&bars[kBarHfree + hs]);  // the halo is no longer read
      // the LePE (f32) into the O tile, where the epilogue adds O
      mbar_wait(&bars[kBarOfree + ot], free_parity(k >> 1));
      float *otile = reinterpret_cast<float *>(smem + g.off_o + ot * 16384);
#pragma unroll
      for (int dx = 0; dx < 2; ++dx)
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          const int t = rr * 8 + 2 * xp + dx;
          *reinterpret_cast<float2 *>(otile + t * 64 + (((c >> 2) ^ (t & 7)) << 2) + (c & 3)) =
              acc[dx][rr];
        }
      mbar_arrive(&bars[kBarOfill + ot]);
    }
  }

  // ---- tear-down: every MMA has completed (warp 1 waited for that)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTcTmemCols);
  if (tid == 0) settle_after_timeout();
}

}  // namespace bra

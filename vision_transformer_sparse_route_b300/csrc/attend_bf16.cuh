// attend_bf16.cuh -- fused routed attention + LePE for bf16 maps on sm_103a.
//
// For one query region i of image b (a "unit"), with routing I = idx[b, i, :]:
//   out[t] = softmax_j(q_t . k_j * d^-1/2) v_j  over the keys j of the topk
//            routed regions jointly, per head,          (routed attention)
//          + bias + sum_{u,w} w[u, w] v[t + (u, w) - ks/2] (LePE, depthwise)
// (page "CVPR2023：BiFormer中的双层路由注意力机制解析" §3: k_g = gather(k, I_r),
// attn = softmax(q k_g^T * scale), out = attn v_g, out += lce(v); page
// "从静态到动态：BRA双层路由注意力如何革新视觉Transformer的计算范式" §4: LePE
// nn.Conv2d(dim, dim, ks, padding ks//2, groups=dim); page "BiFormer: Vision
// Transformer mit Bi-Level-Routing-Attention": attention over the union of the
// routed regions.)
//
// Persistent and warp-specialised: one CTA per SM walks the units
// blockIdx.x, blockIdx.x + gridDim.x, ... Warp 0 is the producer: one lane
// reads the routing index and issues TMA box copies for the unit's Q tile, the
// routed regions' K and V tiles (the gather lives only in shared memory;
// gathered K/V never exist in global memory) and the V halo (region plus
// ks/2 border; TMA's zero fill outside the image is the conv's zero padding)
// into a ring of pipeline stages, running up to `stages` units ahead.
// Warps 1..8 consume. Phase A: each warp owns 16 query rows of one head and
// runs mma.sync m16n8k16 (bf16 in, f32 accumulate) for S = Q K^T over 64 keys
// at a time, an online softmax in registers, and O += P V with P re-packed
// from the S accumulators; an extra MMA against a ones vector accumulates the
// row sums of the very bf16 P that multiplies V. Phase B: every thread computes
// the LePE of one column of one channel pair (a register block of up to 8
// rows, packed f32x2 FMAs, weights resident in registers), adds the
// normalised O, rounds to bf16 once and writes a staging tile that a TMA store
// sends out while the next unit is computed.
#pragma once

#include "ptx.cuh"

namespace bra {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kAttendThreads = 32 + kConsumerThreads;
constexpr int kMaxStages = 4;

struct AttendGeom {
  int H, W, C, S, heads, topk;
  int hr, wr, n, R;
  int nc;         // 64-channel chunks, C / 64
  int slot;       // key rows per routed region in K/V slots (n rounded to 8)
  int kv_rows;    // rows of one K or V chunk buffer (topk * slot rounded to 64)
  int q_blocks;   // 16-row query blocks per region
  int halo_w, halo_h;
  int units;      // B * S * S
  int stages;     // pipeline depth
  int masked;     // keys need masking (padded slots or a partial 64-key block)
  int lepe_items; // (C / 2) * wr * ceil(hr / RB)
  uint32_t q_chunk, kv_chunk, h_chunk, o_chunk;  // bytes per chunk buffer
  uint32_t off_k, off_v, off_h;  // within a stage
  uint32_t stage_bytes, tx_bytes;
  uint32_t off_out, off_o, off_w, off_bar;  // from the 1024-aligned base
  int o_stride;      // floats per row of the f32 O tile (C + 8)
  float scale_log2;  // d^-1/2 * log2(e)
};

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Waits for the grids this launch depends on (programmatic dependent launch);
// a no-op when launched without that attribute.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Waits until at most N committed bulk stores still read shared memory.
template <int N>
__device__ __forceinline__ void tma_store_wait_read_n() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// ----------------------------------------------------------------- phase A
// One attention task: 16 query rows (block qb) of head h for the unit whose
// tiles sit at q_base / k_base / v_base. Writes normalised O (f32) to so.
template <bool MASKED>
__device__ __forceinline__ void attention_task(const AttendGeom &g, int h,
                                               int qb, uint32_t q_base,
                                               uint32_t k_base, uint32_t v_base,
                                               float *so, int lane) {
  const int cb = (h & 1) * 4;  // first 16-byte column of the head in its chunk
  const int nslots = g.topk * g.slot;
  uint32_t qa[2][4];
#pragma unroll
  for (int ks = 0; ks < 2; ++ks)
    ldsm_x4(q_base + swz128(qb * 16 + (lane & 15), cb + ks * 2 + (lane >> 4)),
            qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);

  float o[4][4], l4[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    l4[a] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) o[a][e] = 0.f;
  }
  float m_run[2] = {-INFINITY, -INFINITY};
  const uint32_t ones = 0x3f803f80u;  // two bf16 1.0

  for (int kb = 0; kb < nslots; kb += 64) {
    float s[8][4];
#pragma unroll
    for (int jt = 0; jt < 8; ++jt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[jt][e] = 0.f;
      const int key0 = kb + jt * 8;
      if (!MASKED || key0 < nslots) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(k_base + swz128(key0 + (lane & 7), cb + (lane >> 3)), b0, b1, b2, b3);
        mma_bf16_16816(s[jt], qa[0], b0, b1);
        mma_bf16_16816(s[jt], qa[1], b2, b3);
      }
    }
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int jt = 0; jt < 8; ++jt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (MASKED) {
          const int key = kb + jt * 8 + 2 * (lane & 3) + (e & 1);
          if (key >= nslots || (key % g.slot) >= g.n) s[jt][e] = -INFINITY;
        }
        mx[e >> 1] = fmaxf(mx[e >> 1], s[jt][e]);
      }
    float base[2], alpha[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float m_new = fmaxf(m_run[r], mx[r] * g.scale_log2);
      base[r] = (m_new == -INFINITY) ? 0.f : m_new;
      alpha[r] = exp2f(m_run[r] - base[r]);
      m_run[r] = m_new;
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      o[a][0] *= alpha[0]; o[a][1] *= alpha[0];
      o[a][2] *= alpha[1]; o[a][3] *= alpha[1];
    }
    l4[0] *= alpha[0]; l4[1] *= alpha[0];
    l4[2] *= alpha[1]; l4[3] *= alpha[1];
    // P = exp2(S * scale - max), packed to bf16 for the P V product
    uint32_t p[8][2];
#pragma unroll
    for (int jt = 0; jt < 8; ++jt) {
      p[jt][0] = pack_bf16x2(exp2f(fmaf(s[jt][0], g.scale_log2, -base[0])),
                             exp2f(fmaf(s[jt][1], g.scale_log2, -base[0])));
      p[jt][1] = pack_bf16x2(exp2f(fmaf(s[jt][2], g.scale_log2, -base[1])),
                             exp2f(fmaf(s[jt][3], g.scale_log2, -base[1])));
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (!MASKED || kb + t * 16 < nslots) {
        const uint32_t pa[4] = {p[2 * t][0], p[2 * t][1], p[2 * t + 1][0],
                                p[2 * t + 1][1]};
        const int vrow = kb + t * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4_trans(v_base + swz128(vrow, cb + np * 2 + (lane >> 4)), r0, r1,
                        r2, r3);
          mma_bf16_16816(o[2 * np], pa, r0, r1);
          mma_bf16_16816(o[2 * np + 1], pa, r2, r3);
        }
        mma_bf16_16816(l4, pa, ones, ones);  // row sums of the bf16 P
      }
    }
  }
  const float inv0 = 1.f / l4[0], inv1 = 1.f / l4[2];
  const int row0 = qb * 16 + (lane >> 2);
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int ch = h * 32 + a * 8 + 2 * (lane & 3);
    if (row0 < g.n)
      *reinterpret_cast<float2 *>(so + row0 * g.o_stride + ch) =
          make_float2(o[a][0] * inv0, o[a][1] * inv0);
    if (row0 + 8 < g.n)
      *reinterpret_cast<float2 *>(so + (row0 + 8) * g.o_stride + ch) =
          make_float2(o[a][2] * inv1, o[a][3] * inv1);
  }
}

// ----------------------------------------------------------------- phase B
// LePE of rows ry0 .. ry0+RB-1, column x, channels c, c+1 of one unit, plus
// the attention output from so; bf16 result into the (unswizzled) staging
// tile ob. wgt holds the pair's KS*KS weights, bias the pair's bias.
template <int KS, int RB>
__device__ __forceinline__ void lepe_item(const AttendGeom &g, const uint8_t *hb,
                                          const float *so, uint8_t *ob, int c,
                                          int x, int ry0, const float2 (&wgt)[KS * KS],
                                          float2 bias) {
  const int cc = c >> 6, cw = (c & 63) * 2;
  float2 acc[RB];
#pragma unroll
  for (int r = 0; r < RB; ++r) acc[r] = bias;
  const uint8_t *col = hb + cc * g.h_chunk + ((size_t)ry0 * g.halo_w + x) * 128 + cw;
  const int row_step = g.halo_w * 128;
#pragma unroll
  for (int yy = 0; yy < RB + KS - 1; ++yy) {
    if (ry0 + yy < g.halo_h) {
      const uint8_t *rp = col + yy * row_step;
#pragma unroll
      for (int w = 0; w < KS; ++w) {
        const uint32_t t2 = *reinterpret_cast<const uint32_t *>(rp + w * 128);
        const float2 v = make_float2(bf16_lo(t2), bf16_hi(t2));
#pragma unroll
        for (int u = 0; u < KS; ++u) {
          const int r = yy - u;
          if (r >= 0 && r < RB) acc[r] = __ffma2_rn(wgt[u * KS + w], v, acc[r]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < RB; ++r) {
    const int row = ry0 + r;
    if (row < g.hr) {
      const int t = row * g.wr + x;
      const float2 ov = *reinterpret_cast<const float2 *>(so + t * g.o_stride + c);
      const float2 sum = __fadd2_rn(acc[r], ov);
      *reinterpret_cast<uint32_t *>(ob + cc * g.o_chunk + t * 128 + cw) =
          pack_bf16x2(sum.x, sum.y);
    }
  }
}

template <int KS>
__device__ __forceinline__ void load_pair_weights(const float *sw, int C, int c,
                                                  float2 (&wgt)[KS * KS],
                                                  float2 &bias) {
#pragma unroll
  for (int e = 0; e < KS * KS; ++e)
    wgt[e] = *reinterpret_cast<const float2 *>(sw + e * C + c);
  bias = *reinterpret_cast<const float2 *>(sw + KS * KS * C + c);
}

// ------------------------------------------------------------------ kernel
template <int KS, int RB>
__global__ void __launch_bounds__(kAttendThreads, 1)
    bra_attend_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_vh,
                           const __grid_constant__ CUtensorMap tm_o,
                           const int32_t *__restrict__ idx,
                           const float *__restrict__ lepe_w,
                           const float *__restrict__ lepe_b, AttendGeom g) {
  extern __shared__ uint8_t attend_smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(attend_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *stage0 = smem;                                 // [stages][stage_bytes]
  uint8_t *sout = smem + g.off_out;                       // [2][nc][n x 128 B]
  float *so = reinterpret_cast<float *>(smem + g.off_o);  // [n][o_stride]
  float *sw = reinterpret_cast<float *>(smem + g.off_w);  // [KS*KS][C], bias [C]
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + g.off_bar);
  uint64_t *empty = full + kMaxStages;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nslots = g.topk * g.slot;
  constexpr int PAD = KS / 2;

  if (tid == 0) {
    for (int s = 0; s < g.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
  }
  if (warp > 0) {
    const int ct = tid - 32;
    // LePE weights, tap-major so that a warp reads 32 consecutive channel pairs
    for (int e = ct; e < g.C * KS * KS; e += kConsumerThreads) {
      const int tap = e / g.C, c = e % g.C;
      sw[e] = __ldg(lepe_w + (size_t)c * KS * KS + tap);
    }
    for (int c = ct; c < g.C; c += kConsumerThreads)
      sw[KS * KS * g.C + c] = lepe_b ? __ldg(lepe_b + c) : 0.f;
    // Rows of the K/V slots that no copy writes (region slots padded to 8
    // rows, the buffer tail) hold zeros for the whole kernel: P is zero there
    // but 0 * NaN is not.
    if (g.masked) {
      for (int e = ct; e < g.stages * 2 * g.nc * g.kv_rows * 8; e += kConsumerThreads) {
        const int c16 = e & 7, row = (e >> 3) % g.kv_rows;
        const int buf = (e >> 3) / g.kv_rows;  // stage * 2nc + tensor * nc + chunk
        const int st = buf / (2 * g.nc), tb = buf % (2 * g.nc);
        if (row >= nslots || (row % g.slot) >= g.n) {
          uint8_t *base = stage0 + st * g.stage_bytes +
                          (tb < g.nc ? g.off_k : g.off_v) + (tb % g.nc) * g.kv_chunk;
          *reinterpret_cast<uint4 *>(base + row * 128 + c16 * 16) = make_uint4(0, 0, 0, 0);
        }
      }
    }
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      prefetch_tensormap(&tm_vh);
      grid_dependency_wait();  // the routing index comes from the previous grid
      int it = 0;
      for (int u = blockIdx.x; u < g.units; u += gridDim.x, ++it) {
        const int s = it % g.stages;
        if (it >= g.stages) mbar_wait(&empty[s], ((it / g.stages) - 1) & 1);
        uint8_t *st = stage0 + s * g.stage_bytes;
        const int b = u / g.R, i = u % g.R;
        const int y0 = (i / g.S) * g.hr, x0 = (i % g.S) * g.wr;
        mbar_arrive_expect_tx(&full[s], g.tx_bytes);
        for (int cc = 0; cc < g.nc; ++cc)
          tma_load_4d(st + cc * g.q_chunk, &tm_q, &full[s], cc * 64, x0, y0, b);
        const int32_t *ri = idx + (size_t)u * g.topk;
        for (int m = 0; m < g.topk; ++m) {
          const int j = __ldg(ri + m);
          int xj, yj;
          if (j < 0 || j >= g.R) {  // out of range: read zeros, flag it
            atomicOr(&g_status, kStatusBadIndex);
            xj = 0;
            yj = g.H;  // a box wholly below the image is all fill (zeros)
          } else {
            xj = (j % g.S) * g.wr;
            yj = (j / g.S) * g.hr;
          }
          for (int cc = 0; cc < g.nc; ++cc) {
            const uint32_t off = cc * g.kv_chunk + m * g.slot * 128u;
            tma_load_4d(st + g.off_k + off, &tm_k, &full[s], cc * 64, xj, yj, b);
            tma_load_4d(st + g.off_v + off, &tm_v, &full[s], cc * 64, xj, yj, b);
          }
        }
        for (int cc = 0; cc < g.nc; ++cc)
          tma_load_4d(st + g.off_h + cc * g.h_chunk, &tm_vh, &full[s], cc * 64,
                      x0 - PAD, y0 - PAD, b);
      }
    }
    return;
  }

  // --------------------------------------------------------- consumers
  const int ct = tid - 32, cw = warp - 1;
  const int pairs = g.C / 2;
  // with one LePE item per thread the pair is fixed: keep its weights resident
  const bool fixed_item = g.lepe_items == kConsumerThreads;
  float2 wgt[KS * KS], bias = make_float2(0.f, 0.f);
  if (fixed_item) load_pair_weights<KS>(sw, g.C, 2 * (ct % pairs), wgt, bias);

  int it = 0;
  for (int u = blockIdx.x; u < g.units; u += gridDim.x, ++it) {
    const int s = it % g.stages;
    mbar_wait(&full[s], (it / g.stages) & 1);
    const uint8_t *st = stage0 + s * g.stage_bytes;
    const int b = u / g.R, i = u % g.R;
    const int y0 = (i / g.S) * g.hr, x0 = (i % g.S) * g.wr;

    // phase A: attention
    for (int task = cw; task < g.heads * g.q_blocks; task += kConsumerWarps) {
      const int h = task % g.heads, qb = task / g.heads;
      const int cc = h >> 1;
      const uint32_t qb_ = smem_u32(st + cc * g.q_chunk);
      const uint32_t kb_ = smem_u32(st + g.off_k + cc * g.kv_chunk);
      const uint32_t vb_ = smem_u32(st + g.off_v + cc * g.kv_chunk);
      if (g.masked)
        attention_task<true>(g, h, qb, qb_, kb_, vb_, so, lane);
      else
        attention_task<false>(g, h, qb, qb_, kb_, vb_, so, lane);
    }
    consumer_sync();

    // phase B: LePE + O -> bf16 staging tile
    uint8_t *ob = sout + (it & 1) * (g.nc * g.o_chunk);
    const uint8_t *hb = st + g.off_h;
    for (int item = ct; item < g.lepe_items; item += kConsumerThreads) {
      const int cp = item % pairs, rest = item / pairs;
      const int x = rest % g.wr, ry0 = (rest / g.wr) * RB;
      if (!fixed_item) load_pair_weights<KS>(sw, g.C, 2 * cp, wgt, bias);
      lepe_item<KS, RB>(g, hb, so, ob, 2 * cp, x, ry0, wgt, bias);
    }
    fence_async_shared();
    consumer_sync();
    if (ct == 0) {
      mbar_arrive(&empty[s]);  // stage s fully read
      for (int cc = 0; cc < g.nc; ++cc)
        tma_store_4d(&tm_o, ob + cc * g.o_chunk, cc * 64, x0, y0, b);
      tma_store_commit();
      tma_store_wait_read_n<1>();  // the other staging buffer is free again
    }
  }
  if (ct == 0) tma_store_wait_read();
}

}  // namespace bra

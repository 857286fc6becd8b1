// attend_image.cuh -- routed attention + LePE for bf16 maps small enough that
// one 64-channel chunk of a whole image's q, k and v fits in shared memory
// (the stage-3 shape: 14 x 14 tokens, regions of 2 x 2).
//
// Same operation as attend_bf16.cuh (page "CVPR2023：BiFormer中的双层路由
// 注意力机制解析" §3; LePE of page "从静态到动态：BRA双层路由注意力如何革新
// 视觉Transformer的计算范式" §4), organised around the image instead of the
// query region: regions of a few tokens make per-region copies tiny (a 2 x 2
// region is 512 bytes per channel chunk), while the whole image chunk is a
// handful of large box copies.
//
// One CTA per (image, 64-channel chunk). Four TMA box copies bring the chunk
// of Q, K and V for the whole image (128-byte swizzled, one row per token)
// and the V halo (image plus ks/2 border, zero filled). The routed keys are
// gathered without copying: a key table names the image token of every key
// of every query region, and ldmatrix takes one row address per lane, so each
// lane points at the token it loads. For regions of at most 8 tokens each
// warp runs whole query regions (both heads of the chunk) in transposed form,
// keys as the MMA's rows and queries as its columns; larger regions run
// (query region, head, 16 query rows) tasks with the region kernel's
// mma.sync attention. O (f32) goes to shared memory, and every thread then
// computes the LePE of (channel pair, column, block of rows) items over the
// whole image, adds O and stores bf16 to the output.
#pragma once

#include "attend_bf16.cuh"

namespace bra {

constexpr int kImgWarps = 16;
constexpr int kImgThreads = 32 * kImgWarps;

struct ImageGeom {
  int H, W, C, S, heads, topk;
  int hr, wr, n, R;
  int nc;            // 64-channel chunks
  int nkeys;         // topk * n keys per query
  int nkp;           // nkeys rounded up to 64 (key table row length)
  int q_blocks;      // 16-row query blocks per region
  int halo_w, halo_h;
  uint32_t tile;     // bytes of one [H*W + 1][128 B] tile (the last row stays
                     // zero), rounded to 1024
  uint32_t off_k, off_v, off_h, off_o, off_w, off_tab, off_bar;
  float scale_log2;  // d^-1/2 * log2(e)
};

// Byte offset of 16-byte chunk `chunk` of token row `tok` in a swizzled tile.
__device__ __forceinline__ uint32_t tok_addr(int tok, int chunk) {
  return static_cast<uint32_t>(tok * 128 + ((chunk ^ (tok & 7)) << 4));
}

// One attention task: query rows qb*16 .. +15 of region i, head hl of the
// chunk. Leaves the normalised O rows (row0 = qb*16 + lane/4 and row0 + 8,
// channels hl*32 + a*8 + 2*(lane%4)) in o.
template <bool MASKED>
__device__ __forceinline__ void image_attention_task(const ImageGeom &g, int i, int hl,
                                                     int qb, uint32_t q_base,
                                                     uint32_t k_base, uint32_t v_base,
                                                     const uint16_t *kt, float (&o)[4][4],
                                                     int lane) {
  const int cb = hl * 4;  // first 16-byte chunk of the head in the 128-byte row
  const int y0 = (i / g.S) * g.hr, x0 = (i % g.S) * g.wr;
  uint32_t qa[2][4];
  {
    int r = qb * 16 + (lane & 15);
    r = r < g.n ? r : 0;  // rows past the region repeat its first token
    const int tok = (y0 + r / g.wr) * g.W + x0 + r % g.wr;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks)
      ldsm_x4(q_base + tok_addr(tok, cb + ks * 2 + (lane >> 4)), qa[ks][0], qa[ks][1],
              qa[ks][2], qa[ks][3]);
  }
  float l4[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    l4[a] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) o[a][e] = 0.f;
  }
  float m_run[2] = {-INFINITY, -INFINITY};
  const uint32_t ones = 0x3f803f80u;  // two bf16 1.0
  const float2 sc2 = make_float2(g.scale_log2, g.scale_log2);

  for (int kb = 0; kb < g.nkeys; kb += 64) {
    float s[8][4];
#pragma unroll
    for (int jt = 0; jt < 8; ++jt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[jt][e] = 0.f;
      const int tok = kt[kb + jt * 8 + (lane & 7)];
      uint32_t b0, b1, b2, b3;
      ldsm_x4(k_base + tok_addr(tok, cb + (lane >> 3)), b0, b1, b2, b3);
      mma_bf16_16816(s[jt], qa[0], b0, b1);
      mma_bf16_16816(s[jt], qa[1], b2, b3);
    }
    if (MASKED) {
#pragma unroll
      for (int jt = 0; jt < 8; ++jt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (kb + jt * 8 + 2 * (lane & 3) + (e & 1) >= g.nkeys) s[jt][e] = -INFINITY;
    }
    float mx[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float m = max3(s[0][2 * r], s[0][2 * r + 1], s[1][2 * r]);
      m = max3(m, s[1][2 * r + 1], s[2][2 * r]);
      m = max3(m, s[2][2 * r + 1], s[3][2 * r]);
      m = max3(m, s[3][2 * r + 1], s[4][2 * r]);
      m = max3(m, s[4][2 * r + 1], s[5][2 * r]);
      m = max3(m, s[5][2 * r + 1], s[6][2 * r]);
      m = max3(m, s[6][2 * r + 1], s[7][2 * r]);
      m = fmaxf(m, s[7][2 * r + 1]);
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      mx[r] = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    }
    float2 nb[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float m_new = fmaxf(m_run[r], mx[r] * g.scale_log2);
      const float base = (m_new == -INFINITY) ? 0.f : m_new;
      if (kb > 0) {
        const float alpha = exp2f(m_run[r] - base);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          o[a][2 * r] *= alpha;
          o[a][2 * r + 1] *= alpha;
        }
        l4[2 * r] *= alpha;
        l4[2 * r + 1] *= alpha;
      }
      m_run[r] = m_new;
      nb[r] = make_float2(-base, -base);
    }
    uint32_t p[8][2];
#pragma unroll
    for (int jt = 0; jt < 8; ++jt) {
      const float2 x0v = __ffma2_rn(make_float2(s[jt][0], s[jt][1]), sc2, nb[0]);
      const float2 x1v = __ffma2_rn(make_float2(s[jt][2], s[jt][3]), sc2, nb[1]);
      p[jt][0] = exp2_bf16x2(x0v.x, x0v.y);
      p[jt][1] = exp2_bf16x2(x1v.x, x1v.y);
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t pa[4] = {p[2 * t][0], p[2 * t][1], p[2 * t + 1][0], p[2 * t + 1][1]};
      const int tok = kt[kb + t * 16 + (lane & 7) + ((lane >> 3) & 1) * 8];
      uint32_t r0, r1, r2, r3;
      ldsm_x4_trans(v_base + tok_addr(tok, cb + (lane >> 4)), r0, r1, r2, r3);
      mma_bf16_16816(o[0], pa, r0, r1);
      mma_bf16_16816(o[1], pa, r2, r3);
      ldsm_x4_trans(v_base + tok_addr(tok, cb + 2 + (lane >> 4)), r0, r1, r2, r3);
      mma_bf16_16816(o[2], pa, r0, r1);
      mma_bf16_16816(o[3], pa, r2, r3);
      mma_bf16_16816(l4, pa, ones, ones);  // row sums of the bf16 P
    }
  }
  const float inv0 = 1.f / l4[0], inv1 = 1.f / l4[2];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    o[a][0] *= inv0; o[a][1] *= inv0;
    o[a][2] *= inv1; o[a][3] *= inv1;
  }
}

// The same attention in transposed form, for regions of at most 8 tokens,
// both heads of the chunk at once (two independent MMA chains for the warp;
// the key table lookups and token addresses are shared): the keys are the
// MMA's 16 rows and the region's queries its 8 columns, so that half of each
// MMA carries a query instead of a quarter. S^T = K Q^T; the softmax runs
// down each column (a lane holds 8 of a column's 64 keys, three shuffles
// combine them); movmatrix turns each 8x8 block of the bf16 P^T into the B
// operand of O^T = V^T P^T; the column sums are an MMA of ones against the
// same bf16 P^T. Leaves O^T of head h (channels h*32 + ct*16 + lane/4 and +8,
// queries 2*(lane%4) and +1) in ot[h][ct][0..3] = (ch, q0), (ch, q1),
// (ch+8, q0), (ch+8, q1).
template <bool MASKED>
__device__ __forceinline__ void image_attention_region_t(const ImageGeom &g, int i,
                                                         uint32_t q_base, uint32_t k_base,
                                                         uint32_t v_base, const uint16_t *kt,
                                                         float (&ot)[2][2][4], int lane) {
  const int y0 = (i / g.S) * g.hr, x0 = (i % g.S) * g.wr;
  // Q^T as the B operand: one 8x8 block (queries x 8 channels) per chunk
  uint32_t qb[2][2][2];
  {
    int r = lane & 7;
    r = r < g.n ? r : 0;  // columns past the region repeat its first token
    const int tok = (y0 + r / g.wr) * g.W + x0 + r % g.wr;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      ldsm_x4(q_base + tok_addr(tok, h * 4 + (lane >> 3)), qb[h][0][0], qb[h][0][1],
              qb[h][1][0], qb[h][1][1]);
  }
  float l4[2][4];
  float m_run[2][2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    m_run[h][0] = m_run[h][1] = -INFINITY;  // columns 2*(lane%4) and +1
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      l4[h][e] = 0.f;
      ot[h][0][e] = 0.f;
      ot[h][1][e] = 0.f;
    }
  }
  const uint32_t ones[4] = {0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u};
  const float2 sc2 = make_float2(g.scale_log2, g.scale_log2);
  const int kr = (lane & 7) + ((lane >> 3) & 1) * 8;  // K block row of this lane
  const int vr = (lane & 7) + (lane >> 4) * 8;        // V block row of this lane

  for (int kb = 0; kb < g.nkeys; kb += 64) {
    float s[2][4][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const int tok = kt[kb + mt * 16 + kr];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int e = 0; e < 4; ++e) s[h][mt][e] = 0.f;
        uint32_t a[4];
        ldsm_x4(k_base + tok_addr(tok, h * 4 + (lane >> 4)), a[0], a[1], a[2], a[3]);
        mma_bf16_16816(s[h][mt], a, qb[h][0][0], qb[h][0][1]);
        ldsm_x4(k_base + tok_addr(tok, h * 4 + 2 + (lane >> 4)), a[0], a[1], a[2], a[3]);
        mma_bf16_16816(s[h][mt], a, qb[h][1][0], qb[h][1][1]);
      }
    }
    if (MASKED) {
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (kb + mt * 16 + (lane >> 2) + (e >> 1) * 8 >= g.nkeys) s[h][mt][e] = -INFINITY;
    }
    float2 nb[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float m0 = max3(s[h][0][0], s[h][0][2], s[h][1][0]);
      m0 = max3(m0, s[h][1][2], s[h][2][0]);
      m0 = max3(m0, s[h][2][2], s[h][3][0]);
      m0 = fmaxf(m0, s[h][3][2]);
      float m1 = max3(s[h][0][1], s[h][0][3], s[h][1][1]);
      m1 = max3(m1, s[h][1][3], s[h][2][1]);
      m1 = max3(m1, s[h][2][3], s[h][3][1]);
      m1 = fmaxf(m1, s[h][3][3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, off));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, off));
      }
      const float mx[2] = {m0, m1};
      float base[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float m_new = fmaxf(m_run[h][q], mx[q] * g.scale_log2);
        base[q] = (m_new == -INFINITY) ? 0.f : m_new;
        if (kb > 0) {
          const float alpha = exp2f(m_run[h][q] - base[q]);
          ot[h][0][q] *= alpha;
          ot[h][0][q + 2] *= alpha;
          ot[h][1][q] *= alpha;
          ot[h][1][q + 2] *= alpha;
          l4[h][q] *= alpha;
          l4[h][q + 2] *= alpha;
        }
        m_run[h][q] = m_new;
      }
      nb[h] = make_float2(-base[0], -base[1]);
    }
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const int tok = kt[kb + mt * 16 + vr];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // bf16 P^T rows g (keys mt*16 + g) and g + 8, columns q0, q1;
        // transposed into the B fragments of keys 0-7 and 8-15 of this block
        const float2 xt = __ffma2_rn(make_float2(s[h][mt][0], s[h][mt][1]), sc2, nb[h]);
        const float2 xb = __ffma2_rn(make_float2(s[h][mt][2], s[h][mt][3]), sc2, nb[h]);
        const uint32_t pb0 = movmatrix_trans(exp2_bf16x2(xt.x, xt.y));
        const uint32_t pb1 = movmatrix_trans(exp2_bf16x2(xb.x, xb.y));
#pragma unroll
        for (int ct = 0; ct < 2; ++ct) {
          uint32_t a[4];
          ldsm_x4_trans(v_base + tok_addr(tok, h * 4 + ct * 2 + ((lane >> 3) & 1)), a[0], a[1],
                        a[2], a[3]);
          mma_bf16_16816(ot[h][ct], a, pb0, pb1);
        }
        mma_bf16_16816(l4[h], ones, pb0, pb1);  // column sums of the bf16 P^T
      }
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float inv0 = 1.f / l4[h][0], inv1 = 1.f / l4[h][1];
#pragma unroll
    for (int ct = 0; ct < 2; ++ct) {
      ot[h][ct][0] *= inv0; ot[h][ct][1] *= inv1;
      ot[h][ct][2] *= inv0; ot[h][ct][3] *= inv1;
    }
  }
}

// LePE of image rows ry0 .. ry0+RB-1, column x, chunk channels c, c+1, plus O
// from so ([H*W][64] f32, o_index layout), rounded to bf16 and stored to
// gout (the image's first token at this chunk's first channel).
template <int KS, int RB>
__device__ __forceinline__ void image_lepe_item(const ImageGeom &g, const uint8_t *hb,
                                                const float *so, __nv_bfloat16 *gout, int c,
                                                int x, int ry0, const float *sw) {
  float2 wgt[KS * KS];
#pragma unroll
  for (int e = 0; e < KS * KS; ++e) wgt[e] = *reinterpret_cast<const float2 *>(sw + e * 64 + c);
  const float2 bias = *reinterpret_cast<const float2 *>(sw + KS * KS * 64 + c);
  float2 acc[RB];
#pragma unroll
  for (int r = 0; r < RB; ++r) acc[r] = bias;
  const uint8_t *col = hb + (ry0 * g.halo_w + x) * 128 + c * 2;
#pragma unroll
  for (int yy = 0; yy < RB + KS - 1; ++yy) {
    if (ry0 + yy < g.halo_h) {
      const uint8_t *rp = col + yy * g.halo_w * 128;
#pragma unroll
      for (int w = 0; w < KS; ++w) {
        const uint32_t t2 = *reinterpret_cast<const uint32_t *>(rp + w * 128);
        const float2 v = make_float2(__uint_as_float(__byte_perm(t2, 0u, 0x1044u)),
                                     __uint_as_float(__byte_perm(t2, 0u, 0x3244u)));
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
    if (row < g.H) {
      const int t = row * g.W + x;
      const float2 ov = *reinterpret_cast<const float2 *>(so + o_index(64, t, c));
      const float2 sum = __fadd2_rn(acc[r], ov);
      *reinterpret_cast<uint32_t *>(gout + (size_t)t * g.C + c) = pack_bf16x2(sum.x, sum.y);
    }
  }
}

template <int KS, int RB>
__global__ void __launch_bounds__(kImgThreads, 1)
    bra_attend_image_kernel(const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_vh,
                            __nv_bfloat16 *__restrict__ out,
                            const int32_t *__restrict__ idx,
                            const float *__restrict__ lepe_w,
                            const float *__restrict__ lepe_b, ImageGeom g) {
  extern __shared__ uint8_t image_smem_raw[];
  uint8_t *smem = image_smem_raw + ((1024u - (smem_u32(image_smem_raw) & 1023u)) & 1023u);
  float *so = reinterpret_cast<float *>(smem + g.off_o);    // [H*W][64]
  float *sw = reinterpret_cast<float *>(smem + g.off_w);    // [KS*KS][64], bias [64]
  // key table: image token of key `key` of query region i at [i][key]
  uint16_t *ktab = reinterpret_cast<uint16_t *>(smem + g.off_tab);  // [R][nkp]
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + g.off_bar);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x / g.nc, cc = blockIdx.x % g.nc;
  constexpr int PAD = KS / 2;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, 3 * g.H * g.W * 128 + g.halo_w * g.halo_h * 128);
    tma_load_4d(smem, &tm_q, bar, cc * 64, 0, 0, b);
    tma_load_4d(smem + g.off_k, &tm_k, bar, cc * 64, 0, 0, b);
    tma_load_4d(smem + g.off_v, &tm_v, bar, cc * 64, 0, 0, b);
    tma_load_4d(smem + g.off_h, &tm_vh, bar, cc * 64, -PAD, -PAD, b);
  }
  // this chunk's LePE weights, read in their [c][tap] order (every load
  // issued before the first store), stored tap-major
  constexpr int NW = (64 * KS * KS + kImgThreads - 1) / kImgThreads;
  float wv[NW];
#pragma unroll
  for (int u = 0; u < NW; ++u) {
    const int e = tid + u * kImgThreads;
    wv[u] = e < 64 * KS * KS ? __ldg(lepe_w + (size_t)cc * 64 * KS * KS + e) : 0.f;
  }
  const float bv = (tid < 64 && lepe_b) ? __ldg(lepe_b + cc * 64 + tid) : 0.f;
  // the first routing entry of this thread (it comes from the previous grid),
  // loaded before the weights are stored so that the two loads overlap
  grid_dependency_wait();
  const int slots = g.R * g.topk;
  const int j0 = tid < slots ? __ldg(idx + (size_t)b * slots + tid) : 0;
#pragma unroll
  for (int u = 0; u < NW; ++u) {
    const int e = tid + u * kImgThreads;
    if (e < 64 * KS * KS) {
      const int c = e / (KS * KS), tap = e - c * (KS * KS);
      sw[tap * 64 + c] = wv[u];
    }
  }
  if (tid < 64) sw[KS * KS * 64 + tid] = bv;
  // the zero row of K and V (no copy writes it)
  if (tid < 16)
    *reinterpret_cast<uint4 *>(smem + (tid < 8 ? g.off_k : g.off_v) + g.H * g.W * 128 +
                               (tid & 7) * 16) = make_uint4(0, 0, 0, 0);
  // The key table, one (query region i, routed slot m) at a time: keys
  // m*n .. m*n+n-1 of region i are the tokens of routed region idx[b, i, m]
  // in row-major order. An out-of-range region's keys and the keys past nkeys
  // (masked) read the zero row after the image's tokens.
  const uint16_t zero_row = static_cast<uint16_t>(g.H * g.W);
  for (int e = tid; e < slots; e += kImgThreads) {
    const int i = e / g.topk, m = e - i * g.topk;
    const int j = e == tid ? j0 : __ldg(idx + (size_t)b * slots + e);
    uint16_t *row = ktab + i * g.nkp + m * g.n;
    if (j < 0 || j >= g.R) {  // out of range: flag it
      atomicOr(&g_status, kStatusBadIndex);
      for (int t = 0; t < g.n; ++t) row[t] = zero_row;
    } else {
      const int y0 = (j / g.S) * g.hr, x0 = (j % g.S) * g.wr;
      for (int ty = 0; ty < g.hr; ++ty)
        for (int tx = 0; tx < g.wr; ++tx)
          row[ty * g.wr + tx] = static_cast<uint16_t>((y0 + ty) * g.W + x0 + tx);
    }
  }
  const int tail = g.nkp - g.nkeys;
  for (int e = tid; e < g.R * tail; e += kImgThreads) {
    const int i = e / tail;
    ktab[i * g.nkp + g.nkeys + (e - i * tail)] = zero_row;
  }
  __syncthreads();
  mbar_wait(bar, 0);

  // ---- attention: (query region, head of the chunk, query block) tasks
  const uint32_t q_base = smem_u32(smem), k_base = smem_u32(smem + g.off_k),
                 v_base = smem_u32(smem + g.off_v);
  if (g.n <= 8) {
    // transposed form, one region (both heads of the chunk) per task
    for (int i = warp; i < g.R; i += kImgWarps) {
      float ot[2][2][4];
      if (g.nkeys % 64)
        image_attention_region_t<true>(g, i, q_base, k_base, v_base, ktab + i * g.nkp, ot, lane);
      else
        image_attention_region_t<false>(g, i, q_base, k_base, v_base, ktab + i * g.nkp, ot,
                                        lane);
      const int y0 = (i / g.S) * g.hr, x0 = (i % g.S) * g.wr;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = 2 * (lane & 3) + e;  // query of column e
        if (r < g.n) {
          const int tok = (y0 + r / g.wr) * g.W + x0 + r % g.wr;
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int ct = 0; ct < 2; ++ct)
#pragma unroll
              for (int half = 0; half < 2; ++half)
                so[o_index(64, tok, h * 32 + ct * 16 + half * 8 + (lane >> 2))] =
                    ot[h][ct][2 * half + e];
        }
      }
    }
  }
  const int tasks = g.n <= 8 ? 0 : g.R * 2 * g.q_blocks;
  for (int task = warp; task < tasks; task += kImgWarps) {
    const int i = task / (2 * g.q_blocks), rest = task % (2 * g.q_blocks);
    const int hl = rest % 2, qb = rest / 2;
    const int y0 = (i / g.S) * g.hr, x0 = (i % g.S) * g.wr;
    float o[4][4];
    if (g.nkeys % 64)
      image_attention_task<true>(g, i, hl, qb, q_base, k_base, v_base, ktab + i * g.nkp, o,
                                 lane);
    else
      image_attention_task<false>(g, i, hl, qb, q_base, k_base, v_base, ktab + i * g.nkp, o,
                                  lane);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = qb * 16 + (lane >> 2) + half * 8;
      if (r < g.n) {
        const int tok = (y0 + r / g.wr) * g.W + x0 + r % g.wr;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const int ch = hl * 32 + a * 8 + 2 * (lane & 3);
          *reinterpret_cast<float2 *>(so + o_index(64, tok, ch)) =
              make_float2(o[a][2 * half], o[a][2 * half + 1]);
        }
      }
    }
  }
  __syncthreads();

  // ---- LePE + O -> bf16 output
  __nv_bfloat16 *gout = out + (size_t)b * g.H * g.W * g.C + cc * 64;
  const uint8_t *hb = smem + g.off_h;
  const int rblocks = (g.H + RB - 1) / RB;
  for (int item = tid; item < 32 * g.W * rblocks; item += kImgThreads) {
    const int cp = item % 32, rest = item / 32;
    const int x = rest % g.W, ry0 = (rest / g.W) * RB;
    image_lepe_item<KS, RB>(g, hb, so, gout, 2 * cp, x, ry0, sw);
  }
  if (tid == 0) settle_after_timeout();
}

}  // namespace bra

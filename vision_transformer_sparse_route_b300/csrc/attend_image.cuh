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
  uint32_t off_rt;   // local form: region and token offset tables
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
// NH heads of the chunk from head h0 on at once (NH = 2: two independent MMA
// chains for the warp, sharing the key table lookups and token addresses;
// NH = 1 keeps the registers under 64): the keys are the
// MMA's 16 rows and the region's queries its 8 columns, so that half of each
// MMA carries a query instead of a quarter. S^T = K Q^T; the softmax runs
// down each column (a lane holds 8 of a column's 64 keys, three shuffles
// combine them); movmatrix turns each 8x8 block of the bf16 P^T into the B
// operand of O^T = V^T P^T; the column sums are an MMA of ones against the
// same bf16 P^T. Leaves O^T of head h0 + h (channels (h0+h)*32 + ct*16 +
// lane/4 and +8, queries 2*(lane%4) and +1) in ot[h][ct][0..3] = (ch, q0),
// (ch, q1), (ch+8, q0), (ch+8, q1).
template <bool MASKED, int NH = 2>
__device__ __forceinline__ void image_attention_region_t(const ImageGeom &g, int i,
                                                         uint32_t q_base, uint32_t k_base,
                                                         uint32_t v_base, const uint16_t *kt,
                                                         float (&ot)[NH][2][4], int lane,
                                                         int h0 = 0) {
  const int y0 = (i / g.S) * g.hr, x0 = (i % g.S) * g.wr;
  // Q^T as the B operand: one 8x8 block (queries x 8 channels) per chunk
  uint32_t qb[NH][2][2];
  {
    int r = lane & 7;
    r = r < g.n ? r : 0;  // columns past the region repeat its first token
    const int tok = (y0 + r / g.wr) * g.W + x0 + r % g.wr;
#pragma unroll
    for (int h = 0; h < NH; ++h)
      ldsm_x4(q_base + tok_addr(tok, (h0 + h) * 4 + (lane >> 3)), qb[h][0][0], qb[h][0][1],
              qb[h][1][0], qb[h][1][1]);
  }
  float l4[NH][4];
  float m_run[NH][2];
#pragma unroll
  for (int h = 0; h < NH; ++h) {
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
    float s[NH][4][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const int tok = kt[kb + mt * 16 + kr];
#pragma unroll
      for (int h = 0; h < NH; ++h) {
#pragma unroll
        for (int e = 0; e < 4; ++e) s[h][mt][e] = 0.f;
        uint32_t a[4];
        ldsm_x4(k_base + tok_addr(tok, (h0 + h) * 4 + (lane >> 4)), a[0], a[1], a[2], a[3]);
        mma_bf16_16816(s[h][mt], a, qb[h][0][0], qb[h][0][1]);
        ldsm_x4(k_base + tok_addr(tok, (h0 + h) * 4 + 2 + (lane >> 4)), a[0], a[1], a[2], a[3]);
        mma_bf16_16816(s[h][mt], a, qb[h][1][0], qb[h][1][1]);
      }
    }
    if (MASKED) {
#pragma unroll
      for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (kb + mt * 16 + (lane >> 2) + (e >> 1) * 8 >= g.nkeys) s[h][mt][e] = -INFINITY;
    }
    float2 nb[NH];
#pragma unroll
    for (int h = 0; h < NH; ++h) {
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
      for (int h = 0; h < NH; ++h) {
        // bf16 P^T rows g (keys mt*16 + g) and g + 8, columns q0, q1;
        // transposed into the B fragments of keys 0-7 and 8-15 of this block
        const float2 xt = __ffma2_rn(make_float2(s[h][mt][0], s[h][mt][1]), sc2, nb[h]);
        const float2 xb = __ffma2_rn(make_float2(s[h][mt][2], s[h][mt][3]), sc2, nb[h]);
        const uint32_t pb0 = movmatrix_trans(exp2_bf16x2(xt.x, xt.y));
        const uint32_t pb1 = movmatrix_trans(exp2_bf16x2(xb.x, xb.y));
#pragma unroll
        for (int ct = 0; ct < 2; ++ct) {
          uint32_t a[4];
          ldsm_x4_trans(v_base + tok_addr(tok, (h0 + h) * 4 + ct * 2 + ((lane >> 3) & 1)), a[0],
                        a[1], a[2], a[3]);
          mma_bf16_16816(ot[h][ct], a, pb0, pb1);
        }
        mma_bf16_16816(l4[h], ones, pb0, pb1);  // column sums of the bf16 P^T
      }
    }
  }
#pragma unroll
  for (int h = 0; h < NH; ++h) {
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

// The chunk's LePE weights, all threads: read in their [c][tap] order (every
// load issued before the first store), stored tap-major with the bias after
// them. sync_before_store runs between the loads and the stores (it lets the
// weight loads overlap a wait for the previous grid).
template <int KS, int NT, typename F>
__device__ __forceinline__ void image_weights(float *sw, const float *__restrict__ lepe_w,
                                              const float *__restrict__ lepe_b, int cc, int tid,
                                              F sync_before_store) {
  constexpr int NW = (64 * KS * KS + NT - 1) / NT;
  float wv[NW];
#pragma unroll
  for (int u = 0; u < NW; ++u) {
    const int e = tid + u * NT;
    wv[u] = e < 64 * KS * KS ? __ldg(lepe_w + (size_t)cc * 64 * KS * KS + e) : 0.f;
  }
  const float bv = (tid < 64 && lepe_b) ? __ldg(lepe_b + cc * 64 + tid) : 0.f;
  sync_before_store();
#pragma unroll
  for (int u = 0; u < NW; ++u) {
    const int e = tid + u * NT;
    if (e < 64 * KS * KS) {
      const int c = e / (KS * KS), tap = e - c * (KS * KS);
      sw[tap * 64 + c] = wv[u];
    }
  }
  if (tid < 64) sw[KS * KS * 64 + tid] = bv;
}

// The key tables of an image from its routing rt ([R][topk]; global memory
// written by an earlier grid, read through the read-only path, or, with
// FROM_SMEM, this CTA's shared copy), all threads: keys m*n .. m*n+n-1 of
// query region i are the tokens of routed region rt[i][m] in row-major
// order, as image token numbers in ktab and, when vtab is given, as positions
// in the V halo tile (image plus a border of ks/2, halo_w wide) in vtab. An
// out-of-range region's keys and the keys past nkeys (masked) name the zero
// row after the image's tokens (the zero row after the halo in vtab).
// The thread's first routing entries (up to four), loaded together.
template <int NT, bool FROM_SMEM>
__device__ __forceinline__ void prefetch_routing(const ImageGeom &g, const int32_t *rt, int tid,
                                                 int (&jpre)[4]) {
  const int slots = g.R * g.topk;
#pragma unroll
  for (int u = 0; u < 4; ++u)
    jpre[u] = tid + u * NT < slots ? (FROM_SMEM ? rt[tid + u * NT] : __ldg(rt + tid + u * NT))
                                   : 0;
}

template <int KS, int NT, bool FROM_SMEM>
__device__ __forceinline__ void image_key_tables(const ImageGeom &g, uint16_t *ktab,
                                                 uint16_t *vtab, const int32_t *rt,
                                                 const int (&jpre)[4], int tid) {
  constexpr int PAD = KS / 2;
  const int slots = g.R * g.topk;
  const uint16_t zero_row = static_cast<uint16_t>(g.H * g.W);
  const uint16_t zero_pos = static_cast<uint16_t>(g.halo_w * g.halo_h);
  for (int e = tid, u = 0; e < slots; e += NT, ++u) {
    const int i = e / g.topk, m = e - i * g.topk;
    int j = jpre[0];
#pragma unroll
    for (int v = 1; v < 4; ++v) j = u == v ? jpre[v] : j;
    if (u >= 4) j = FROM_SMEM ? rt[e] : __ldg(rt + e);
    uint16_t *row = ktab + i * g.nkp + m * g.n;
    uint16_t *vrow = vtab ? vtab + i * g.nkp + m * g.n : nullptr;
    if (j < 0 || j >= g.R) {  // out of range: flag it
      atomicOr(&g_status, kStatusBadIndex);
      for (int t = 0; t < g.n; ++t) {
        row[t] = zero_row;
        if (vrow) vrow[t] = zero_pos;
      }
    } else {
      const int y0 = (j / g.S) * g.hr, x0 = (j % g.S) * g.wr;
      for (int ty = 0; ty < g.hr; ++ty)
        for (int tx = 0; tx < g.wr; ++tx) {
          row[ty * g.wr + tx] = static_cast<uint16_t>((y0 + ty) * g.W + x0 + tx);
          if (vrow)
            vrow[ty * g.wr + tx] =
                static_cast<uint16_t>((y0 + ty + PAD) * g.halo_w + x0 + tx + PAD);
        }
    }
  }
  const int tail = g.nkp - g.nkeys;
  for (int e = tid; e < g.R * tail; e += NT) {
    const int i = e / tail, key = g.nkeys + (e - i * tail);
    ktab[i * g.nkp + key] = zero_row;
    if (vtab) vtab[i * g.nkp + key] = zero_pos;
  }
}

// Weights and key tables of the attend kernels (routing from the previous
// grid; the weight loads overlap the wait for it).
template <int KS, int NT = kImgThreads>
__device__ __forceinline__ void image_tables(const ImageGeom &g, float *sw, uint16_t *ktab,
                                             uint16_t *vtab, const int32_t *__restrict__ idx,
                                             const float *__restrict__ lepe_w,
                                             const float *__restrict__ lepe_b, int b, int cc,
                                             int tid) {
  const int32_t *rt = idx + (size_t)b * g.R * g.topk;
  int jpre[4];
  image_weights<KS, NT>(sw, lepe_w, lepe_b, cc, tid, [&] {
    grid_dependency_wait();
    prefetch_routing<NT, false>(g, rt, tid, jpre);
  });
  image_key_tables<KS, NT, false>(g, ktab, vtab, rt, jpre, tid);
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
  // the zero row of K and V (no copy writes it)
  if (tid < 16)
    *reinterpret_cast<uint4 *>(smem + (tid < 8 ? g.off_k : g.off_v) + g.H * g.W * 128 +
                               (tid & 7) * 16) = make_uint4(0, 0, 0, 0);
  image_tables<KS>(g, sw, ktab, nullptr, idx, lepe_w, lepe_b, b, cc, tid);
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

// ---- the local form, regions of at most 8 tokens: about half the shared
// memory of the form above, so that two CTAs share an SM. K is the swizzled
// tile as above; V is a zero-bordered halo tile (image plus ks/2 on every
// side) with 144-byte rows (the 64 channels of the chunk and 16 unused
// bytes; the odd 16-byte pitch keeps ldmatrix free of bank conflicts as the
// swizzle does); Q is read by each task from global memory straight into its
// MMA fragment, and there is no f32 O tile. Each warp runs (query region,
// head) tasks; after a task's attention the warp computes the LePE of the
// region's tokens over the head's 32 channels from the halo tile, adds the
// task's O and stores bf16.

constexpr int kStgStride = 68;  // floats a staged O row (64 channels + pad)
constexpr int kLocalWarps = 8;
constexpr int kLocalThreads = 32 * kLocalWarps;
constexpr int kHaloPitch = 144;  // bytes a V halo row

// O^T of a region's NH heads from head h0 on (t0: the region's first image
// token, toff: each token's offset from it), as image_attention_region_t,
// with Q taken from global memory (qg: the image's first token at the
// chunk's first channel) and V from the halo tile through the halo-position
// key table vt.
template <bool MASKED, int NH>
__device__ __forceinline__ void local_attention(const ImageGeom &g, int t0, const uint16_t *toff,
                                                int h0, const __nv_bfloat16 *qg,
                                                uint32_t k_base, uint32_t vh_base,
                                                const uint16_t *kt, const uint16_t *vt,
                                                float (&ot)[NH][2][4], int lane) {
  // Q^T as the B operand: lane holds query lane/4 (queries past the region
  // repeat its first token), channels kb*16 + 2*(lane%4) + {0, 1} and + 8
  uint32_t qb[NH][2][2];
  {
    const int r = lane >> 2;
    const int tok = t0 + (r < g.n ? toff[r] : 0);
    const uint32_t *qp = reinterpret_cast<const uint32_t *>(qg + (size_t)tok * g.C) +
                         (lane & 3);
#pragma unroll
    for (int h = 0; h < NH; ++h)
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
        qb[h][kb][0] = __ldg(qp + (h0 + h) * 16 + kb * 8);
        qb[h][kb][1] = __ldg(qp + (h0 + h) * 16 + kb * 8 + 4);
      }
  }
  float l4[NH][4], m_run[NH][2];
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    m_run[h][0] = m_run[h][1] = -INFINITY;
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
    float s[NH][4][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const int tok = kt[kb + mt * 16 + kr];
#pragma unroll
      for (int h = 0; h < NH; ++h) {
#pragma unroll
        for (int e = 0; e < 4; ++e) s[h][mt][e] = 0.f;
        uint32_t a[4];
        ldsm_x4(k_base + tok_addr(tok, (h0 + h) * 4 + (lane >> 4)), a[0], a[1], a[2], a[3]);
        mma_bf16_16816(s[h][mt], a, qb[h][0][0], qb[h][0][1]);
        ldsm_x4(k_base + tok_addr(tok, (h0 + h) * 4 + 2 + (lane >> 4)), a[0], a[1], a[2], a[3]);
        mma_bf16_16816(s[h][mt], a, qb[h][1][0], qb[h][1][1]);
      }
    }
    if (MASKED) {
#pragma unroll
      for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (kb + mt * 16 + (lane >> 2) + (e >> 1) * 8 >= g.nkeys) s[h][mt][e] = -INFINITY;
    }
    float2 nb[NH];
#pragma unroll
    for (int h = 0; h < NH; ++h) {
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
      const uint32_t vrow = vh_base + vt[kb + mt * 16 + vr] * kHaloPitch;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const float2 xt = __ffma2_rn(make_float2(s[h][mt][0], s[h][mt][1]), sc2, nb[h]);
        const float2 xb = __ffma2_rn(make_float2(s[h][mt][2], s[h][mt][3]), sc2, nb[h]);
        const uint32_t pb0 = movmatrix_trans(exp2_bf16x2(xt.x, xt.y));
        const uint32_t pb1 = movmatrix_trans(exp2_bf16x2(xb.x, xb.y));
#pragma unroll
        for (int ct = 0; ct < 2; ++ct) {
          uint32_t a[4];
          ldsm_x4_trans(vrow + ((h0 + h) * 4 + ct * 2 + ((lane >> 3) & 1)) * 16, a[0], a[1],
                        a[2], a[3]);
          mma_bf16_16816(ot[h][ct], a, pb0, pb1);
        }
        mma_bf16_16816(l4[h], ones, pb0, pb1);  // column sums of the bf16 P^T
      }
    }
  }
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    const float inv0 = 1.f / l4[h][0], inv1 = 1.f / l4[h][1];
#pragma unroll
    for (int ct = 0; ct < 2; ++ct) {
      ot[h][ct][0] *= inv0; ot[h][ct][1] *= inv1;
      ot[h][ct][2] *= inv0; ot[h][ct][3] *= inv1;
    }
  }
}

// LePE + O of a region over the chunk's 64 channels: t0 and h0 are the
// region's first image token and the halo position of that token's top-left
// tap, toff and hoff each token's offset from them; ot is the region's O^T
// fragment (both heads), stg the warp's staging rows ([n][kStgStride] f32),
// vh the halo tile, sw the chunk's weights (tap-major, bias after them),
// gout the image's first token at the chunk's first channel. Lane l takes
// channels 2l, 2l+1 of every token of the region, its 25 weights in
// registers and one 4-byte load of V a tap (the warp reads 128 contiguous
// bytes). Each output is bias, then the taps in row-major order, then O,
// rounded once; the halo's zero border stands for the padding. With the
// region's shape HR x WR fixed at compile time the lane slides over the
// region's window ((HR + KS - 1) x (WR + KS - 1) loads, each feeding every
// output whose kernel covers it, in the same tap order); with HR = 0 it takes
// the tokens one by one.
template <int KS, int HR, int WR>
__device__ __forceinline__ void local_lepe(const ImageGeom &g, int t0, int h0,
                                           const uint16_t *toff, const uint16_t *hoff,
                                           const float (&ot)[2][2][4], float *stg,
                                           const uint8_t *vh, const float *sw,
                                           __nv_bfloat16 *gout, int lane) {
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int q = 2 * (lane & 3) + e;
    if (q < g.n) {
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int ct = 0; ct < 2; ++ct)
#pragma unroll
          for (int half = 0; half < 2; ++half)
            stg[q * kStgStride + h * 32 + ct * 16 + half * 8 + (lane >> 2)] =
                ot[h][ct][2 * half + e];
    }
  }
  const int c = 2 * lane;
  float2 wgt[KS * KS];
#pragma unroll
  for (int e = 0; e < KS * KS; ++e) wgt[e] = *reinterpret_cast<const float2 *>(sw + e * 64 + c);
  const float2 bias = *reinterpret_cast<const float2 *>(sw + KS * KS * 64 + c);
  const uint32_t row_bytes = g.halo_w * kHaloPitch;
  __syncwarp();
  if constexpr (HR > 0) {
    float2 acc[HR][WR];
#pragma unroll
    for (int ty = 0; ty < HR; ++ty)
#pragma unroll
      for (int tx = 0; tx < WR; ++tx) acc[ty][tx] = bias;
    const uint8_t *tap0 = vh + h0 * kHaloPitch + 2 * c;
#pragma unroll
    for (int yy = 0; yy < HR + KS - 1; ++yy) {
      const uint8_t *row = tap0 + yy * row_bytes;
#pragma unroll
      for (int xx = 0; xx < WR + KS - 1; ++xx) {
        const uint32_t t2 = *reinterpret_cast<const uint32_t *>(row + xx * kHaloPitch);
        const float2 v =
            make_float2(__uint_as_float(t2 << 16), __uint_as_float(t2 & 0xffff0000u));
#pragma unroll
        for (int ty = 0; ty < HR; ++ty)
#pragma unroll
          for (int tx = 0; tx < WR; ++tx) {
            const int u = yy - ty, w = xx - tx;
            if (u >= 0 && u < KS && w >= 0 && w < KS)
              acc[ty][tx] = __ffma2_rn(wgt[u * KS + w], v, acc[ty][tx]);
          }
      }
    }
#pragma unroll
    for (int ty = 0; ty < HR; ++ty)
#pragma unroll
      for (int tx = 0; tx < WR; ++tx) {
        const float2 ov =
            *reinterpret_cast<const float2 *>(stg + (ty * WR + tx) * kStgStride + c);
        const float2 sum = __fadd2_rn(acc[ty][tx], ov);
        *reinterpret_cast<uint32_t *>(gout + (size_t)(t0 + ty * g.W + tx) * g.C + c) =
            pack_bf16x2(sum.x, sum.y);
      }
  } else {
    for (int r = 0; r < g.n; ++r) {
      const uint8_t *tap0 = vh + (h0 + hoff[r]) * kHaloPitch + 2 * c;
      float2 acc = bias;
#pragma unroll
      for (int u = 0; u < KS; ++u) {
        const uint8_t *row = tap0 + u * row_bytes;
#pragma unroll
        for (int w = 0; w < KS; ++w) {
          const uint32_t t2 = *reinterpret_cast<const uint32_t *>(row + w * kHaloPitch);
          acc = __ffma2_rn(
              wgt[u * KS + w],
              make_float2(__uint_as_float(t2 << 16), __uint_as_float(t2 & 0xffff0000u)), acc);
        }
      }
      const float2 ov = *reinterpret_cast<const float2 *>(stg + r * kStgStride + c);
      const float2 sum = __fadd2_rn(acc, ov);
      *reinterpret_cast<uint32_t *>(gout + (size_t)(t0 + toff[r]) * g.C + c) =
          pack_bf16x2(sum.x, sum.y);
    }
  }
  __syncwarp();
}

template <int KS, int HR, int WR>
__global__ void __launch_bounds__(kLocalThreads, 2)
    bra_attend_image_local_kernel(const __grid_constant__ CUtensorMap tm_k,
                                  const __grid_constant__ CUtensorMap tm_vh,
                                  const __nv_bfloat16 *__restrict__ q,
                                  __nv_bfloat16 *__restrict__ out,
                                  const int32_t *__restrict__ idx,
                                  const float *__restrict__ lepe_w,
                                  const float *__restrict__ lepe_b, ImageGeom g) {
  extern __shared__ uint8_t image_smem_raw[];
  uint8_t *smem = image_smem_raw + ((1024u - (smem_u32(image_smem_raw) & 1023u)) & 1023u);
  float *sw = reinterpret_cast<float *>(smem + g.off_w);
  uint16_t *ktab = reinterpret_cast<uint16_t *>(smem + g.off_tab);
  uint16_t *vtab = reinterpret_cast<uint16_t *>(smem + g.off_v);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + g.off_bar);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x / g.nc, cc = blockIdx.x % g.nc;
  constexpr int PAD = KS / 2;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, g.H * g.W * 128 + g.halo_w * g.halo_h * kHaloPitch);
    tma_load_4d(smem + g.off_k, &tm_k, bar, cc * 64, 0, 0, b);
    tma_load_4d(smem + g.off_h, &tm_vh, bar, cc * 64, -PAD, -PAD, b);
  }
  // the zero rows after the K tile and after the halo (no copy writes them)
  if (tid < 8)
    *reinterpret_cast<uint4 *>(smem + g.off_k + g.H * g.W * 128 + tid * 16) =
        make_uint4(0, 0, 0, 0);
  else if (tid < 17)
    *reinterpret_cast<uint4 *>(smem + g.off_h + g.halo_w * g.halo_h * kHaloPitch +
                               (tid - 8) * 16) = make_uint4(0, 0, 0, 0);
  image_tables<KS, kLocalThreads>(g, sw, ktab, vtab, idx, lepe_w, lepe_b, b, cc, tid);
  // region tables: first image token and the halo position of its top-left
  // tap ([R][2]); token offsets within a region, image and halo ([n][2])
  uint16_t *rt = reinterpret_cast<uint16_t *>(smem + g.off_rt);
  uint16_t *ot_tab = rt + 2 * g.R;
  for (int e = tid; e < g.R + g.n; e += kLocalThreads) {
    if (e < g.R) {
      const int y0 = (e / g.S) * g.hr, x0 = (e % g.S) * g.wr;
      rt[2 * e] = static_cast<uint16_t>(y0 * g.W + x0);
      rt[2 * e + 1] = static_cast<uint16_t>(y0 * g.halo_w + x0);
    } else {
      const int r = e - g.R, dy = r / g.wr, dx = r % g.wr;
      ot_tab[r] = static_cast<uint16_t>(dy * g.W + dx);
      ot_tab[8 + r] = static_cast<uint16_t>(dy * g.halo_w + dx);
    }
  }
  __syncthreads();
  mbar_wait(bar, 0);

  const uint32_t k_base = smem_u32(smem + g.off_k), vh_base = smem_u32(smem + g.off_h);
  float *stg = reinterpret_cast<float *>(smem + g.off_o) + warp * g.n * kStgStride;
  const size_t img = (size_t)b * g.H * g.W * g.C + cc * 64;
  for (int i = warp; i < g.R; i += kLocalWarps) {
    const int t0 = rt[2 * i], h0 = rt[2 * i + 1];
    float ot[2][2][4];
    if (g.nkeys % 64)
      local_attention<true, 2>(g, t0, ot_tab, 0, q + img, k_base, vh_base, ktab + i * g.nkp,
                               vtab + i * g.nkp, ot, lane);
    else
      local_attention<false, 2>(g, t0, ot_tab, 0, q + img, k_base, vh_base, ktab + i * g.nkp,
                                vtab + i * g.nkp, ot, lane);
    local_lepe<KS, HR, WR>(g, t0, h0, ot_tab, ot_tab + 8, ot, stg, smem + g.off_h, sw,
                           out + img, lane);
  }
  if (tid == 0) settle_after_timeout();
}

}  // namespace bra

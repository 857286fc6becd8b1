// attend_bf16.cuh -- fused routed attention + LePE for bf16 maps on sm_103a.
//
// For one query region i of image b (one CTA), with routing I = idx[b, i, :]:
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
// The gathered K/V never exist in global memory: thread 0 reads the routing
// index and issues one TMA box copy per routed region and 64-channel chunk,
// straight into 128-byte-swizzled shared-memory slots. The region's Q tile and
// its V halo (region plus ks/2 border; the TMA zero fill outside the image is
// the conv's zero padding) arrive the same way. Eight warps then run the
// attention with mma.sync m16n8k16 (bf16 in, f32 accumulate): each warp owns
// 16 query rows of one head, computes S = Q K^T for 64 keys at a time,
// keeps an online softmax (running max and sum) in registers and accumulates
// O += P V with P re-packed from the S accumulators. The normalised O goes
// to shared memory as f32; every thread then computes the LePE of a column
// of its channel pair from the V halo, adds O, rounds to bf16 once and writes
// the tile back in swizzled order, and one TMA store writes it out.
#pragma once

#include "ptx.cuh"

namespace bra {

constexpr int kAttendThreads = 256;
constexpr int kLepeRows = 4;  // output rows per LePE register block

struct AttendGeom {
  int H, W, C, S, heads, topk;
  int hr, wr, n, R;
  int nc;         // 64-channel chunks, C / 64
  int slot;       // key rows per routed region in K/V slots (n rounded to 8)
  int kv_rows;    // rows of one K or V chunk buffer (topk * slot rounded to 64)
  int q_blocks;   // 16-row query blocks per region
  int halo_w, halo_h;
  uint32_t q_chunk, kv_chunk, h_chunk;  // bytes per chunk buffer
  uint32_t off_k, off_v, off_h, off_o, off_bar;  // from the 1024-aligned base
  int o_stride;   // floats per row of the f32 O tile (C + 8)
  float scale_log2;  // d^-1/2 * log2(e)
};

template <int KS>
__global__ void __launch_bounds__(kAttendThreads)
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
  uint8_t *sq = smem;              // [nc][q_rows x 128 B]  Q, later the output
  uint8_t *sk = smem + g.off_k;    // [nc][kv_rows x 128 B] routed K slots
  uint8_t *sv = smem + g.off_v;    // [nc][kv_rows x 128 B] routed V slots
  uint8_t *sh = smem + g.off_h;    // [nc][halo rows x 128 B] V halo
  float *so = reinterpret_cast<float *>(smem + g.off_o);  // [n][o_stride]
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + g.off_bar);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x / g.R, i = blockIdx.x % g.R;
  const int y0 = (i / g.S) * g.hr, x0 = (i % g.S) * g.wr;
  const int nslots = g.topk * g.slot;
  constexpr int PAD = KS / 2;

  if (tid == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_vh);
    prefetch_tensormap(&tm_o);
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  // Rows of the K/V slots that no copy writes (region slots padded to 8 rows,
  // the buffer tail) must hold zeros: P is zero there but 0 * NaN is not.
  if (g.slot != g.n || g.kv_rows != nslots) {
    const int rows_pad = g.kv_rows;
    for (int e = tid; e < 2 * g.nc * rows_pad * 8; e += kAttendThreads) {
      const int c16 = e & 7, row = (e >> 3) % rows_pad, buf = (e >> 3) / rows_pad;
      const bool pad = row >= nslots || (row % g.slot) >= g.n;
      if (pad) {
        uint8_t *base = (buf < g.nc ? sk : sv) + (buf % g.nc) * g.kv_chunk;
        *reinterpret_cast<uint4 *>(base + row * 128 + c16 * 16) =
            make_uint4(0, 0, 0, 0);
      }
    }
  }
  __syncthreads();

  if (tid == 0) {
    const uint32_t halo_bytes = g.nc * g.halo_w * g.halo_h * 128u;
    mbar_arrive_expect_tx(&bar[1], halo_bytes);
    for (int cc = 0; cc < g.nc; ++cc)
      tma_load_4d(sh + cc * g.h_chunk, &tm_vh, &bar[1], cc * 64, x0 - PAD,
                  y0 - PAD, b);
    const uint32_t tile = g.n * 128u;
    mbar_arrive_expect_tx(&bar[0], g.nc * tile * (1u + 2u * g.topk));
    for (int cc = 0; cc < g.nc; ++cc)
      tma_load_4d(sq + cc * g.q_chunk, &tm_q, &bar[0], cc * 64, x0, y0, b);
    const int32_t *ri = idx + ((size_t)b * g.R + i) * g.topk;
    for (int m = 0; m < g.topk; ++m) {
      int j = __ldg(ri + m);
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
        tma_load_4d(sk + off, &tm_k, &bar[0], cc * 64, xj, yj, b);
        tma_load_4d(sv + off, &tm_v, &bar[0], cc * 64, xj, yj, b);
      }
    }
  }

  // ---------------------------------------------------------- attention
  mbar_wait(&bar[0], 0);
  const int tasks = g.heads * g.q_blocks;
  for (int task = warp; task < tasks; task += kAttendThreads / 32) {
    const int h = task % g.heads, qb = task / g.heads;
    const int cc = h >> 1, cb = (h & 1) * 4;  // chunk, first 16-B column
    const uint32_t q_base = smem_u32(sq + cc * g.q_chunk);
    const uint32_t k_base = smem_u32(sk + cc * g.kv_chunk);
    const uint32_t v_base = smem_u32(sv + cc * g.kv_chunk);

    uint32_t qa[2][4];
#pragma unroll
    for (int ks = 0; ks < 2; ++ks)
      ldsm_x4(q_base + swz128(qb * 16 + (lane & 15), cb + ks * 2 + (lane >> 4)),
              qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);

    float o[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[a][e] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    for (int kb = 0; kb < nslots; kb += 64) {
      float s[8][4];
#pragma unroll
      for (int jt = 0; jt < 8; ++jt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) s[jt][e] = 0.f;
        const int key0 = kb + jt * 8;
        if (key0 < nslots) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(k_base + swz128(key0 + (lane & 7), cb + (lane >> 3)), b0, b1,
                  b2, b3);
          mma_bf16_16816(s[jt], qa[0], b0, b1);
          mma_bf16_16816(s[jt], qa[1], b2, b3);
        }
      }
      // scale to log2 units and mask padding / absent keys
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int jt = 0; jt < 8; ++jt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = kb + jt * 8 + 2 * (lane & 3) + (e & 1);
          const bool ok = key < nslots && (key % g.slot) < g.n;
          s[jt][e] = ok ? s[jt][e] * g.scale_log2 : -INFINITY;
          mx[e >> 1] = fmaxf(mx[e >> 1], s[jt][e]);
        }
      float base[2], alpha[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        const float m_new = fmaxf(m_run[r], mx[r]);
        base[r] = (m_new == -INFINITY) ? 0.f : m_new;
        alpha[r] = exp2f(m_run[r] - base[r]);
        m_run[r] = m_new;
      }
      // P = exp2(S - max), rounded to bf16 once; the row sum adds the
      // rounded values so the weights used by P V sum exactly to l.
      uint32_t p[8][2];
      float rs[2] = {0.f, 0.f};
#pragma unroll
      for (int jt = 0; jt < 8; ++jt) {
        p[jt][0] = pack_bf16x2(exp2f(s[jt][0] - base[0]), exp2f(s[jt][1] - base[0]));
        p[jt][1] = pack_bf16x2(exp2f(s[jt][2] - base[1]), exp2f(s[jt][3] - base[1]));
        rs[0] += bf16_lo(p[jt][0]) + bf16_hi(p[jt][0]);
        rs[1] += bf16_lo(p[jt][1]) + bf16_hi(p[jt][1]);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) l_run[r] = l_run[r] * alpha[r] + rs[r];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        o[a][0] *= alpha[0]; o[a][1] *= alpha[0];
        o[a][2] *= alpha[1]; o[a][3] *= alpha[1];
      }
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        if (kb + t * 16 < nslots) {
          const uint32_t pa[4] = {p[2 * t][0], p[2 * t][1], p[2 * t + 1][0],
                                  p[2 * t + 1][1]};
          const int vrow = kb + t * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
          for (int np = 0; np < 2; ++np) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4_trans(v_base + swz128(vrow, cb + np * 2 + (lane >> 4)), r0,
                          r1, r2, r3);
            mma_bf16_16816(o[2 * np], pa, r0, r1);
            mma_bf16_16816(o[2 * np + 1], pa, r2, r3);
          }
        }
      }
    }
    // normalise and park O (f32) for the epilogue
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
    }
    const float inv0 = 1.f / l_run[0], inv1 = 1.f / l_run[1];
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
  __syncthreads();

  // ------------------------------------------------- LePE + add + bf16
  mbar_wait(&bar[1], 0);
  const int pairs = g.C / 2;
  const int groups = (g.hr + kLepeRows - 1) / kLepeRows;
  for (int item = tid; item < pairs * g.wr * groups; item += kAttendThreads) {
    const int cp = item % pairs, rest = item / pairs;
    const int x = rest % g.wr, ry0 = (rest / g.wr) * kLepeRows;
    const int c = 2 * cp, cc = c >> 6, c16 = (c & 63) >> 3, cw = (c & 7) * 2;
    float w0[KS * KS], w1[KS * KS];
#pragma unroll
    for (int e = 0; e < KS * KS; ++e) {
      w0[e] = __ldg(lepe_w + (size_t)c * KS * KS + e);
      w1[e] = __ldg(lepe_w + (size_t)(c + 1) * KS * KS + e);
    }
    const float b0 = lepe_b ? __ldg(lepe_b + c) : 0.f;
    const float b1 = lepe_b ? __ldg(lepe_b + c + 1) : 0.f;
    float acc[kLepeRows][2];
#pragma unroll
    for (int r = 0; r < kLepeRows; ++r) { acc[r][0] = b0; acc[r][1] = b1; }
    const uint8_t *hb = sh + cc * g.h_chunk;
#pragma unroll
    for (int yy = 0; yy < kLepeRows + KS - 1; ++yy) {
      const int hy = ry0 + yy;  // halo row
      if (hy < g.halo_h) {
#pragma unroll
        for (int w = 0; w < KS; ++w) {
          const int hrow = hy * g.halo_w + x + w;
          const uint32_t t2 =
              *reinterpret_cast<const uint32_t *>(hb + swz128(hrow, c16) + cw);
          const float v0 = bf16_lo(t2), v1 = bf16_hi(t2);
#pragma unroll
          for (int u = 0; u < KS; ++u) {
            const int r = yy - u;  // output row in the block using this tap
            if (r >= 0 && r < kLepeRows) {
              acc[r][0] = fmaf(w0[u * KS + w], v0, acc[r][0]);
              acc[r][1] = fmaf(w1[u * KS + w], v1, acc[r][1]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kLepeRows; ++r) {
      const int row = ry0 + r;
      if (row < g.hr) {
        const int t = row * g.wr + x;
        const float2 ov = *reinterpret_cast<const float2 *>(so + t * g.o_stride + c);
        *reinterpret_cast<uint32_t *>(sq + cc * g.q_chunk + swz128(t, c16) + cw) =
            pack_bf16x2(acc[r][0] + ov.x, acc[r][1] + ov.y);
      }
    }
  }
  fence_async_shared();
  __syncthreads();
  if (tid == 0) {
    for (int cc = 0; cc < g.nc; ++cc)
      tma_store_4d(&tm_o, sq + cc * g.q_chunk, cc * 64, x0, y0, b);
    tma_store_commit();
    tma_store_wait_read();
  }
}

}  // namespace bra

// forward_image.cuh -- the whole BRA forward in one launch for bf16 maps
// whose image fits in shared memory one 64-channel chunk at a time and whose
// region grid is small (the stage-3 shape: 14 x 14 tokens, 2 x 2 regions,
// 49 regions, top-16).
//
// One thread-block cluster per image, one CTA per 64-channel chunk. Each CTA
// brings its chunk of the whole image's Q and K (first) and V and the V halo
// (second) into shared memory with four TMA box copies. Then
//   1. routing (page "CVPR2023：BiFormer中的双层路由注意力机制解析" §3:
//      q_r = q.mean, A_r = q_r k_r^T, I_r = topk(A_r)): the region means of
//      the chunk's 64 channels from the tiles, the chunk's partial affinity
//      (an FMA chain over its channels), a cluster barrier; then, for the
//      rows i with i % nc == rank, the full affinity as the partials of all
//      chunks added in chunk order (read from the peers' shared memory) and
//      the top-k, written to global memory and into every CTA of the
//      cluster; a second cluster barrier;
//   2. the key table from the routing, then routed attention and LePE
//      exactly as the image-resident attend kernel (attend_image.cuh).
//
// The routing follows the arithmetic of the routing kernel (route.cuh) step
// for step, so that both give the same index bit for bit: a region mean
// sums the tokens in L interleaved partial sums (tokens t = j, j + L, ...),
// adds the partials pairwise and scales by 1/n; the affinity is one FMA chain
// per 64 channels, the chains added in channel order. Q and K are read from
// HBM once, by TMA.
#pragma once

#include "attend_image.cuh"
#include "route.cuh"

namespace bra {

constexpr int kRouteWarps = kImgWarps;  // every warp routes
constexpr int kRouteThreads = 32 * kRouteWarps;

struct FusedGeom {
  ImageGeom img;
  int L;              // interleaved partial sums of a region mean (32 / G: 1, 2, 4)
  int rp;             // R rounded up to a multiple of 4
  float inv_n;        // 1 / tokens per region
  uint32_t off_qm;    // Q means, channel-major [64][rp] f32
  uint32_t off_km;    // K means [64][rp] f32
  uint32_t off_a;     // full affinity of this CTA's rows [ceil(R/nc)][R] f32
  uint32_t off_p;     // this chunk's partial affinity [R][R] f32
  uint32_t off_ridx;  // routing [R][topk] int32
  uint32_t off_tok;   // region first tokens [64] and token offsets [16], uint16
  uint32_t off_bar;   // two mbarriers: Q and K; V and halo
};

// Cluster barrier halves (every thread of every CTA of the cluster arrives
// once per phase, then waits for it).
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The means of the eight channels of 16-byte chunk `chunk` of region r over
// its tokens, from a swizzled tile of the image chunk, in the routing
// kernel's order: partial j (j < L) sums the tokens t = j, j + L, ... in
// row-major order, the partials are added pairwise ((0 + 1) + (2 + 3);
// partials from L on are zero, which leaves the sums unchanged) and the sums
// are scaled by 1/n. L is 1, 2 or 4. base is the region's first token, toff
// the offset of each of its tokens from it.
__device__ __forceinline__ void region_mean_chunk(const uint8_t *tile, int base,
                                                  const uint16_t *toff, int n, int chunk,
                                                  int L, float inv_n, float (&m)[8]) {
  float2 part[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) part[j][e] = make_float2(0.f, 0.f);
    if (j < L)
      for (int t = j; t < n; t += L) {
        const int tok = base + toff[t];
        const uint4 w = *reinterpret_cast<const uint4 *>(tile + tok_addr(tok, chunk));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          part[j][e] = __fadd2_rn(part[j][e],
                                  make_float2(__uint_as_float(__byte_perm(ws[e], 0u, 0x1044u)),
                                              __uint_as_float(__byte_perm(ws[e], 0u, 0x3244u))));
      }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    m[2 * e] = ((part[0][e].x + part[1][e].x) + (part[2][e].x + part[3][e].x)) * inv_n;
    m[2 * e + 1] = ((part[0][e].y + part[1][e].y) + (part[2][e].y + part[3][e].y)) * inv_n;
  }
}

// The rest of the routing by the CTA with chunk cc of a cluster of nc, all
// its threads, once this chunk's region means are in qm and km (channel-major
// [64][RP], columns 0 .. R-1): the chunk's partial affinity, a cluster
// barrier, the full affinity of the rows i with i % nc == cc (partials added
// in chunk order, from the peers' shared memory), their top-k to idx_out (and
// the full rows to aff_out when given) and, when ridx is given, into every
// CTA's copy of the routing; a last cluster barrier.
template <int NT = kRouteThreads>
__device__ __forceinline__ void route_cluster_rows(const ImageGeom &g, const FusedGeom &fg,
                                                   float *qm, float *km, float *aff,
                                                   float *part, int32_t *ridx,
                                                   int32_t *idx_out, float *aff_out, int b,
                                                   int cc, int nc, int tid, int warp, int lane,
                                                   cg::cluster_group &cluster) {
  const int R = g.R, RP = fg.rp;
  // the padding columns R .. RP-1 are zero (their products are dropped)
  for (int e = tid; e < 2 * 64 * (RP - R); e += NT) {
    const int tensor = e / (64 * (RP - R)), rest = e - tensor * (64 * (RP - R));
    (tensor ? km : qm)[(rest / (RP - R)) * RP + R + rest % (RP - R)] = 0.f;
  }
  __syncthreads();

  // ---- partial affinity over this chunk: one thread per 4 x 4 tile (rows
  // i0.., columns j0..), sixteen FMA chains in channel order
  const int tiles = RP / 4;
  for (int t = tid; t < tiles * tiles; t += NT) {
    const int i0 = (t / tiles) * 4, j0 = (t % tiles) * 4;
    // the chains in pairs (columns j0 + 2h, j0 + 2h + 1): each half of a
    // paired FMA rounds as a single one
    float2 acc[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[r][0] = acc[r][1] = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int c = 0; c < 64; ++c) {
      const float4 q4 = *reinterpret_cast<const float4 *>(qm + c * RP + i0);
      const float4 k4 = *reinterpret_cast<const float4 *>(km + c * RP + j0);
      const float qv[4] = {q4.x, q4.y, q4.z, q4.w};
      const float2 k01 = make_float2(k4.x, k4.y), k23 = make_float2(k4.z, k4.w);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float2 q2 = make_float2(qv[r], qv[r]);
        acc[r][0] = __ffma2_rn(q2, k01, acc[r][0]);
        acc[r][1] = __ffma2_rn(q2, k23, acc[r][1]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float a[4] = {acc[r][0].x, acc[r][0].y, acc[r][1].x, acc[r][1].y};
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (i0 + r < R && j0 + c < R) part[(i0 + r) * R + j0 + c] = a[c];
    }
  }
  cluster_arrive_release();
  cluster_wait_acquire();  // every chunk's partial affinity is complete

  // ---- the full affinity of this CTA's rows i = cc, cc + nc, ...: partials
  // added in chunk order
  const int ro = (R - cc + nc - 1) / nc;
  for (int e = tid; e < ro * R; e += NT) {
    const int s = e / R, j = e - s * R;
    const int i = cc + nc * s;
    float a = 0.f;
    for (int rk = 0; rk < nc; ++rk) {
      const float p = rk == cc ? part[i * R + j] : cluster.map_shared_rank(part, rk)[i * R + j];
      a = rk == 0 ? p : a + p;
    }
    aff[s * R + j] = a;
    if (aff_out) aff_out[((size_t)b * R + i) * R + j] = a;
  }
  __syncthreads();

  // ---- top-k of this CTA's rows (one warp per row), to global memory and
  // into every CTA's copy of the routing
  for (int s = warp; s < ro; s += (NT / 32)) {
    const int i = cc + nc * s;
    constexpr int MAXJ = 2;  // at most 64 regions
    float val[MAXJ];
#pragma unroll
    for (int t = 0; t < MAXJ; ++t) {
      const int j = lane + 32 * t;
      float a = -INFINITY;
      if (j < R) {
        a = aff[s * R + j];
        a = (a == a) ? a : -INFINITY;  // a NaN never wins
      }
      val[t] = a;
    }
    select_topk<MAXJ>(val, aff + s * R, R, g.topk, lane,
                      idx_out + ((size_t)b * R + i) * g.topk, ridx ? ridx + i * g.topk : nullptr);
    __syncwarp();
    if (!ridx) continue;
    for (int e = lane; e < (nc - 1) * g.topk; e += 32) {
      const int rk = (cc + 1 + e / g.topk) % nc, m = e % g.topk;
      cluster.map_shared_rank(ridx, rk)[i * g.topk + m] = ridx[i * g.topk + m];
    }
  }
  // every CTA's rows are complete (and have reached every CTA); no CTA reads
  // a peer's shared memory after this
  cluster_arrive_release();
  cluster_wait_acquire();
}


// Routing of image b by the CTA with chunk cc of a cluster of nc (see
// above), all its threads. Leaves the whole routing [R][topk] in ridx of
// every CTA of the cluster; writes this CTA's rows to idx_out.
__device__ __forceinline__ void route_in_cluster(
    const ImageGeom &g, const FusedGeom &fg, const uint8_t *smem, float *qm, float *km,
    float *aff, float *part, int32_t *ridx, const uint16_t *rbase, const uint16_t *toff,
    int32_t *idx_out, uint64_t *bar_qk, int b, int cc, int nc, int tid, int warp, int lane,
    cg::cluster_group &cluster) {
  const int R = g.R, RP = fg.rp;
  mbar_wait(bar_qk, 0);

  // ---- region means of this chunk's 64 channels: one thread per (tensor,
  // region, 16-byte chunk); stored channel-major, [64][RP]
  for (int e = tid; e < 2 * R * 8; e += kRouteThreads) {
    const int tensor = e / (R * 8), rest = e - tensor * (R * 8);
    const int r = rest >> 3, chunk = rest & 7;
    float m[8];
    region_mean_chunk(tensor ? smem + g.off_k : smem, rbase[r], toff, g.n, chunk, fg.L,
                      fg.inv_n, m);
    float *dst = (tensor ? km : qm) + chunk * 8 * RP + r;
#pragma unroll
    for (int c = 0; c < 8; ++c) dst[c * RP] = m[c];
  }
  route_cluster_rows(g, fg, qm, km, aff, part, ridx, idx_out, nullptr, b, cc, nc, tid, warp,
                     lane, cluster);
}

template <int KS, int RB>
__global__ void __launch_bounds__(kImgThreads, 1)
    bra_forward_image_kernel(const __grid_constant__ CUtensorMap tm_q,
                             const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v,
                             const __grid_constant__ CUtensorMap tm_vh,
                             __nv_bfloat16 *__restrict__ out, int32_t *__restrict__ idx_out,
                             const float *__restrict__ lepe_w,
                             const float *__restrict__ lepe_b, FusedGeom fg) {
  const ImageGeom &g = fg.img;
  extern __shared__ uint8_t fused_smem_raw[];
  uint8_t *smem = fused_smem_raw + ((1024u - (smem_u32(fused_smem_raw) & 1023u)) & 1023u);
  float *so = reinterpret_cast<float *>(smem + g.off_o);    // [H*W][64]
  float *sw = reinterpret_cast<float *>(smem + g.off_w);    // [KS*KS][64], bias [64]
  uint16_t *ktab = reinterpret_cast<uint16_t *>(smem + g.off_tab);  // [R][nkp]
  float *qm = reinterpret_cast<float *>(smem + fg.off_qm);
  float *km = reinterpret_cast<float *>(smem + fg.off_km);
  float *aff = reinterpret_cast<float *>(smem + fg.off_a);
  float *part = reinterpret_cast<float *>(smem + fg.off_p);
  int32_t *ridx = reinterpret_cast<int32_t *>(smem + fg.off_ridx);
  uint16_t *rbase = reinterpret_cast<uint16_t *>(smem + fg.off_tok);  // [R]
  uint16_t *toff = rbase + 64;                                        // [n]
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + fg.off_bar);

  cg::cluster_group cluster = cg::this_cluster();
  const int nc = static_cast<int>(cluster.num_blocks());
  const int cc = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.x / nc;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = g.R;
  constexpr int PAD = KS / 2;

  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar[0], 2 * g.H * g.W * 128);
    tma_load_4d(smem, &tm_q, &bar[0], cc * 64, 0, 0, b);
    tma_load_4d(smem + g.off_k, &tm_k, &bar[0], cc * 64, 0, 0, b);
    mbar_arrive_expect_tx(&bar[1], g.H * g.W * 128 + g.halo_w * g.halo_h * 128);
    tma_load_4d(smem + g.off_v, &tm_v, &bar[1], cc * 64, 0, 0, b);
    tma_load_4d(smem + g.off_h, &tm_vh, &bar[1], cc * 64, -PAD, -PAD, b);
  }
  // this chunk's LePE weights, tap-major
  constexpr int NW = (64 * KS * KS + kImgThreads - 1) / kImgThreads;
  float wv[NW];
#pragma unroll
  for (int u = 0; u < NW; ++u) {
    const int e = tid + u * kImgThreads;
    wv[u] = e < 64 * KS * KS ? __ldg(lepe_w + (size_t)cc * 64 * KS * KS + e) : 0.f;
  }
  const float bv = (tid < 64 && lepe_b) ? __ldg(lepe_b + cc * 64 + tid) : 0.f;
#pragma unroll
  for (int u = 0; u < NW; ++u) {
    const int e = tid + u * kImgThreads;
    if (e < 64 * KS * KS) {
      const int c = e / (KS * KS), tap = e - c * (KS * KS);
      sw[tap * 64 + c] = wv[u];
    }
  }
  if (tid < 64) sw[KS * KS * 64 + tid] = bv;
  // the zero rows of K and V (no copy writes them)
  if (tid < 16)
    *reinterpret_cast<uint4 *>(smem + (tid < 8 ? g.off_k : g.off_v) + g.H * g.W * 128 +
                               (tid & 7) * 16) = make_uint4(0, 0, 0, 0);
  // each region's first token, and each token's offset from its region's first
  if (tid < R) rbase[tid] = static_cast<uint16_t>((tid / g.S) * g.hr * g.W + (tid % g.S) * g.wr);
  if (tid >= 256 && tid - 256 < g.n) {
    const int t = tid - 256;
    toff[t] = static_cast<uint16_t>((t / g.wr) * g.W + t % g.wr);
  }
  __syncthreads();

  route_in_cluster(g, fg, smem, qm, km, aff, part, ridx, rbase, toff, idx_out, &bar[0], b, cc,
                   nc, tid, warp, lane, cluster);
  __syncthreads();  // the routing is complete in this CTA

  // ---- the key table: keys m*n .. m*n+n-1 of region i are the tokens of
  // routed region ridx[i][m] in row-major order; keys past nkeys read the
  // zero row after the image's tokens
  const int slots = R * g.topk;
  const uint16_t zero_row = static_cast<uint16_t>(g.H * g.W);
  for (int slot = tid; slot < slots; slot += kImgThreads) {
    const int i = slot / g.topk, m = slot - i * g.topk;
    const int base = rbase[ridx[slot]];
    uint16_t *row = ktab + i * g.nkp + m * g.n;
    for (int t = 0; t < g.n; ++t) row[t] = static_cast<uint16_t>(base + toff[t]);
  }
  const int tail = g.nkp - g.nkeys;
  for (int e = tid; e < R * tail; e += kImgThreads) {
    const int i = e / tail;
    ktab[i * g.nkp + g.nkeys + (e - i * tail)] = zero_row;
  }
  __syncthreads();

  mbar_wait(&bar[1], 0);

  // ---- 2. attention: (query region, both heads of the chunk) tasks
  const uint32_t q_base = smem_u32(smem), k_base = smem_u32(smem + g.off_k),
                 v_base = smem_u32(smem + g.off_v);
  if (g.n <= 8) {
    for (int i = warp; i < R; i += kImgWarps) {
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
  const int tasks = g.n <= 8 ? 0 : R * 2 * g.q_blocks;
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

// The region means of chunk cc's 64 channels of Q and K of image b, read
// from global memory, all NT threads: one thread per (tensor, region, 16-byte
// chunk), the region's tokens loaded together, then summed in the routing
// kernel's order (as region_mean_chunk does); stored channel-major, [64][RP].
template <int L, int NT>
__device__ __forceinline__ void chunk_means(const __nv_bfloat16 *__restrict__ q,
                                            const __nv_bfloat16 *__restrict__ k,
                                            const ImageGeom &g, const FusedGeom &fg, float *qm,
                                            float *km, int b, int cc, int tid) {
  const int R = g.R, RP = fg.rp;
  const size_t img = (size_t)b * g.H * g.W;
  for (int e = tid; e < 2 * R * 8; e += NT) {
    const int tensor = e / (R * 8), rest = e - tensor * (R * 8);
    const int r = rest >> 3, chunk = rest & 7;
    const int y0 = (r / g.S) * g.hr, x0 = (r % g.S) * g.wr;
    const uint4 *src = reinterpret_cast<const uint4 *>((tensor ? k : q) + cc * 64 + chunk * 8);
    uint4 v[8];
#pragma unroll
    for (int t = 0; t < 8; ++t)
      if (t < g.n)
        v[t] = __ldg(src + (img + (size_t)(y0 + t / g.wr) * g.W + x0 + t % g.wr) * (g.C / 8));
    // partial j (j < L) sums the tokens t = j, j + L, ... in increasing order
    float2 p[L][4];
#pragma unroll
    for (int j = 0; j < L; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) p[j][c] = make_float2(0.f, 0.f);
#pragma unroll
    for (int t = 0; t < 8; ++t)
      if (t < g.n) {
        const uint32_t ws[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
#pragma unroll
        for (int c = 0; c < 4; ++c)
          p[t % L][c] = __fadd2_rn(p[t % L][c],
                                   make_float2(__uint_as_float(__byte_perm(ws[c], 0u, 0x1044u)),
                                               __uint_as_float(__byte_perm(ws[c], 0u, 0x3244u))));
      }
    float *dst = (tensor ? km : qm) + chunk * 8 * RP + r;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      // the partials added pairwise, ((0 + 1) + (2 + 3)), missing ones zero
      float2 m = p[0][c];
      if (L == 2) m = __fadd2_rn(p[0][c], p[1][c]);
      if (L == 4) m = __fadd2_rn(__fadd2_rn(p[0][c], p[1 % L][c]), __fadd2_rn(p[2 % L][c], p[3 % L][c]));
      dst[(2 * c) * RP] = m.x * fg.inv_n;
      dst[(2 * c + 1) * RP] = m.y * fg.inv_n;
    }
  }
}

// ---- routing alone (steps a1-a4) for the maps of the local image kernel:
// bf16, at most 64 regions of at most 8 tokens, C / 64 in {1, 2, 4}. One
// cluster of C / 64 CTAs per image; CTA cc pools its 64 channels of Q and K
// straight from global memory (one thread per (tensor, region, 16-byte
// chunk), the region's tokens loaded together, then summed in the routing
// kernel's order, as region_mean_chunk does), then route_cluster_rows. The
// per-chunk form needs no copy of every K mean in every CTA, and its index
// is the routing kernel's bit for bit.
template <int L>
__global__ void __launch_bounds__(kRouteThreads, 2)
    bra_route_chunked_kernel(const __nv_bfloat16 *__restrict__ q,
                             const __nv_bfloat16 *__restrict__ k, FusedGeom fg,
                             int32_t *__restrict__ idx, float *__restrict__ aff_out) {
  // A dependent grid launched with programmatic serialization may start now;
  // it waits for this grid before it reads the routing index.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ __align__(16) uint8_t rc_smem[];
  const ImageGeom &g = fg.img;
  cg::cluster_group cluster = cg::this_cluster();
  const int nc = g.nc, cc = (int)cluster.block_rank(), b = blockIdx.x / nc;
  float *qm = reinterpret_cast<float *>(rc_smem + fg.off_qm);
  float *km = reinterpret_cast<float *>(rc_smem + fg.off_km);
  float *aff = reinterpret_cast<float *>(rc_smem + fg.off_a);
  float *part = reinterpret_cast<float *>(rc_smem + fg.off_p);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  chunk_means<L, kRouteThreads>(q, k, g, fg, qm, km, b, cc, tid);
  route_cluster_rows(g, fg, qm, km, aff, part, nullptr, idx, aff_out, b, cc, nc, tid, warp,
                     lane, cluster);
}

// ---- the whole forward in one launch on the local image kernel's layout
// (two CTAs per SM, so that every image's cluster is resident at once on the
// stage-3 shape): one cluster of C / 64 CTAs of kLocalThreads per image. CTA
// cc issues the TMA copy of its chunk of K, stages the LePE weights, routes
// the image with its peers (chunk_means from global memory, then
// route_cluster_rows, which leaves the whole routing in every CTA), then
// copies the V halo into the space the routing used, builds the key tables
// from its copy of the routing and runs the local kernel's attention and
// LePE (attend_image.cuh).
template <int KS, int HR, int WR, int L>
__global__ void __launch_bounds__(kLocalThreads, 2)
    bra_forward_local_kernel(const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_vh,
                             const __nv_bfloat16 *__restrict__ q,
                             const __nv_bfloat16 *__restrict__ k,
                             __nv_bfloat16 *__restrict__ out, int32_t *__restrict__ idx_out,
                             const float *__restrict__ lepe_w, const float *__restrict__ lepe_b,
                             FusedGeom fg) {
  extern __shared__ uint8_t image_smem_raw[];
  uint8_t *smem = image_smem_raw + ((1024u - (smem_u32(image_smem_raw) & 1023u)) & 1023u);
  const ImageGeom &g = fg.img;
  cg::cluster_group cluster = cg::this_cluster();
  const int nc = g.nc, cc = (int)cluster.block_rank(), b = blockIdx.x / nc;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float *sw = reinterpret_cast<float *>(smem + g.off_w);
  uint16_t *ktab = reinterpret_cast<uint16_t *>(smem + g.off_tab);
  uint16_t *vtab = reinterpret_cast<uint16_t *>(smem + g.off_v);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + g.off_bar);  // [0] K, [1] V halo
  // the routing's scratch lies in the halo's space (the halo is copied after
  // the routing); the routing itself ([R][topk]) has its own
  float *qm = reinterpret_cast<float *>(smem + fg.off_qm);
  float *km = reinterpret_cast<float *>(smem + fg.off_km);
  float *aff = reinterpret_cast<float *>(smem + fg.off_a);
  float *part = reinterpret_cast<float *>(smem + fg.off_p);
  int32_t *ridx = reinterpret_cast<int32_t *>(smem + fg.off_ridx);
  constexpr int PAD = KS / 2;
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar[0], g.H * g.W * 128);
    tma_load_4d(smem + g.off_k, &tm_k, &bar[0], cc * 64, 0, 0, b);
  }
  // the zero rows after the K tile and after the halo (no copy writes them;
  // the routing's scratch ends before the halo's zero row)
  if (tid < 8)
    *reinterpret_cast<uint4 *>(smem + g.off_k + g.H * g.W * 128 + tid * 16) =
        make_uint4(0, 0, 0, 0);
  else if (tid < 17)
    *reinterpret_cast<uint4 *>(smem + g.off_h + g.halo_w * g.halo_h * kHaloPitch +
                               (tid - 8) * 16) = make_uint4(0, 0, 0, 0);
  image_weights<KS, kLocalThreads>(sw, lepe_w, lepe_b, cc, tid, [] {});
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

  // ---- routing (steps a1-a4)
  chunk_means<L, kLocalThreads>(q, k, g, fg, qm, km, b, cc, tid);
  route_cluster_rows<kLocalThreads>(g, fg, qm, km, aff, part, ridx, idx_out, nullptr, b, cc,
                                    nc, tid, warp, lane, cluster);
  __syncthreads();  // no thread here or in a peer touches the scratch any more
  if (tid == 0) {
    fence_async_shared();  // the scratch's generic accesses before the copy
    mbar_arrive_expect_tx(&bar[1], g.halo_w * g.halo_h * kHaloPitch);
    tma_load_4d(smem + g.off_h, &tm_vh, &bar[1], cc * 64, -PAD, -PAD, b);
  }
  int jpre[4];
  prefetch_routing<kLocalThreads, true>(g, ridx, tid, jpre);
  image_key_tables<KS, kLocalThreads, true>(g, ktab, vtab, ridx, jpre, tid);
  __syncthreads();
  mbar_wait(&bar[0], 0);
  mbar_wait(&bar[1], 0);

  // ---- attention + LePE (steps a5-a7)
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

// route.cuh -- region-level routing of BRA on sm_103a.
//
// Computes, per image, the region means of Q and K, the region affinity
// A = mean(q_r) mean(k_r)^T over all C channels and the top-k regions of each
// row (page "CVPR2023：BiFormer中的双层路由注意力机制解析" §3: q_r = q.mean,
// A_r = q_r k_r^T, I_r = topk(A_r); page "从静态到动态：BRA双层路由注意力
// 如何革新视觉Transformer的计算范式" §2 mean pooling and §4 TopkRouting).
//
// One thread-block cluster per image. Each CTA of the cluster owns the
// regions r with r % CL == rank. One warp pools one (tensor, region): a
// region's rows are contiguous runs of wr*C elements, read with 16-byte loads
// that a lane issues back to back (every lane always lands on the same 16-byte
// channel group, since a token holds a power-of-two number of them), then a
// few shuffles sum the lanes of each group. Then the cluster synchronises,
// every CTA copies all K means out of its peers' shared memory (distributed
// shared memory; for grids too large to copy, it reads them from the peers in
// place), and computes the affinity rows and the top-k of its own regions.
// Nothing goes through global memory but the inputs and the outputs.
// Arithmetic is float32 in a fixed order: a region mean sums its tokens in
// L = 32 / G interleaved partial sums (lane j of a channel group takes the
// tokens t = j, j + L, ... in row-major order), adds the partials pairwise
// (j with j ^ 1, then with j ^ 2, ...) and multiplies by 1/n; the affinity
// follows kAffChunk below.
#pragma once

#include <cooperative_groups.h>

#include "ptx.cuh"

namespace bra {

namespace cg = cooperative_groups;

// Threads per CTA: 256 when there are enough clusters to fill the GPU (four
// CTAs per SM), 512 when there are few (more warps per image; clusters of 16
// such CTAs still pack several to a GPC).
constexpr int kRouteThreadsMany = 256;
constexpr int kRouteThreadsFew = 512;
constexpr int kRouteUnroll = 8;  // 16-byte loads a lane keeps in flight

constexpr int kAffRows = 4;  // owned rows of one affinity tile

// The affinity A[i][j] = sum_c Qm[i][c] Km[j][c] is formed as one float32 FMA
// chain per run of kAffChunk channels (in channel order, from zero), and the
// chains' results are added in run order. Every kernel that computes the
// routing follows this order, so that their routing indices agree bit for bit.
constexpr int kAffChunk = 64;

struct RouteGeom {
  int H, W, C, S, topk;
  int hr, wr, n, R;
  int G;        // 16-byte channel groups per token (a power of two <= 32)
  uint32_t off_qm, off_km, off_kall;  // bytes into shared memory
  uint32_t off_aff;  // owned affinity rows [ro][R] (0: rows not staged)
};

template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void add(const uint4 &v, float2 (&acc)[4]) {
    acc[0] = __fadd2_rn(acc[0], make_float2(__uint_as_float(v.x), __uint_as_float(v.y)));
    acc[1] = __fadd2_rn(acc[1], make_float2(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
};
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  // the two bf16 of a word as a float pair, by byte permutes
  __device__ static float2 pair(uint32_t w) {
    return make_float2(__uint_as_float(__byte_perm(w, 0u, 0x1044u)),
                       __uint_as_float(__byte_perm(w, 0u, 0x3244u)));
  }
  __device__ static void add(const uint4 &v, float2 (&acc)[4]) {
    acc[0] = __fadd2_rn(acc[0], pair(v.x));
    acc[1] = __fadd2_rn(acc[1], pair(v.y));
    acc[2] = __fadd2_rn(acc[2], pair(v.z));
    acc[3] = __fadd2_rn(acc[3], pair(v.w));
  }
};

// A streaming 16-byte load: not kept in L1, and L2 fetches the surrounding
// 256 bytes (a region row is 1 KB or more of contiguous tokens).
__device__ __forceinline__ uint4 ld_stream16(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Sums this lane's 16-byte chunks of one region (rows of seg chunks, row
// stride row_stride chunks; chunk lane + 32 m of the region). SW = seg / 32
// when seg is a multiple of 32 (then chunk m of a lane sits at row m / SW,
// column lane + 32 (m % SW), all offsets known at compile time); SW = 0 is
// the general case.
template <typename T, int SW>
__device__ __forceinline__ void pool_region(const uint4 *base, size_t row_stride, int hr,
                                            int seg, int lane, float2 (&acc)[4]) {
  if constexpr (SW > 0) {
    const uint4 *p = base + lane;
    constexpr int RU = (SW <= 0 || SW >= kRouteUnroll) ? 1 : kRouteUnroll / SW;  // rows per batch
    for (int y0 = 0; y0 < hr; y0 += RU) {
      uint4 v[RU][SW];
#pragma unroll
      for (int y = 0; y < RU; ++y)
#pragma unroll
        for (int c = 0; c < SW; ++c)
          v[y][c] = y0 + y < hr ? ld_stream16(p + (size_t)y * row_stride + 32 * c)
                                : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int y = 0; y < RU; ++y)
#pragma unroll
        for (int c = 0; c < SW; ++c) Vec16<T>::add(v[y][c], acc);
      p += RU * row_stride;
    }
    return;
  }
  const int total = hr * seg;
  int row = lane / seg, col = lane % seg;
  for (int j0 = lane; j0 < total; j0 += 32 * kRouteUnroll) {
    uint4 v[kRouteUnroll];
#pragma unroll
    for (int u = 0; u < kRouteUnroll; ++u) {
      v[u] = make_uint4(0, 0, 0, 0);
      if (j0 + 32 * u < total) v[u] = __ldg(base + row * row_stride + col);
      col += 32;
      while (col >= seg) {
        col -= seg;
        ++row;
      }
    }
#pragma unroll
    for (int u = 0; u < kRouteUnroll; ++u) Vec16<T>::add(v[u], acc);
  }
}

// The top-k of one affinity row, chosen by one warp: columns in order of
// decreasing value, equal values by increasing column; a NaN never wins.
// val[t] holds the row's value at column lane + 32 t (-inf from column R on,
// NaN already replaced by -inf). When the row also sits in shared memory
// (row != nullptr), the grid is small (R <= 64) and many regions are routed
// (topk > 4), each lane ranks its values against the whole row (one
// broadcast load per column, no shuffles) and writes each to its place;
// otherwise topk rounds of a warp arg-max. The topk columns go to dst (and
// to dst2 when given).
template <int MAXJ>
__device__ __forceinline__ void select_topk(const float (&val)[MAXJ], const float *row, int R,
                                            int topk, int lane, int32_t *dst, int32_t *dst2) {
  if (row && R <= 64 && topk > 4) {
    int rank_of[MAXJ];
#pragma unroll
    for (int t = 0; t < MAXJ; ++t) rank_of[t] = 0;
    // eight columns at a time, their loads issued together
    for (int jj0 = 0; jj0 < R; jj0 += 8) {
      float a8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) a8[u] = row[min(jj0 + u, R - 1)];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int jj = jj0 + u;
        const float a = (a8[u] == a8[u]) ? a8[u] : -INFINITY;
#pragma unroll
        for (int t = 0; t < MAXJ; ++t) {
          const int j = lane + 32 * t;
          rank_of[t] += (jj < R && (a > val[t] || (a == val[t] && jj < j))) ? 1 : 0;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < MAXJ; ++t) {
      const int j = lane + 32 * t;
      if (j < R && rank_of[t] < topk) {
        dst[rank_of[t]] = j;
        if (dst2) dst2[rank_of[t]] = j;
      }
    }
    return;
  }
  unsigned taken = 0;  // bit t: column lane + 32 t already chosen
  for (int m = 0; m < topk; ++m) {
    float bv = -INFINITY;
    int bj = 0x7fffffff;
#pragma unroll
    for (int t = 0; t < MAXJ; ++t) {
      const int j = lane + 32 * t;
      if (j < R && !((taken >> t) & 1u) && (val[t] > bv || (val[t] == bv && j < bj))) {
        bv = val[t];
        bj = j;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oj = __shfl_xor_sync(0xffffffffu, bj, off);
      if (ov > bv || (ov == bv && oj < bj)) {
        bv = ov;
        bj = oj;
      }
    }
    if ((bj & 31) == lane) taken |= 1u << (bj >> 5);
    if (lane == 0) {
      dst[m] = bj;
      if (dst2) dst2[m] = bj;
    }
  }
}

// The routing of image b by one CTA of a cluster of CL CTAs (NT threads):
// the CTA of rank r owns the regions r, r + CL, ... and writes their rows of
// the routing index (and of the affinity, when given). route_smem is the
// CTA's dynamic shared memory (layout of RouteGeom). On return no peer reads
// this CTA's shared memory any more.
// MAXJ = ceil(R / 32): affinity values each lane keeps for the top-k.
// LOCAL_K: copy every K mean into local shared memory first (fast path);
// otherwise read them from the peers' shared memory in the affinity loop.
template <typename T, int MAXJ, bool LOCAL_K, int NT, int SW>
__device__ __forceinline__ void route_cta(const T *__restrict__ q, const T *__restrict__ k,
                                          const RouteGeom &g, int32_t *__restrict__ idx,
                                          float *__restrict__ affinity, uint8_t *route_smem,
                                          int b) {
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int R = g.R, C = g.C;
  const int ro = (R - rank + CL - 1) / CL;  // owned regions rank, rank+CL, ...
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int VEC = Vec16<T>::N;

  float *qm = reinterpret_cast<float *>(route_smem + g.off_qm);      // [ro_max][C]
  float *km = reinterpret_cast<float *>(route_smem + g.off_km);      // [ro_max][C]
  float *kall = reinterpret_cast<float *>(route_smem + g.off_kall);  // [R][C+1]

  // ---- 1. region means of q and k: one warp per (tensor, owned region) ----
  const int seg = g.wr * g.G;  // 16-byte chunks in one region row
  const size_t row_stride = (size_t)g.W * g.G;
  const float inv_n = 1.0f / static_cast<float>(g.n);
  for (int task = warp; task < 2 * ro; task += NT / 32) {
    const int tensor = task & 1, s = task >> 1;
    const int r = rank + CL * s;
    const int y0 = (r / g.S) * g.hr, x0 = (r % g.S) * g.wr;
    const uint4 *base = reinterpret_cast<const uint4 *>(tensor ? k : q) +
                        (((size_t)b * g.H + y0) * g.W + x0) * g.G;
    float2 acc2[4] = {};
    pool_region<T, SW>(base, row_stride, g.hr, seg, lane, acc2);
    float acc[8] = {acc2[0].x, acc2[0].y, acc2[1].x, acc2[1].y,
                    acc2[2].x, acc2[2].y, acc2[3].x, acc2[3].y};
    // lanes l and l + G, l + 2G, ... hold the same channel group
    for (int off = g.G; off < 32; off <<= 1)
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
    float *dst = (tensor ? km : qm) + s * C;
    if (lane < g.G)
#pragma unroll
      for (int e = 0; e < VEC; ++e) dst[lane * VEC + e] = acc[e] * inv_n;
  }

  cluster.sync();

  // ---- 2. gather every region's K mean from the cluster ----
  if (LOCAL_K) {
    const int c4n = C / 4;
    for (int e = tid; e < R * c4n; e += NT) {
      const int r = e / c4n, c4 = e % c4n;
      const float *peer = cluster.map_shared_rank(km, r % CL);
      const float4 v = *reinterpret_cast<const float4 *>(peer + (r / CL) * C + 4 * c4);
      float *d = kall + r * (C + 1) + 4 * c4;
      d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
    }
    cluster.sync();  // peers are done reading our km; kall complete
  }

  // ---- 3. affinity rows and top-k ----
  float *arow = reinterpret_cast<float *>(route_smem + g.off_aff);  // [ro][R]
  if (LOCAL_K && g.off_aff) {
    // tiles of kAffRows owned rows x 32 columns (lane = column j), spread over
    // all warps: per four channels, four K-mean values of the lane's column
    // and one broadcast 16-byte load of each row's Q mean; the FMAs still run
    // channel by channel in order
    const int rtiles = (ro + kAffRows - 1) / kAffRows, ctiles = (R + 31) / 32;
    for (int t = warp; t < rtiles * ctiles; t += NT / 32) {
      const int r0 = (t / ctiles) * kAffRows, j = (t % ctiles) * 32 + lane;
      const float *kj = kall + min(j, R - 1) * (C + 1);
      const float *q0 = qm + min(r0, ro - 1) * C;
      float tot[kAffRows];
      for (int c0 = 0; c0 < C; c0 += kAffChunk) {
        const int c1 = min(c0 + kAffChunk, C);
        float acc[kAffRows];
#pragma unroll
        for (int r = 0; r < kAffRows; ++r) acc[r] = 0.f;
#pragma unroll 2
        for (int c = c0; c < c1; c += 4) {
          const float k0 = kj[c], k1 = kj[c + 1], k2 = kj[c + 2], k3 = kj[c + 3];
#pragma unroll
          for (int r = 0; r < kAffRows; ++r) {
            // rows past the owned ones repeat the last (their results are dropped)
            const float4 q4 = *reinterpret_cast<const float4 *>(
                q0 + (r0 + r < ro ? r : 0) * C + c);
            float a = fmaf(q4.x, k0, acc[r]);
            a = fmaf(q4.y, k1, a);
            a = fmaf(q4.z, k2, a);
            acc[r] = fmaf(q4.w, k3, a);
          }
        }
#pragma unroll
        for (int r = 0; r < kAffRows; ++r) tot[r] = c0 == 0 ? acc[r] : tot[r] + acc[r];
      }
      if (j < R)
#pragma unroll
        for (int r = 0; r < kAffRows; ++r)
          if (r0 + r < ro) arow[(r0 + r) * R + j] = tot[r];
    }
    __syncthreads();
  }
  for (int s = warp; s < ro; s += NT / 32) {
    const int i = rank + CL * s;
    float dot[MAXJ];
    if (LOCAL_K && g.off_aff) {
#pragma unroll
      for (int t = 0; t < MAXJ; ++t) dot[t] = arow[s * R + min(lane + 32 * t, R - 1)];
    } else {
      // one warp per row, lanes over columns (rows too long to stage)
      const float *qi = qm + s * C;
      const float *kj[MAXJ];
#pragma unroll
      for (int t = 0; t < MAXJ; ++t) {
        const int j = min(lane + 32 * t, R - 1);
        kj[t] = LOCAL_K ? kall + j * (C + 1)
                        : cluster.map_shared_rank(km, j % CL) + (j / CL) * C;
      }
      for (int c0 = 0; c0 < C; c0 += kAffChunk) {
        const int c1 = min(c0 + kAffChunk, C);
        float acc[MAXJ];
#pragma unroll
        for (int t = 0; t < MAXJ; ++t) acc[t] = 0.f;
        for (int c = c0; c < c1; ++c) {
          const float qc = qi[c];
#pragma unroll
          for (int t = 0; t < MAXJ; ++t) acc[t] = fmaf(qc, kj[t][c], acc[t]);
        }
#pragma unroll
        for (int t = 0; t < MAXJ; ++t) dot[t] = c0 == 0 ? acc[t] : dot[t] + acc[t];
      }
    }
    float val[MAXJ];
#pragma unroll
    for (int t = 0; t < MAXJ; ++t) {
      const int j = lane + 32 * t;
      float a = -INFINITY;
      if (j < R) {
        if (affinity) affinity[((size_t)b * R + i) * R + j] = dot[t];
        a = (dot[t] == dot[t]) ? dot[t] : -INFINITY;  // a NaN never wins
      }
      val[t] = a;
    }
    select_topk<MAXJ>(val, (LOCAL_K && g.off_aff) ? arow + s * R : nullptr, R, g.topk, lane,
                      idx + ((size_t)b * R + i) * g.topk, nullptr);
  }
  if (!LOCAL_K) cluster.sync();  // keep km alive until every peer is done
}

// Grid (CL, B), cluster (CL, 1, 1), NT threads: route_cta for image blockIdx.y.
// At most 64 registers a thread (4 CTAs of 256 or one of 1024 per SM), except
// for grids of more than 256 regions, whose rows keep more values a lane.
template <typename T, int MAXJ, bool LOCAL_K, int NT, int SW>
__global__ void __launch_bounds__(NT, (MAXJ <= 8 ? 65536 / (64 * NT) : 1))
    bra_route_kernel(const T *__restrict__ q, const T *__restrict__ k, RouteGeom g,
                     int32_t *__restrict__ idx, float *__restrict__ affinity) {
  // A dependent grid launched with programmatic serialization may start now;
  // it waits for this grid before it reads the routing index.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ __align__(16) uint8_t route_smem[];
  route_cta<T, MAXJ, LOCAL_K, NT, SW>(q, k, g, idx, affinity, route_smem, (int)blockIdx.y);
}

}  // namespace bra

// route.cuh -- region-level routing of BRA on sm_103a.
//
// Computes, per image, the region means of Q and K, the region affinity
// A = mean(q_r) mean(k_r)^T over all C channels and the top-k regions of each
// row (page "CVPR2023：BiFormer中的双层路由注意力机制解析" §3: q_r = q.mean,
// A_r = q_r k_r^T, I_r = topk(A_r); page "从静态到动态：BRA双层路由注意力
// 如何革新视觉Transformer的计算范式" §2 mean pooling and §4 TopkRouting).
//
// One thread-block cluster per image. Each CTA of the cluster pools a share
// of the regions (regions r with r % CL == rank) into its shared memory, the
// cluster synchronises, every CTA copies all K means out of its peers' shared
// memory (distributed shared memory; for grids too large to copy, it reads
// them from the peers in place), and then computes the affinity rows and the
// top-k of its own query regions. Nothing goes through global memory but
// the inputs and the outputs. Arithmetic is float32 with FMA in a fixed
// channel order.
#pragma once

#include <cooperative_groups.h>

#include "ptx.cuh"

namespace bra {

namespace cg = cooperative_groups;

constexpr int kRouteThreads = 256;
constexpr int kRouteMaxCluster = 8;

template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void load(const float *p, float (&o)[4]) {
    float4 v = __ldg(reinterpret_cast<const float4 *>(p));
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
};
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const __nv_bfloat16 *p, float (&o)[8]) {
    uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
    o[0] = bf16_lo(v.x); o[1] = bf16_hi(v.x);
    o[2] = bf16_lo(v.y); o[3] = bf16_hi(v.y);
    o[4] = bf16_lo(v.z); o[5] = bf16_hi(v.z);
    o[6] = bf16_lo(v.w); o[7] = bf16_hi(v.w);
  }
};

// Shared-memory floats of the route kernel: own Q and K means, plus (when
// the K means of all regions are copied locally) an [R][C+1] table.
struct RouteSmem {
  __host__ __device__ static size_t floats(int R, int C, int CL, bool local_k) {
    const size_t ro_max = (size_t)(R + CL - 1) / CL;
    return 2 * ro_max * C + (local_k ? (size_t)R * (C + 1) : 0);
  }
};

// Grid (CL, B), cluster (CL, 1, 1), kRouteThreads threads.
// MAXJ = ceil(R / 32): affinity values each lane keeps for the top-k.
// LOCAL_K: copy every K mean into local shared memory first (fast path);
// otherwise read them from the peers' shared memory in the affinity loop.
template <typename T, int MAXJ, bool LOCAL_K>
__global__ void __launch_bounds__(kRouteThreads)
    bra_route_kernel(const T *__restrict__ q, const T *__restrict__ k, int H,
                     int W, int C, int S, int topk, int32_t *__restrict__ idx,
                     float *__restrict__ affinity) {
  // A dependent grid launched with programmatic serialization may start now;
  // it waits for this grid before it reads the routing index.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.y;
  const int R = S * S, hr = H / S, wr = W / S, n = hr * wr;
  const int ro = (R - rank + CL - 1) / CL;  // regions rank, rank+CL, ...
  const int ro_max = (R + CL - 1) / CL;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kRouteThreads / 32;

  extern __shared__ __align__(16) float route_smem[];
  float *qm = route_smem;            // [ro_max][C] own query-region means
  float *km = qm + ro_max * C;       // [ro_max][C] own key-region means
  float *kall = km + ro_max * C;     // [R][C+1] all key-region means

  // ---- 1. region means of q and k: one warp per (tensor, owned region) ----
  constexpr int VEC = Vec16<T>::N;
  const int G = C / VEC;                       // 16-byte groups per token
  const int GW = G < 32 ? G : 32;              // lanes across channel groups
  int TL = 1;                                  // lanes across tokens (pow2)
  while (TL * 2 * GW <= 32) TL *= 2;
  const int tl = lane / GW, gl = lane % GW;
  const bool active = lane < TL * GW;
  const float inv_n = 1.0f / static_cast<float>(n);
  for (int task = warp; task < 2 * ro; task += kWarps) {
    const int tensor = task & 1, s = task >> 1;
    const int r = rank + CL * s;
    const int y0 = (r / S) * hr, x0 = (r % S) * wr;
    const T *src = (tensor ? k : q) + (size_t)b * H * W * C;
    float *dst = (tensor ? km : qm) + s * C;
    for (int g0 = 0; g0 < G; g0 += GW) {
      float acc[VEC];
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
      const int g = g0 + gl;
      if (active && g < G) {
#pragma unroll 8
        for (int t = tl; t < n; t += TL) {
          const int y = y0 + t / wr, x = x0 + t % wr;
          float v[VEC];
          Vec16<T>::load(src + ((size_t)y * W + x) * C + g * VEC, v);
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[e] += v[e];
        }
      }
      // sum the TL token lanes of each channel group (lanes gl, gl+GW, ...)
      for (int off = GW; off < TL * GW; off <<= 1)
#pragma unroll
        for (int e = 0; e < VEC; ++e)
          acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
      if (active && tl == 0 && g < G)
#pragma unroll
        for (int e = 0; e < VEC; ++e) dst[g * VEC + e] = acc[e] * inv_n;
    }
  }

  cluster.sync();

  // ---- 2. gather every region's K mean from the cluster ----
  if (LOCAL_K) {
    for (int e = threadIdx.x; e < R * C; e += kRouteThreads) {
      const int r = e / C, c = e % C;
      const float *peer = cluster.map_shared_rank(km, r % CL);
      kall[r * (C + 1) + c] = peer[(r / CL) * C + c];
    }
    cluster.sync();  // peers are done reading our km; kall complete
  }

  // ---- 3. affinity rows and top-k: one warp per owned query region ----
  for (int s = warp; s < ro; s += kWarps) {
    const int i = rank + CL * s;
    const float *qi = qm + s * C;
    float val[MAXJ];
#pragma unroll
    for (int t = 0; t < MAXJ; ++t) {
      const int j = lane + 32 * t;
      float a = -INFINITY;
      if (j < R) {
        const float *kj = LOCAL_K ? kall + j * (C + 1)
                                  : cluster.map_shared_rank(km, j % CL) + (j / CL) * C;
        float dot = 0.f;
        for (int c = 0; c < C; ++c) dot = fmaf(qi[c], kj[c], dot);
        if (affinity) affinity[((size_t)b * R + i) * R + j] = dot;
        a = (dot == dot) ? dot : -INFINITY;  // a NaN never wins
      }
      val[t] = a;
    }
    unsigned taken = 0;  // bit t: column lane + 32 t already chosen
    for (int m = 0; m < topk; ++m) {
      float bv = -INFINITY;
      int bj = 0x7fffffff;
#pragma unroll
      for (int t = 0; t < MAXJ; ++t) {
        const int j = lane + 32 * t;
        if (j < R && !((taken >> t) & 1u) &&
            (val[t] > bv || (val[t] == bv && j < bj))) {
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
      if (lane == 0) idx[((size_t)b * R + i) * topk + m] = bj;
    }
  }
  if (!LOCAL_K) cluster.sync();  // keep km alive until every peer is done
}

}  // namespace bra

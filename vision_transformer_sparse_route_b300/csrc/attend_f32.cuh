// attend_f32.cuh -- routed attention + LePE for float32 maps on sm_103a.
//
// Same operation as the bf16 kernel (page "CVPR2023：BiFormer中的双层路由
// 注意力机制解析" §3; LePE of page "从静态到动态：BRA双层路由注意力如何革新
// 视觉Transformer的计算范式" §4), in float32 on the FMA pipe so that it stays
// within 1e-4 of the double-precision definition (TF32 tensor cores would
// not). One CTA per query region: it copies the region's Q, the routed
// regions' K and V (the gather lives only in shared memory) and the V halo
// into shared memory; one warp per (query token, head) then computes the
// logits (lanes over keys), the softmax with warp reductions, the weighted
// sum of V (lanes over channels) and the LePE of the same channels.
#pragma once

#include "ptx.cuh"

namespace bra {

constexpr int kAttendF32Threads = 256;

struct AttendF32Geom {
  int H, W, C, S, heads, topk;
  int hr, wr, n, R;
  int halo_w, halo_h;
  int nk;        // topk * n keys per query
  float scale;   // d^-1/2
  // float offsets into shared memory
  int off_k, off_v, off_h, off_p;
};

// One (query token t, head h) of a region whose tiles sit in shared memory
// (sq [n][C], sk [nk][C + 1], sv [nk][C], sh halo [halo_h * halo_w][C]), by
// one warp: the logits with lanes over keys, the softmax with warp
// reductions, the weighted sum of V with lanes over channels and the LePE of
// the same channels; pw holds the warp's nk probabilities. (y0, x0) is the
// region's first token. KS = 0 takes the conv size from ks at run time (the
// same arithmetic in the same order).
template <int KS>
__device__ __forceinline__ void attend_f32_task(const float *sq, const float *sk, const float *sv,
                                                const float *sh, float *pw,
                                                const float *__restrict__ lepe_w,
                                                const float *__restrict__ lepe_b,
                                                float *__restrict__ out, const AttendF32Geom &g,
                                                int b, int y0, int x0, int t, int h, int ks,
                                                int lane) {
  const int C = g.C;
  const int K = KS ? KS : ks;
  const int d = C / g.heads;
  const float *qt = sq + t * C + h * d;
  // logits, lanes over keys: four interleaved partial dot products (channels
  // e = 0, 1, 2, 3 mod 4) added pairwise
  float mx = -INFINITY;
  for (int key = lane; key < g.nk; key += 32) {
    const float *kr = sk + key * (C + 1) + h * d;
    float p4[4] = {0.f, 0.f, 0.f, 0.f};
    int e = 0;
    for (; e + 4 <= d; e += 4)
#pragma unroll
      for (int z = 0; z < 4; ++z) p4[z] = fmaf(qt[e + z], kr[e + z], p4[z]);
    for (; e < d; ++e) p4[0] = fmaf(qt[e], kr[e], p4[0]);
    float dot = (p4[0] + p4[1]) + (p4[2] + p4[3]);
    dot *= g.scale;
    pw[key] = dot;
    mx = fmaxf(mx, dot);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float sum = 0.f;
  for (int key = lane; key < g.nk; key += 32) {
    const float p = expf(pw[key] - mx);
    pw[key] = p;
    sum += p;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float inv = 1.f / sum;
  __syncwarp();
  const int ty = t / g.wr, tx = t % g.wr;
  for (int e = lane; e < d; e += 32) {
    const int c = h * d + e;
    // P V: two interleaved partial sums (even and odd keys)
    float a2[2] = {0.f, 0.f};
    int key = 0;
    for (; key + 2 <= g.nk; key += 2) {
      a2[0] = fmaf(pw[key], sv[key * C + c], a2[0]);
      a2[1] = fmaf(pw[key + 1], sv[(key + 1) * C + c], a2[1]);
    }
    if (key < g.nk) a2[0] = fmaf(pw[key], sv[key * C + c], a2[0]);
    const float acc = a2[0] + a2[1];
    // LePE: one partial sum per kernel row u, then the bias and the rows in order
    float lr[7] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < 7; ++u) {
      if (u < K) {
#pragma unroll
        for (int w = 0; w < 7; ++w)
          if (w < K)
            lr[u] = fmaf(__ldg(lepe_w + ((size_t)c * K + u) * K + w),
                         sh[((ty + u) * g.halo_w + tx + w) * C + c], lr[u]);
      }
    }
    float lp = lepe_b ? __ldg(lepe_b + c) : 0.f;
#pragma unroll
    for (int u = 0; u < 7; ++u)
      if (u < K) lp += lr[u];
    out[(((size_t)b * g.H + y0 + ty) * g.W + x0 + tx) * C + c] = acc * inv + lp;
  }
  __syncwarp();
}

// Query region i of image b by one CTA of NT threads, shared memory at
// f32_smem (layout of AttendF32Geom, its probability rows for NT / 32 warps).
template <int KS, int NT>
__device__ __forceinline__ void attend_f32_region(const float *__restrict__ q,
                                                  const float *__restrict__ k,
                                                  const float *__restrict__ v,
                                                  const int32_t *idx,
                                                  const float *__restrict__ lepe_w,
                                                  const float *__restrict__ lepe_b,
                                                  float *__restrict__ out,
                                                  const AttendF32Geom &g, int b, int i,
                                                  float *f32_smem) {
  float *sq = f32_smem;           // [n][C]
  float *sk = f32_smem + g.off_k; // [nk][C + 1]
  float *sv = f32_smem + g.off_v; // [nk][C]
  float *sh = f32_smem + g.off_h; // [halo_h * halo_w][C]
  float *sp = f32_smem + g.off_p; // [warps][nk] probabilities

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int y0 = (i / g.S) * g.hr, x0 = (i % g.S) * g.wr;
  const int C = g.C, C4 = C / 4;
  constexpr int PAD = KS / 2;
  const float *qb = q + (size_t)b * g.H * g.W * C;
  const float *kb = k + (size_t)b * g.H * g.W * C;
  const float *vb = v + (size_t)b * g.H * g.W * C;

  // Q tile of this region
  for (int e = tid; e < g.n * C4; e += NT) {
    const int t = e / C4, c4 = e % C4;
    const int y = y0 + t / g.wr, x = x0 + t % g.wr;
    *reinterpret_cast<float4 *>(sq + t * C + 4 * c4) =
        __ldg(reinterpret_cast<const float4 *>(qb + ((size_t)y * g.W + x) * C) + c4);
  }
  // routed K and V, concatenated region by region
  for (int e = tid; e < g.nk * C4; e += NT) {
    const int key = e / C4, c4 = e % C4;
    const int m = key / g.n, t = key % g.n;
    const int j = __ldg(idx + ((size_t)b * g.R + i) * g.topk + m);
    float4 kv4 = make_float4(0.f, 0.f, 0.f, 0.f), vv4 = kv4;
    if (j >= 0 && j < g.R) {
      const int y = (j / g.S) * g.hr + t / g.wr, x = (j % g.S) * g.wr + t % g.wr;
      const size_t off = ((size_t)y * g.W + x) * C;
      kv4 = __ldg(reinterpret_cast<const float4 *>(kb + off) + c4);
      vv4 = __ldg(reinterpret_cast<const float4 *>(vb + off) + c4);
    } else if (t == 0 && c4 == 0) {
      atomicOr(&g_status, kStatusBadIndex);
    }
    float *kr = sk + key * (C + 1) + 4 * c4;
    kr[0] = kv4.x; kr[1] = kv4.y; kr[2] = kv4.z; kr[3] = kv4.w;
    *reinterpret_cast<float4 *>(sv + key * C + 4 * c4) = vv4;
  }
  // V halo with zero padding outside the image
  for (int e = tid; e < g.halo_h * g.halo_w * C4; e += NT) {
    const int ht = e / C4, c4 = e % C4;
    const int y = y0 - PAD + ht / g.halo_w, x = x0 - PAD + ht % g.halo_w;
    float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
    if (y >= 0 && y < g.H && x >= 0 && x < g.W)
      val = __ldg(reinterpret_cast<const float4 *>(vb + ((size_t)y * g.W + x) * C) + c4);
    *reinterpret_cast<float4 *>(sh + ht * C + 4 * c4) = val;
  }
  __syncthreads();

  for (int task = warp; task < g.n * g.heads; task += NT / 32)
    attend_f32_task<KS>(sq, sk, sv, sh, sp + warp * g.nk, lepe_w, lepe_b, out, g, b, y0, x0,
                        task / g.heads, task % g.heads, KS, lane);
}

// One CTA per query region (grid B * R).
template <int KS>
__global__ void __launch_bounds__(kAttendF32Threads)
    bra_attend_f32_kernel(const float *__restrict__ q,
                          const float *__restrict__ k,
                          const float *__restrict__ v,
                          const int32_t *__restrict__ idx,
                          const float *__restrict__ lepe_w,
                          const float *__restrict__ lepe_b,
                          float *__restrict__ out, AttendF32Geom g) {
  extern __shared__ __align__(16) float f32_smem[];
  attend_f32_region<KS, kAttendF32Threads>(q, k, v, idx, lepe_w, lepe_b, out, g,
                                            (int)blockIdx.x / g.R, (int)blockIdx.x % g.R,
                                            f32_smem);
}

}  // namespace bra

// backward.cuh -- the backward of attend (routed attention + LePE) with the
// routing held fixed (page "从静态到动态：BRA双层路由注意力如何革新视觉
// Transformer的计算范式" §4: TopkRouting with diff_routing=False passes no
// gradient to the routing). Given dout = dL/dout, for one query with softmax
// row P over its k*n routed keys, attention output O and D = dout . O:
//   dv[key] += P[key] dout,   dS[key] = P[key] (dout . v[key] - D),
//   dq += scale dS[key] k[key],   dk[key] += scale dS[key] q,
// and for the LePE (cross-correlation with zero padding): dv gains its
// transpose applied to dout, dw[c][u][s] = sum dout[y][x][c] v[y+u-p][x+s-p][c]
// and db[c] = sum dout[..][c]. Arithmetic is float32; the gradients are
// float32 and accumulated with atomic adds where several queries or rows
// meet (a key routed by several regions, the LePE weights).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace bra {

constexpr int kBwdThreads = 256;
constexpr int kBwdWarps = kBwdThreads / 32;

struct BwdGeom {
  int H, W, C, S, heads, topk;
  int hr, wr, n, R, d;
  int nk;         // topk * n keys a query
  int ds;         // row stride of the Q, dO, K and V tiles (d + 1 floats)
  int ps;         // row stride of P (nk + 1 floats)
  float scale;    // d^-1/2
  uint32_t off_do, off_k, off_v, off_p, off_d, off_tok;  // bytes into shared memory
};

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

// One CTA per (image b, query region i, head h): the region's Q and dout, the
// routed keys' K and V (float32, padded rows), P recomputed (the scaled
// logits, then one softmax per query over all routed keys), then dv and dk
// (atomic adds, one per key and channel) and dq (plain stores: a query
// belongs to one region). Out-of-range routing reads zero keys, as the
// forward does, sets the status word and sends no gradient to them.
template <typename T>
__global__ void __launch_bounds__(kBwdThreads)
    bra_attend_bwd_kernel(const T *__restrict__ q, const T *__restrict__ k,
                          const T *__restrict__ v, const int32_t *__restrict__ idx,
                          const T *__restrict__ dout, BwdGeom g, float *__restrict__ dq,
                          float *__restrict__ dk, float *__restrict__ dv) {
  extern __shared__ __align__(16) uint8_t bwd_smem[];
  float *sq = reinterpret_cast<float *>(bwd_smem);                 // [n][ds]
  float *sdo = reinterpret_cast<float *>(bwd_smem + g.off_do);     // [n][ds]
  float *sk = reinterpret_cast<float *>(bwd_smem + g.off_k);       // [nk][ds]
  float *sv = reinterpret_cast<float *>(bwd_smem + g.off_v);       // [nk][ds]
  float *sp = reinterpret_cast<float *>(bwd_smem + g.off_p);       // [n][ps]
  float *sd = reinterpret_cast<float *>(bwd_smem + g.off_d);       // [n]
  int *ktok = reinterpret_cast<int *>(bwd_smem + g.off_tok);       // [nk], -1: none
  int *qtok = ktok + g.nk;                                         // [n]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x % g.heads, i = (blockIdx.x / g.heads) % g.R;
  const int b = blockIdx.x / (g.heads * g.R);
  const int n = g.n, nk = g.nk, d = g.d;
  const size_t img = (size_t)b * g.H * g.W;

  // token of every query and key (image-relative), -1 for out-of-range keys
  for (int e = tid; e < n + nk; e += kBwdThreads) {
    if (e < n) {
      const int y = (i / g.S) * g.hr + e / g.wr, x = (i % g.S) * g.wr + e % g.wr;
      qtok[e] = y * g.W + x;
    } else {
      const int a = e - n, m = a / n, t = a - m * n;
      const int j = __ldg(idx + ((size_t)b * g.R + i) * g.topk + m);
      if (j < 0 || j >= g.R) {
        atomicOr(&g_status, kStatusBadIndex);
        ktok[a] = -1;
      } else {
        const int y = (j / g.S) * g.hr + t / g.wr, x = (j % g.S) * g.wr + t % g.wr;
        ktok[a] = y * g.W + x;
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < n * d; e += kBwdThreads) {
    const int t = e / d, c = e - t * d;
    const size_t o = (img + qtok[t]) * g.C + h * d + c;
    sq[t * g.ds + c] = to_f32(q[o]);
    sdo[t * g.ds + c] = to_f32(dout[o]);
  }
  for (int e = tid; e < nk * d; e += kBwdThreads) {
    const int a = e / d, c = e - a * d;
    float kv = 0.f, vv = 0.f;
    if (ktok[a] >= 0) {
      const size_t o = (img + ktok[a]) * g.C + h * d + c;
      kv = to_f32(k[o]);
      vv = to_f32(v[o]);
    }
    sk[a * g.ds + c] = kv;
    sv[a * g.ds + c] = vv;
  }
  __syncthreads();

  // scaled logits, one thread per (query, key)
  for (int e = tid; e < n * nk; e += kBwdThreads) {
    const int t = e / nk, a = e - t * nk;
    float s = 0.f;
    for (int c = 0; c < d; ++c) s = fmaf(sq[t * g.ds + c], sk[a * g.ds + c], s);
    sp[t * g.ps + a] = s * g.scale;
  }
  __syncthreads();
  // softmax of each query's row (a warp a row), then O and D = dout . O
  for (int t = warp; t < n; t += kBwdWarps) {
    float *row = sp + t * g.ps;
    float m = -INFINITY;
    for (int a = lane; a < nk; a += 32) m = fmaxf(m, row[a]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float sum = 0.f;
    for (int a = lane; a < nk; a += 32) {
      const float p = __expf(row[a] - m);
      row[a] = p;
      sum += p;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    const float inv = 1.f / sum;
    for (int a = lane; a < nk; a += 32) row[a] *= inv;
    __syncwarp();
    float dd = 0.f;
    for (int c = lane; c < d; c += 32) {
      float o = 0.f;
      for (int a = 0; a < nk; ++a) o = fmaf(row[a], sv[a * g.ds + c], o);
      dd = fmaf(sdo[t * g.ds + c], o, dd);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, off);
    if (lane == 0) sd[t] = dd;
  }
  __syncthreads();
  // dv[key] = sum_t P[t][key] dout[t], one thread per (key, channel)
  for (int e = tid; e < nk * d; e += kBwdThreads) {
    const int a = e / d, c = e - a * d;
    if (ktok[a] < 0) continue;
    float acc = 0.f;
    for (int t = 0; t < n; ++t) acc = fmaf(sp[t * g.ps + a], sdo[t * g.ds + c], acc);
    atomicAdd(dv + (img + ktok[a]) * g.C + h * d + c, acc);
  }
  __syncthreads();
  // dS = P (dout . v[key] - D), in place of P, one thread per (query, key)
  for (int e = tid; e < n * nk; e += kBwdThreads) {
    const int t = e / nk, a = e - t * nk;
    float dp = 0.f;
    for (int c = 0; c < d; ++c) dp = fmaf(sdo[t * g.ds + c], sv[a * g.ds + c], dp);
    sp[t * g.ps + a] = sp[t * g.ps + a] * (dp - sd[t]);
  }
  __syncthreads();
  // dq = scale dS k (each query once), dk = scale dS^T q (atomic)
  for (int e = tid; e < n * d; e += kBwdThreads) {
    const int t = e / d, c = e - t * d;
    float acc = 0.f;
    for (int a = 0; a < nk; ++a) acc = fmaf(sp[t * g.ps + a], sk[a * g.ds + c], acc);
    dq[(img + qtok[t]) * g.C + h * d + c] = acc * g.scale;
  }
  for (int e = tid; e < nk * d; e += kBwdThreads) {
    const int a = e / d, c = e - a * d;
    if (ktok[a] < 0) continue;
    float acc = 0.f;
    for (int t = 0; t < n; ++t) acc = fmaf(sp[t * g.ps + a], sq[t * g.ds + c], acc);
    atomicAdd(dk + (img + ktok[a]) * g.C + h * d + c, acc * g.scale);
  }
}

// The LePE's part, one CTA per image row (b, y), one thread per channel:
// dv[y][x][c] += sum_{u,s} w[c][u][s] dout[y-u+p][x-s+p][c] (a plain add:
// this grid runs after the attention's and owns each element), and the row's
// sums of dout[y][x][c] v[y+u-p][x+s-p][c] and of dout, added to dw and db.
template <typename T, int KS>
__global__ void __launch_bounds__(1024)
    bra_lepe_bwd_kernel(const T *__restrict__ v, const float *__restrict__ w,
                        const T *__restrict__ dout, int H, int W, int C,
                        float *__restrict__ dv, float *__restrict__ dw,
                        float *__restrict__ db) {
  constexpr int PAD = KS / 2;
  const int c = threadIdx.x, y = blockIdx.x % H, b = blockIdx.x / H;
  if (c >= C) return;
  float wt[KS * KS], gw[KS * KS];
#pragma unroll
  for (int e = 0; e < KS * KS; ++e) {
    wt[e] = __ldg(w + (size_t)c * KS * KS + e);
    gw[e] = 0.f;
  }
  float gb = 0.f;
  const size_t img = (size_t)b * H * W;
  for (int x = 0; x < W; ++x) {
    const float go = to_f32(dout[(img + (size_t)y * W + x) * C + c]);
    gb += go;
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < KS; ++u) {
      const int yy = y + u - PAD;  // input row of tap u for output (y, x)
      const int yo = y - u + PAD;  // output row that reads (y, x) through tap u
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        const int xx = x + s - PAD, xo = x - s + PAD;
        if (yy >= 0 && yy < H && xx >= 0 && xx < W)
          gw[u * KS + s] = fmaf(go, to_f32(v[(img + (size_t)yy * W + xx) * C + c]), gw[u * KS + s]);
        if (yo >= 0 && yo < H && xo >= 0 && xo < W)
          acc = fmaf(wt[u * KS + s], to_f32(dout[(img + (size_t)yo * W + xo) * C + c]), acc);
      }
    }
    dv[(img + (size_t)y * W + x) * C + c] += acc;
  }
#pragma unroll
  for (int e = 0; e < KS * KS; ++e) atomicAdd(dw + (size_t)c * KS * KS + e, gw[e]);
  if (db) atomicAdd(db + c, gb);
}

}  // namespace bra

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
  int vec4;       // d % 4 == 0 and dq, dk, dv 16-byte aligned: 16-byte stores and atomics
  uint32_t off_do, off_k, off_v, off_p, off_g, off_d, off_tok;  // bytes into shared memory
};

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

// out[i][j] = sum_r a[i * as_i + r * as_r] b[j * bs_j + r * bs_r] for i < M,
// j < N over shared-memory operands, all threads of the CTA: each thread
// computes 4 x 4 blocks of out in registers (eight loads feed sixteen FMAs)
// and hands each row of a block to consume(i, j0, vals, count): out[i][j0 +
// e] = vals[e] for e < count (count < 4 only at the right edge).
template <typename F>
__device__ __forceinline__ void smem_gemm4x4(const float *a, int as_i, int as_r, const float *b,
                                             int bs_j, int bs_r, int M, int N, int R, int tid,
                                             F &&consume) {
  const int tm = (M + 3) / 4, tn = (N + 3) / 4;
  for (int e = tid; e < tm * tn; e += kBwdThreads) {
    const int i0 = (e / tn) * 4, j0 = (e % tn) * 4;
    int ia[4], jb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      ia[u] = min(i0 + u, M - 1) * as_i;
      jb[u] = min(j0 + u, N - 1) * bs_j;
    }
    float acc[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int w = 0; w < 4; ++w) acc[u][w] = 0.f;
    for (int r = 0; r < R; ++r) {
      float av[4], bv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        av[u] = a[ia[u] + r * as_r];
        bv[u] = b[jb[u] + r * bs_r];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int w = 0; w < 4; ++w) acc[u][w] = fmaf(av[u], bv[w], acc[u][w]);
    }
    const int count = min(4, N - j0);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i0 + u < M) consume(i0 + u, j0, acc[u], count);
  }
}

// Adds vals[0 .. count-1] to dst[0 .. count-1]: one 16-byte vector atomic
// when the four are there and vec4 (dst 16-byte aligned), else one a value.
__device__ __forceinline__ void atomic_add_row(float *dst, const float (&vals)[4], int count,
                                               float scale, bool vec4) {
  if (vec4 && count == 4) {
    atomicAdd(reinterpret_cast<float4 *>(dst),
              make_float4(vals[0] * scale, vals[1] * scale, vals[2] * scale, vals[3] * scale));
  } else {
    for (int e = 0; e < count; ++e) atomicAdd(dst + e, vals[e] * scale);
  }
}

// One CTA per (image b, query region i, head h): the region's Q and dout, the
// routed keys' K and V (float32, padded rows), then, each contraction by
// smem_gemm4x4: the scaled logits and one softmax per query over all routed
// keys (P); dP = dout V^T; D = sum_key P dP (which is dout . O); dv = P^T dout
// (atomic adds, one per key and channel); dS = P (dP - D) in dP's place;
// dq = scale dS K (plain stores: a query belongs to one region) and dk =
// scale dS^T Q (atomic adds). Out-of-range routing reads zero keys, as the
// forward does, sets the status word and sends no gradient to them. D and NK,
// when not zero, fix the head dimension and the keys a query at compile time
// (the strides and loop bounds of the contractions then fold).
template <typename T, int D, int NK>
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
  float *sp = reinterpret_cast<float *>(bwd_smem + g.off_p);       // [n][ps]: P
  float *sg = reinterpret_cast<float *>(bwd_smem + g.off_g);       // [n][ps]: dP, then dS
  float *sd = reinterpret_cast<float *>(bwd_smem + g.off_d);       // [n]
  int *ktok = reinterpret_cast<int *>(bwd_smem + g.off_tok);       // [nk], -1: none
  int *qtok = ktok + g.nk;                                         // [n]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x % g.heads, i = (blockIdx.x / g.heads) % g.R;
  const int b = blockIdx.x / (g.heads * g.R);
  const int n = g.n;
  const int nk = NK ? NK : g.nk, ps = NK ? NK + 1 : g.ps;
  const int d = D ? D : g.d, ds = D ? D + 1 : g.ds;
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
    sq[t * ds + c] = to_f32(q[o]);
    sdo[t * ds + c] = to_f32(dout[o]);
  }
  for (int e = tid; e < nk * d; e += kBwdThreads) {
    const int a = e / d, c = e - a * d;
    float kv = 0.f, vv = 0.f;
    if (ktok[a] >= 0) {
      const size_t o = (img + ktok[a]) * g.C + h * d + c;
      kv = to_f32(k[o]);
      vv = to_f32(v[o]);
    }
    sk[a * ds + c] = kv;
    sv[a * ds + c] = vv;
  }
  __syncthreads();

  // scaled logits S = scale Q K^T and dP = dout V^T ([n][nk] each)
  smem_gemm4x4(sq, ds, 1, sk, ds, 1, n, nk, d, tid,
               [&](int t, int a0, const float (&x)[4], int cnt) {
                 for (int e = 0; e < cnt; ++e) sp[t * ps + a0 + e] = x[e] * g.scale;
               });
  smem_gemm4x4(sdo, ds, 1, sv, ds, 1, n, nk, d, tid,
               [&](int t, int a0, const float (&x)[4], int cnt) {
                 for (int e = 0; e < cnt; ++e) sg[t * ps + a0 + e] = x[e];
               });
  __syncthreads();
  // softmax of each row of S (a warp a row), then D = sum_key P dP
  for (int t = warp; t < n; t += kBwdWarps) {
    float *row = sp + t * ps;
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
    float dd = 0.f;
    for (int a = lane; a < nk; a += 32) {
      const float p = row[a] * inv;
      row[a] = p;
      dd = fmaf(p, sg[t * ps + a], dd);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, off);
    if (lane == 0) sd[t] = dd;
  }
  __syncthreads();
  // dv = P^T dout ([nk][d], atomic); dS = P (dP - D) in dP's place
  smem_gemm4x4(sp, 1, ps, sdo, 1, ds, nk, d, n, tid,
               [&](int a, int c0, const float (&x)[4], int cnt) {
                 if (ktok[a] >= 0)
                   atomic_add_row(dv + (img + ktok[a]) * g.C + h * d + c0, x, cnt, 1.f, g.vec4);
               });
  for (int e = tid; e < n * nk; e += kBwdThreads) {
    const int t = e / nk, a = e - t * nk;
    sg[t * ps + a] = sp[t * ps + a] * (sg[t * ps + a] - sd[t]);
  }
  __syncthreads();
  // dq = scale dS K (each query once), dk = scale dS^T Q (atomic)
  smem_gemm4x4(sg, ps, 1, sk, 1, ds, n, d, nk, tid,
               [&](int t, int c0, const float (&x)[4], int cnt) {
                 float *dst = dq + (img + qtok[t]) * g.C + h * d + c0;
                 if (g.vec4 && cnt == 4)
                   *reinterpret_cast<float4 *>(dst) =
                       make_float4(x[0] * g.scale, x[1] * g.scale, x[2] * g.scale, x[3] * g.scale);
                 else
                   for (int e = 0; e < cnt; ++e) dst[e] = x[e] * g.scale;
               });
  smem_gemm4x4(sg, 1, ps, sq, 1, ds, nk, d, n, tid,
               [&](int a, int c0, const float (&x)[4], int cnt) {
                 if (ktok[a] >= 0)
                   atomic_add_row(dk + (img + ktok[a]) * g.C + h * d + c0, x, cnt, g.scale,
                                  g.vec4);
               });
}

// The LePE's part, one CTA per image row (b, y): thread (c, xp) takes
// channel c (c = threadIdx.x % C) at the row's columns x = xp, xp + XP, ...
// (XP = blockDim.x / C): dv[y][x][c] += sum_{u,s} w[c][u][s]
// dout[y-u+p][x-s+p][c] (a plain add: this grid runs after the attention's
// and owns each element), and its sums of dout[y][x][c] v[y+u-p][x+s-p][c]
// and of dout; the XP partial sums of a channel are added in shared memory,
// then to dw and db. blockDim.x is a multiple of C (C <= NT) or NT with the
// channels in turns of NT.
template <int KS>
__host__ __device__ constexpr int lepe_bwd_threads() {
  return KS >= 7 ? 128 : kBwdThreads;  // the partial sums fit in static shared memory
}

template <typename T, int KS>
__global__ void __launch_bounds__(lepe_bwd_threads<KS>())
    bra_lepe_bwd_kernel(const T *__restrict__ v, const float *__restrict__ w,
                        const T *__restrict__ dout, int H, int W, int C,
                        float *__restrict__ dv, float *__restrict__ dw,
                        float *__restrict__ db) {
  constexpr int PAD = KS / 2;
  __shared__ float part[lepe_bwd_threads<KS>()][KS * KS + 1];
  const int y = blockIdx.x % H, b = blockIdx.x / H;
  const size_t img = (size_t)b * H * W;
  const int cw = C < (int)blockDim.x ? C : (int)blockDim.x;  // channels a turn
  const int XP = blockDim.x / cw, xp = threadIdx.x / cw;
  for (int c0 = 0; c0 < C; c0 += cw) {
    const int c = c0 + threadIdx.x % cw;
    float wt[KS * KS], gw[KS * KS];
#pragma unroll
    for (int e = 0; e < KS * KS; ++e) {
      wt[e] = c < C ? __ldg(w + (size_t)c * KS * KS + e) : 0.f;
      gw[e] = 0.f;
    }
    float gb = 0.f;
    for (int x = xp; x < W && c < C; x += XP) {
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
            gw[u * KS + s] =
                fmaf(go, to_f32(v[(img + (size_t)yy * W + xx) * C + c]), gw[u * KS + s]);
          if (yo >= 0 && yo < H && xo >= 0 && xo < W)
            acc = fmaf(wt[u * KS + s], to_f32(dout[(img + (size_t)yo * W + xo) * C + c]), acc);
        }
      }
      dv[(img + (size_t)y * W + x) * C + c] += acc;
    }
#pragma unroll
    for (int e = 0; e < KS * KS; ++e) part[threadIdx.x][e] = gw[e];
    part[threadIdx.x][KS * KS] = gb;
    __syncthreads();
    if (xp == 0 && c < C) {
      for (int e = 0; e <= KS * KS; ++e) {
        float a = part[threadIdx.x][e];
        for (int o = 1; o < XP; ++o) a += part[threadIdx.x + o * cw][e];
        if (e < KS * KS)
          atomicAdd(dw + (size_t)c * KS * KS + e, a);
        else if (db)
          atomicAdd(db + c, a);
      }
    }
    __syncthreads();
  }
}

// The same LePE backward with the rows it reads staged in shared memory: the
// KS rows of dout and of v around row y (rows outside the image and the
// ks/2 columns on each side are zero), as [KS][W + 2 pad][C] in the input's
// type, then the taps as unconditional shared-memory reads. Same arithmetic
// and order as bra_lepe_bwd_kernel.
template <typename T, int KS>
__global__ void __launch_bounds__(lepe_bwd_threads<KS>())
    bra_lepe_bwd_staged_kernel(const T *__restrict__ v, const float *__restrict__ w,
                               const T *__restrict__ dout, int H, int W, int C,
                               float *__restrict__ dv, float *__restrict__ dw,
                               float *__restrict__ db) {
  constexpr int PAD = KS / 2;
  constexpr int EPV = 16 / sizeof(T);  // elements a 16-byte vector
  __shared__ float part[lepe_bwd_threads<KS>()][KS * KS + 1];
  extern __shared__ __align__(16) uint8_t lepe_smem[];
  const int WP = W + 2 * PAD;
  T *sg = reinterpret_cast<T *>(lepe_smem);  // dout rows y-pad .. y+pad
  T *sv = sg + (size_t)KS * WP * C;          // v rows y-pad .. y+pad
  const int y = blockIdx.x % H, b = blockIdx.x / H;
  const size_t img = (size_t)b * H * W;
  // stage both windows, 16 bytes a thread at a time (C * sizeof(T) is a
  // multiple of 16)
  const int vecs = KS * WP * C / EPV;
  for (int e = threadIdx.x; e < 2 * vecs; e += blockDim.x) {
    const int which = e / vecs, r = e - which * vecs;
    const int row = r / (WP * C / EPV), rest = r - row * (WP * C / EPV);
    const int xs = rest / (C / EPV), cv = rest - xs * (C / EPV);
    const int yy = y + row - PAD, xx = xs - PAD;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (yy >= 0 && yy < H && xx >= 0 && xx < W)
      val = __ldg(reinterpret_cast<const uint4 *>((which ? v : dout) +
                                                  (img + (size_t)yy * W + xx) * C) + cv);
    reinterpret_cast<uint4 *>(which ? sv : sg)[r] = val;
  }
  __syncthreads();
  const int cw = C < (int)blockDim.x ? C : (int)blockDim.x;  // channels a turn
  const int XP = blockDim.x / cw, xp = threadIdx.x / cw;
  for (int c0 = 0; c0 < C; c0 += cw) {
    const int c = c0 + threadIdx.x % cw;
    float wt[KS * KS], gw[KS * KS];
#pragma unroll
    for (int e = 0; e < KS * KS; ++e) {
      wt[e] = c < C ? __ldg(w + (size_t)c * KS * KS + e) : 0.f;
      gw[e] = 0.f;
    }
    float gb = 0.f;
    for (int x = xp; x < W && c < C; x += XP) {
      // window row u holds image row y + u - pad; column x + s of it holds
      // image column x + s - pad
      const float go = to_f32(sg[((size_t)PAD * WP + x + PAD) * C + c]);
      gb += go;
      float acc = 0.f;
#pragma unroll
      for (int u = 0; u < KS; ++u) {
#pragma unroll
        for (int s = 0; s < KS; ++s) {
          gw[u * KS + s] =
              fmaf(go, to_f32(sv[((size_t)u * WP + x + s) * C + c]), gw[u * KS + s]);
          // dout at (y - u + pad, x - s + pad): window row KS-1-u, column x + KS-1-s
          acc = fmaf(wt[u * KS + s],
                     to_f32(sg[((size_t)(KS - 1 - u) * WP + x + KS - 1 - s) * C + c]), acc);
        }
      }
      dv[(img + (size_t)y * W + x) * C + c] += acc;
    }
#pragma unroll
    for (int e = 0; e < KS * KS; ++e) part[threadIdx.x][e] = gw[e];
    part[threadIdx.x][KS * KS] = gb;
    __syncthreads();
    if (xp == 0 && c < C) {
      for (int e = 0; e <= KS * KS; ++e) {
        float a = part[threadIdx.x][e];
        for (int o = 1; o < XP; ++o) a += part[threadIdx.x + o * cw][e];
        if (e < KS * KS)
          atomicAdd(dw + (size_t)c * KS * KS + e, a);
        else if (db)
          atomicAdd(db + c, a);
      }
    }
    __syncthreads();
  }
}

}  // namespace bra

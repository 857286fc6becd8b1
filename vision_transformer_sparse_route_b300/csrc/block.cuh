// block.cuh -- the element-wise pieces of the BiFormer block around BRA (page
// "BiFormer架构核心思想解析" §3.1: x = x + self.bra(self.norm1(x)), then
// x = x + self.ffn(self.norm2(x))): the LayerNorm of every token over its
// channels, the residual add, and the ConvFFN's depthwise 3 x 3 convolution
// with the GELU after it. Each moves its data once (HBM-bound); the
// arithmetic is float32 with one rounding to bf16.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace bra {

constexpr int kLnThreads = 256;

__device__ __forceinline__ void unpack_bf16x8(const uint4 &u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// nn.LayerNorm over the C channels of each token: y = (x - mean) / sqrt(var +
// eps) * gamma + beta, biased variance, computed two-pass from registers.
// G = C / 8 lanes hold a token (one 16-byte chunk each, G in 8, 16, 32), so a
// warp normalises 32 / G tokens at once with coalesced loads and stores.
template <int G>
__global__ void __launch_bounds__(kLnThreads)
    bra_layer_norm_kernel(const __nv_bfloat16 *__restrict__ x, const float *__restrict__ gamma,
                          const float *__restrict__ beta, long long M, float eps,
                          __nv_bfloat16 *__restrict__ y) {
  constexpr int C = 8 * G;
  constexpr int TPW = 32 / G;  // tokens a warp
  const int lane = threadIdx.x & 31, sub = lane % G;
  const long long m = ((long long)blockIdx.x * (kLnThreads / 32) + (threadIdx.x >> 5)) * TPW +
                      lane / G;
  const bool live = m < M;
  float v[8];
  if (live) {
    unpack_bf16x8(__ldg(reinterpret_cast<const uint4 *>(x + m * C) + sub), v);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
  }
  float s = ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
#pragma unroll
  for (int off = G / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  const float mean = s * (1.0f / C);
  float d2 = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) d2 = fmaf(v[i] - mean, v[i] - mean, d2);
#pragma unroll
  for (int off = G / 2; off > 0; off >>= 1) d2 += __shfl_xor_sync(0xffffffffu, d2, off);
  const float rstd = rsqrtf(d2 * (1.0f / C) + eps);
  if (!live) return;
  const int c0 = 8 * sub;
  float o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float gi = gamma ? __ldg(gamma + c0 + i) : 1.f;
    const float bi = beta ? __ldg(beta + c0 + i) : 0.f;
    o[i] = fmaf((v[i] - mean) * rstd, gi, bi);
  }
  reinterpret_cast<uint4 *>(y + m * C)[sub] =
      make_uint4(pack2_bf16(o[0], o[1]), pack2_bf16(o[2], o[3]), pack2_bf16(o[4], o[5]),
                 pack2_bf16(o[6], o[7]));
}

// y = x + r element by element (n a multiple of 8), float32 sum rounded once
// to bf16; y may be r.
__global__ void __launch_bounds__(kLnThreads)
    bra_residual_add_kernel(const __nv_bfloat16 *__restrict__ x, const __nv_bfloat16 *r,
                            long long n8, __nv_bfloat16 *y) {
  for (long long i = (long long)blockIdx.x * kLnThreads + threadIdx.x; i < n8;
       i += (long long)gridDim.x * kLnThreads) {
    float a[8], b[8];
    unpack_bf16x8(__ldg(reinterpret_cast<const uint4 *>(x) + i), a);
    unpack_bf16x8(reinterpret_cast<const uint4 *>(r)[i], b);
    reinterpret_cast<uint4 *>(y)[i] =
        make_uint4(pack2_bf16(a[0] + b[0], a[1] + b[1]), pack2_bf16(a[2] + b[2], a[3] + b[3]),
                   pack2_bf16(a[4] + b[4], a[5] + b[5]), pack2_bf16(a[6] + b[6], a[7] + b[7]));
  }
}

// The ConvFFN's hidden layer: y = GELU(dwconv3x3(h) + bias) over Ch channels
// (Ch a multiple of 8), the depthwise 3 x 3 cross-correlation zero-padded by 1
// at the image border, GELU in its exact form x (1 + erf(x / sqrt 2)) / 2.
// A block takes an 8 x 8 tile of tokens (clipped at the image edge) and all
// channels: thread (chunk j, column cx) holds the 9 taps of its 8 channels in
// registers and slides down the tile's 8 rows, so each input it loads (10
// rows x 3 columns) feeds up to three outputs, and consecutive threads read
// and write consecutive 16-byte chunks of a token.
constexpr int kDwTile = 8;
constexpr int kDwMaxThreads = 384;  // Ch / 8 chunks x 8 columns, Ch up to 384

__global__ void __launch_bounds__(kDwMaxThreads, 1)
    bra_dwconv_gelu_kernel(const __nv_bfloat16 *__restrict__ h, const float *__restrict__ w,
                           const float *__restrict__ bias, int B, int H, int W, int Ch,
                           __nv_bfloat16 *__restrict__ y) {
  const int nch = Ch / 8;
  const int j = threadIdx.x % nch, cx = threadIdx.x / nch;  // chunk, tile column
  const int tiles_x = (W + kDwTile - 1) / kDwTile, tiles_y = (H + kDwTile - 1) / kDwTile;
  const int tile = blockIdx.x, b = tile / (tiles_x * tiles_y);
  const int x0 = (tile % tiles_x) * kDwTile, y0 = ((tile / tiles_x) % tiles_y) * kDwTile;
  const int x = x0 + cx;
  if (cx >= kDwTile || x >= W || b >= B) return;
  const int c0 = 8 * j;
  float wt[9][8], acc[kDwTile][8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
#pragma unroll
    for (int tap = 0; tap < 9; ++tap) wt[tap][i] = __ldg(w + (size_t)(c0 + i) * 9 + tap);
    const float bi = bias ? __ldg(bias + c0 + i) : 0.f;
#pragma unroll
    for (int r = 0; r < kDwTile; ++r) acc[r][i] = bi;
  }
  const __nv_bfloat16 *hb = h + (size_t)b * H * W * Ch + c0;
  // input row y0 - 1 + ir feeds output rows ir - dy (dy = 0, 1, 2)
#pragma unroll
  for (int ir = 0; ir < kDwTile + 2; ++ir) {
    const int sy = y0 - 1 + ir;
    if (sy < 0 || sy >= H) continue;
#pragma unroll
    for (int dx = 0; dx < 3; ++dx) {
      const int sx = x + dx - 1;
      if (sx < 0 || sx >= W) continue;
      float v[8];
      unpack_bf16x8(__ldg(reinterpret_cast<const uint4 *>(hb + ((size_t)sy * W + sx) * Ch)), v);
#pragma unroll
      for (int dy = 0; dy < 3; ++dy) {
        const int r = ir - dy;
        if (r < 0 || r >= kDwTile) continue;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[r][i] = fmaf(wt[dy * 3 + dx][i], v[i], acc[r][i]);
      }
    }
  }
  __nv_bfloat16 *yb = y + (size_t)b * H * W * Ch + c0;
#pragma unroll
  for (int r = 0; r < kDwTile; ++r) {
    const int oy = y0 + r;
    if (oy >= H) break;
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      o[i] = 0.5f * acc[r][i] * (1.0f + erff(acc[r][i] * 0.70710678118654752f));
    reinterpret_cast<uint4 *>(yb + ((size_t)oy * W + x) * Ch)[0] =
        make_uint4(pack2_bf16(o[0], o[1]), pack2_bf16(o[2], o[3]), pack2_bf16(o[4], o[5]),
                   pack2_bf16(o[6], o[7]));
  }
}

// The same convolution and GELU, persistent, with the input staged in shared
// memory: a CTA takes the tiles blockIdx.x, + gridDim.x, ... in turn; thread
// 0 copies each tile's (8 + 2) x (8 + 2) input tokens (NB boxes of Ch / NB
// channels, one TMA copy each, zero filled outside the image, which is the
// padding) into one of two buffers, the next tile's copy in flight while the
// current one is computed. Every thread (chunk j, column cx) keeps its
// channels' weights in registers for all the tiles and slides down a tile's
// rows reading its three input columns from shared memory (consecutive
// threads read consecutive 16-byte chunks of a token). The FMAs of a channel
// pair are paired (each half rounds as a single FMA), in the unstaged
// kernel's order.
constexpr int kDwIn = kDwTile + 2;  // input tile side

template <int NB>
__global__ void __launch_bounds__(kDwMaxThreads, 1)
    bra_dwconv_gelu_tma_kernel(const __grid_constant__ CUtensorMap tm_h,
                               const float *__restrict__ w, const float *__restrict__ bias,
                               int B, int H, int W, int Ch, __nv_bfloat16 *__restrict__ y) {
  extern __shared__ uint8_t dw_smem_raw[];
  uint8_t *smem = dw_smem_raw + ((128u - (smem_u32(dw_smem_raw) & 127u)) & 127u);
  const int cb = Ch / NB;  // channels a box
  const uint32_t box_bytes = kDwIn * kDwIn * cb * 2, buf_bytes = NB * box_bytes;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + 2 * buf_bytes);  // one a buffer
  const int nch = Ch / 8;
  const int j = threadIdx.x % nch, cx = threadIdx.x / nch;  // chunk, tile column
  const int tiles_x = (W + kDwTile - 1) / kDwTile, tiles_y = (H + kDwTile - 1) / kDwTile;
  const int tiles = B * tiles_x * tiles_y;
  auto issue = [&](int tile, int buf) {
    const int b = tile / (tiles_x * tiles_y);
    const int x0 = (tile % tiles_x) * kDwTile, y0 = ((tile / tiles_x) % tiles_y) * kDwTile;
    mbar_arrive_expect_tx(&bar[buf], buf_bytes);
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
      tma_load_4d(smem + buf * buf_bytes + nb * box_bytes, &tm_h, &bar[buf], nb * cb, x0 - 1,
                  y0 - 1, b);
  };
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
    if ((int)blockIdx.x < tiles) issue(blockIdx.x, 0);
  }
  const int c0 = 8 * j;
  float2 wt[9][4], bi[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int tap = 0; tap < 9; ++tap)
      wt[tap][i] = make_float2(__ldg(w + (size_t)(c0 + 2 * i) * 9 + tap),
                               __ldg(w + (size_t)(c0 + 2 * i + 1) * 9 + tap));
    bi[i] = bias ? make_float2(__ldg(bias + c0 + 2 * i), __ldg(bias + c0 + 2 * i + 1))
                 : make_float2(0.f, 0.f);
  }
  // chunk j's 16 bytes of input token (row 0, column cx) of a buffer
  const uint32_t col_ofs = (c0 / cb) * box_bytes + (uint32_t)(cx * cb + c0 % cb) * 2;
  int it = 0;
  for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++it) {
    const int buf = it & 1;
    __syncthreads();  // every thread is done with the other buffer (and the barriers exist)
    if (threadIdx.x == 0 && tile + (int)gridDim.x < tiles) {
      fence_async_shared();  // its reads before the copy that overwrites it
      issue(tile + gridDim.x, buf ^ 1);
    }
    mbar_wait(&bar[buf], (it >> 1) & 1);
    const int b = tile / (tiles_x * tiles_y);
    const int x0 = (tile % tiles_x) * kDwTile, y0 = ((tile / tiles_x) % tiles_y) * kDwTile;
    const int x = x0 + cx;
    if (x >= W) continue;
    float2 acc[kDwTile][4];
#pragma unroll
    for (int r = 0; r < kDwTile; ++r)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[r][i] = bi[i];
    const uint8_t *col = smem + buf * buf_bytes + col_ofs;
#pragma unroll
    for (int ir = 0; ir < kDwIn; ++ir) {
#pragma unroll
      for (int dx = 0; dx < 3; ++dx) {
        float v[8];
        unpack_bf16x8(*reinterpret_cast<const uint4 *>(col + (size_t)(ir * kDwIn + dx) * cb * 2),
                      v);
#pragma unroll
        for (int dy = 0; dy < 3; ++dy) {
          const int r = ir - dy;
          if (r < 0 || r >= kDwTile) continue;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            acc[r][i] = __ffma2_rn(wt[dy * 3 + dx][i], make_float2(v[2 * i], v[2 * i + 1]),
                                   acc[r][i]);
        }
      }
    }
    __nv_bfloat16 *yb = y + (size_t)b * H * W * Ch + c0;
#pragma unroll
    for (int r = 0; r < kDwTile; ++r) {
      const int oy = y0 + r;
      if (oy >= H) break;
      float o[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        o[2 * i] = 0.5f * acc[r][i].x * (1.0f + erff(acc[r][i].x * 0.70710678118654752f));
        o[2 * i + 1] = 0.5f * acc[r][i].y * (1.0f + erff(acc[r][i].y * 0.70710678118654752f));
      }
      reinterpret_cast<uint4 *>(yb + ((size_t)oy * W + x) * Ch)[0] =
          make_uint4(pack2_bf16(o[0], o[1]), pack2_bf16(o[2], o[3]), pack2_bf16(o[4], o[5]),
                     pack2_bf16(o[6], o[7]));
    }
  }
  if (threadIdx.x == 0) settle_after_timeout();
}

}  // namespace bra

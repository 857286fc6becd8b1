// bra.cu -- the C ABI of include/bra.h: argument checks, TMA tensor maps and
// kernel launches for the Bi-Level Routing Attention forward on sm_103a.
// All kernels live in this one translation unit so that they share the
// device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "bra.h"
#include "per_device.h"
#include "attend_bf16.cuh"
#include "attend_f32.cuh"
#include "attend_image.cuh"
#include "attend_tc.cuh"
#include "backward.cuh"
#include "block.cuh"
#include "qkv_tc.cuh"
#include "forward_image.cuh"
#include "route.cuh"

namespace {

using bra::AttendF32Geom;
using bra::AttendGeom;
using bra::FusedGeom;
using bra::ImageGeom;
using bra::TcGeom;

constexpr size_t kMaxSmemPerBlock = 227 * 1024;

inline int elem_size(int dtype) { return dtype == BRA_F32 ? 4 : 2; }

inline bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline bool overlap(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a);
  const uintptr_t y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

inline size_t round_up(size_t v, size_t m) { return (v + m - 1) / m * m; }

// Checks shared by every entry point. Returns BRA_OK or an error code.
int check_map_args(int B, int H, int W, int C, int S, int topk, int dtype) {
  if (B < 0 || H <= 0 || W <= 0 || C <= 0 || S <= 0 || topk <= 0)
    return BRA_ERR_INVALID_ARG;
  if (dtype != BRA_F32 && dtype != BRA_BF16) return BRA_ERR_INVALID_ARG;
  if (H % S || W % S) return BRA_ERR_INVALID_ARG;
  if ((long long)S * S < topk) return BRA_ERR_INVALID_ARG;
  if ((long long)B * H * W * C > (1ll << 40)) return BRA_ERR_UNSUPPORTED;
  return BRA_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? BRA_OK : BRA_ERR_CUDA; }

// ------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t,
                                  void *, const cuuint64_t *, const cuuint64_t *,
                                  const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [B, H, W, C] map of bf16 or f32; box = 128 bytes of channels x box_w x
// box_h x 1 image, zero fill outside the map; 128-byte swizzle for tiles
// read by ldmatrix.
bool make_map_t(CUtensorMap *m, const void *base, int dtype, int B, int H, int W, int C,
                int box_w, int box_h, bool swizzle, int box_c = 0) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t e = (cuuint64_t)elem_size(dtype);
  cuuint64_t dims[4] = {(cuuint64_t)C, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)C * e, (cuuint64_t)W * C * e,
                           (cuuint64_t)H * W * C * e};
  // box_c channels (default: 128 bytes of them); 64-byte rows take the
  // 64-byte swizzle
  const cuuint32_t bc = box_c ? (cuuint32_t)box_c : (cuuint32_t)(128 / e);
  cuuint32_t box[4] = {bc, (cuuint32_t)box_w, (cuuint32_t)box_h, 1};
  const CUtensorMapSwizzle sw = !swizzle ? CU_TENSOR_MAP_SWIZZLE_NONE
                                : bc * e == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_128B;
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, dtype == BRA_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
             4, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows][C] bf16 as a 2-D map; box = 64 channels x box_rows rows, 128-byte
// swizzle, zero fill past the last row.
bool make_map_2d(CUtensorMap *m, const void *base, int rows, int C, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)C * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map(CUtensorMap *m, const void *base, int B, int H, int W, int C,
              int box_w, int box_h, bool swizzle) {
  return make_map_t(m, base, BRA_BF16, B, H, W, C, box_w, box_h, swizzle);
}

// Raises a kernel's dynamic shared-memory limit to the per-block maximum,
// once per kernel and device (the attribute holds per device context).
cudaError_t allow_smem(const void *kernel, size_t bytes) {
  static bra::PerDeviceOnce once;
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (once.done(dev, kernel)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kMaxSmemPerBlock);
  if (e == cudaSuccess) once.mark(dev, kernel);
  return e;
}

// ------------------------------------------------------------------ route
int sm_count();
bool allow_wide_clusters(const void *kernel);

// 16-byte channel groups per token, if a power of two no larger than 32.
int route_groups(int C, int dtype) {
  const int bytes = C * elem_size(dtype);
  if (bytes % 16) return 0;
  const int G = bytes / 16;
  return (G <= 32 && (G & (G - 1)) == 0) ? G : 0;
}

// Plans the route kernel for a cluster of CL CTAs; false if it cannot run.
bool plan_route(int B, int H, int W, int C, int S, int topk, int dtype, int CL,
                bra::RouteGeom *g, size_t *smem, bool *local_k) {
  (void)B;
  bra::RouteGeom a = {};
  a.H = H; a.W = W; a.C = C; a.S = S; a.topk = topk;
  a.hr = H / S; a.wr = W / S; a.n = a.hr * a.wr; a.R = S * S;
  a.G = route_groups(C, dtype);
  if (!a.G) return false;
  const int ro_max = (a.R + CL - 1) / CL;
  const size_t means = (size_t)ro_max * C * 4;
  const size_t kall = (size_t)a.R * (C + 1) * 4;
  a.off_qm = 0;
  a.off_km = (uint32_t)means;
  a.off_kall = (uint32_t)round_up(2 * means, 16);
  // a local copy of all K means whenever it fits: remote reads in the
  // affinity loop cost far more than fewer CTAs per SM
  *local_k = a.off_kall + kall <= kMaxSmemPerBlock;
  *smem = a.off_kall + (*local_k ? kall : 0);
  // the owned rows of the affinity, staged for the top-k, when they fit
  const size_t aff = (size_t)ro_max * a.R * 4;
  a.off_aff = 0;
  if (*local_k && C % 4 == 0 &&
      *smem + aff <= std::min<size_t>(kMaxSmemPerBlock, *smem + 48 * 1024)) {
    a.off_aff = (uint32_t)round_up(*smem, 16);
    *smem = a.off_aff + aff;
  }
  *g = a;
  return *smem <= kMaxSmemPerBlock;
}

// Threads per route CTA: few clusters get 1024-thread CTAs.
int route_threads(int B, int CL) {
  return B * CL >= 2 * sm_count() ? bra::kRouteThreadsMany : bra::kRouteThreadsFew;
}

// Chunks of a region row per 32 lanes, when a whole multiple (1, 2 or 4), else 0.
int route_row_chunks(const bra::RouteGeom &g) {
  const int seg = g.wr * g.G;
  if (seg % 32) return 0;
  const int sw = seg / 32;
  return (sw == 1 || sw == 2 || sw == 4) ? sw : 0;
}

template <typename T, int MAXJ, bool LOCAL_K, int NT, int SW>
int launch_route_w(const void *q, const void *k, int B, int CL, const bra::RouteGeom &g,
                   size_t smem, int32_t *idx, float *aff, cudaStream_t s) {
  auto kern = bra::bra_route_kernel<T, MAXJ, LOCAL_K, NT, SW>;
  cudaError_t e = allow_smem(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) return BRA_ERR_CUDA;
  if (CL > 8 && !allow_wide_clusters(reinterpret_cast<const void *>(kern))) return BRA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, B, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, static_cast<const T *>(q), static_cast<const T *>(k), g,
                         idx, aff);
  return cuda_status(e);
}

template <typename T, int MAXJ, bool LOCAL_K, int NT>
int launch_route_n(const void *q, const void *k, int B, int CL, const bra::RouteGeom &g,
                   size_t smem, int32_t *idx, float *aff, cudaStream_t s) {
  switch (route_row_chunks(g)) {
    case 1: return launch_route_w<T, MAXJ, LOCAL_K, NT, 1>(q, k, B, CL, g, smem, idx, aff, s);
    case 2: return launch_route_w<T, MAXJ, LOCAL_K, NT, 2>(q, k, B, CL, g, smem, idx, aff, s);
    case 4: return launch_route_w<T, MAXJ, LOCAL_K, NT, 4>(q, k, B, CL, g, smem, idx, aff, s);
    default: return launch_route_w<T, MAXJ, LOCAL_K, NT, 0>(q, k, B, CL, g, smem, idx, aff, s);
  }
}

template <typename T, int MAXJ, bool LOCAL_K>
int launch_route_k(const void *q, const void *k, int B, int CL, const bra::RouteGeom &g,
                   size_t smem, int32_t *idx, float *aff, cudaStream_t s) {
  if (route_threads(B, CL) == bra::kRouteThreadsMany)
    return launch_route_n<T, MAXJ, LOCAL_K, bra::kRouteThreadsMany>(q, k, B, CL, g, smem, idx,
                                                                      aff, s);
  return launch_route_n<T, MAXJ, LOCAL_K, bra::kRouteThreadsFew>(q, k, B, CL, g, smem, idx,
                                                                   aff, s);
}

template <typename T, int MAXJ>
int launch_route_t(const void *q, const void *k, int B, int CL, const bra::RouteGeom &g,
                   size_t smem, bool local_k, int32_t *idx, float *aff, cudaStream_t s) {
  if (local_k) return launch_route_k<T, MAXJ, true>(q, k, B, CL, g, smem, idx, aff, s);
  return launch_route_k<T, MAXJ, false>(q, k, B, CL, g, smem, idx, aff, s);
}

template <typename T>
int launch_route_dtype(const void *q, const void *k, int B, int CL, const bra::RouteGeom &g,
                       size_t smem, bool local_k, int32_t *idx, float *aff, cudaStream_t s) {
  const int R = g.R;
  if (R <= 32) return launch_route_t<T, 1>(q, k, B, CL, g, smem, local_k, idx, aff, s);
  if (R <= 64) return launch_route_t<T, 2>(q, k, B, CL, g, smem, local_k, idx, aff, s);
  if (R <= 128) return launch_route_t<T, 4>(q, k, B, CL, g, smem, local_k, idx, aff, s);
  if (R <= 256) return launch_route_t<T, 8>(q, k, B, CL, g, smem, local_k, idx, aff, s);
  if (R <= 512) return launch_route_t<T, 16>(q, k, B, CL, g, smem, local_k, idx, aff, s);
  return launch_route_t<T, 32>(q, k, B, CL, g, smem, local_k, idx, aff, s);
}

// Lets a kernel use clusters of 16 CTAs (once per kernel and device).
bool allow_wide_clusters(const void *kernel) {
  static bra::PerDeviceOnce once;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (once.done(dev, kernel)) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
      cudaSuccess)
    return false;
  once.mark(dev, kernel);
  return true;
}

// Whether clusters of 16 route CTAs with this much shared memory can be
// resident on the current device (asked once per device, dtype and size).
bool wide_clusters_ok(int dtype, size_t smem) {
  struct Entry { int dev, dtype; size_t smem; bool ok; };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry &e : cache)
      if (e.dev == dev && e.dtype == dtype && e.smem == smem) return e.ok;
  }
  const void *kern = dtype == BRA_F32
      ? reinterpret_cast<const void *>(
            bra::bra_route_kernel<float, 8, true, bra::kRouteThreadsFew, 0>)
      : reinterpret_cast<const void *>(
            bra::bra_route_kernel<__nv_bfloat16, 8, true, bra::kRouteThreadsFew, 0>);
  int n = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(16, 1, 1);
  cfg.blockDim = dim3(bra::kRouteThreadsFew, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 16;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool ok = allow_smem(kern, smem) == cudaSuccess && allow_wide_clusters(kern) &&
                  cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0;
  (void)cudaGetLastError();
  std::lock_guard<std::mutex> lock(mu);
  cache.push_back({dev, dtype, smem, ok});
  return ok;
}

// Route CTAs of a cluster size that one SM holds at once: limited by threads,
// by the 64 registers a thread of the many-cluster shape and by shared memory
// (228 KB an SM, 1 KB of it reserved per CTA).
int route_ctas_per_sm(int B, int CL, size_t smem) {
  const int nt = route_threads(B, CL);
  const int by_smem = (int)(233472 / (smem + 1024));
  return std::min(std::min(2048 / nt, 65536 / (64 * nt)), by_smem);
}

// Cluster size: 16 when the batch is too small to fill the GPU with 8-CTA
// clusters and the device allows clusters of 16; otherwise the largest of 8,
// 4 and 2 CTAs per image whose whole grid is resident at once (the copy of all
// K means grows with C and limits CTAs per SM), else 8.
int route_cluster(int B, int R, int H, int W, int C, int S, int topk, int dtype) {
  const int CL = std::min(8, R);
  bra::RouteGeom g;
  size_t smem;
  bool lk;
  if (R >= 16 && B * 8 < sm_count()) {
    if (!plan_route(B, H, W, C, S, topk, dtype, 16, &g, &smem, &lk)) return CL;
    return wide_clusters_ok(dtype, smem) ? 16 : CL;
  }
  for (int cl = CL; cl >= 2; cl /= 2) {
    if (!plan_route(B, H, W, C, S, topk, dtype, cl, &g, &smem, &lk)) break;
    if ((long long)B * cl <= (long long)route_ctas_per_sm(B, cl, smem) * sm_count()) return cl;
  }
  return CL;
}

int check_route(const void *q, const void *k, int B, int H, int W, int C, int S,
                int topk, int dtype, const int32_t *idx) {
  int rc = check_map_args(B, H, W, C, S, topk, dtype);
  if (rc) return rc;
  if (B == 0) return BRA_OK;
  if (!q || !k || !idx) return BRA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k)) return BRA_ERR_INVALID_ARG;
  const int R = S * S;
  if (R > 1024 || B > 65535) return BRA_ERR_UNSUPPORTED;
  bra::RouteGeom g;
  size_t smem;
  bool lk;
  if (!plan_route(B, H, W, C, S, topk, dtype, std::min(8, R), &g, &smem, &lk))
    return BRA_ERR_UNSUPPORTED;
  return BRA_OK;
}

// The per-chunk routing kernel (forward_image.cuh): bf16, C / 64 in {1, 2,
// 4} CTAs a cluster, at most 64 regions of at most 8 tokens (the maps the
// local image kernel takes).
bool plan_route_chunked(int H, int W, int C, int S, int topk, bra::FusedGeom *fg,
                        size_t *smem) {
  if (C % 64 || S <= 0 || H % S || W % S) return false;
  bra::FusedGeom f = {};
  bra::ImageGeom &a = f.img;
  a.H = H; a.W = W; a.C = C; a.S = S; a.topk = topk;
  a.hr = H / S; a.wr = W / S; a.n = a.hr * a.wr; a.R = S * S;
  a.nc = C / 64;
  if (a.n > 8 || a.R > 64 || (a.nc != 1 && a.nc != 2 && a.nc != 4)) return false;
  const int G = route_groups(C, BRA_BF16);
  if (!G) return false;
  f.L = 32 / G;
  f.inv_n = 1.0f / static_cast<float>(a.n);
  f.rp = (a.R + 3) / 4 * 4;
  const size_t rows = (size_t)(a.R + a.nc - 1) / a.nc;
  f.off_qm = 0;
  f.off_km = f.off_qm + 64 * f.rp * 4;
  f.off_a = f.off_km + 64 * f.rp * 4;
  f.off_p = (uint32_t)round_up((size_t)f.off_a + rows * a.R * 4, 16);
  *smem = (size_t)f.off_p + (size_t)a.R * a.R * 4;
  *fg = f;
  return true;
}

int launch_route_chunked(const void *q, const void *k, int B, const bra::FusedGeom &f,
                         size_t smem, int32_t *idx, float *aff, cudaStream_t s) {
  auto kern = f.L == 1   ? bra::bra_route_chunked_kernel<1>
              : f.L == 2 ? bra::bra_route_chunked_kernel<2>
                         : bra::bra_route_chunked_kernel<4>;
  if (allow_smem(reinterpret_cast<const void *>(kern), smem) != cudaSuccess)
    return BRA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((size_t)B * f.img.nc), 1, 1);
  cfg.blockDim = dim3(bra::kRouteThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = f.img.nc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, static_cast<const __nv_bfloat16 *>(q),
                                        static_cast<const __nv_bfloat16 *>(k), f, idx, aff));
}

int launch_route(const void *q, const void *k, int B, int H, int W, int C, int S,
                 int topk, int dtype, int32_t *idx, float *aff, cudaStream_t s) {
  if (dtype == BRA_BF16) {
    bra::FusedGeom f;
    size_t smem;
    if (plan_route_chunked(H, W, C, S, topk, &f, &smem))
      return launch_route_chunked(q, k, B, f, smem, idx, aff, s);
  }
  const int CL = route_cluster(B, S * S, H, W, C, S, topk, dtype);
  bra::RouteGeom g;
  size_t smem;
  bool local_k;
  if (!plan_route(B, H, W, C, S, topk, dtype, CL, &g, &smem, &local_k)) return BRA_ERR_UNSUPPORTED;
  if (dtype == BRA_F32)
    return launch_route_dtype<float>(q, k, B, CL, g, smem, local_k, idx, aff, s);
  return launch_route_dtype<__nv_bfloat16>(q, k, B, CL, g, smem, local_k, idx, aff, s);
}

// ----------------------------------------------------------------- attend
bool lepe_ks_supported(int ks) { return ks == 1 || ks == 3 || ks == 5 || ks == 7; }

int sm_count() {
  static int counts[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!counts[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    counts[dev] = n;
  }
  return counts[dev];
}

int lepe_row_block(int hr) { return hr >= 8 ? 8 : hr >= 4 ? 4 : hr >= 2 ? 2 : 1; }

bool plan_attend_bf16(int B, int H, int W, int C, int heads, int S, int topk, int ks,
                      AttendGeom *g, size_t *smem) {
  if (C % 64 || C / heads != 32) return false;
  AttendGeom a = {};
  a.H = H; a.W = W; a.C = C; a.S = S; a.heads = heads; a.topk = topk;
  a.hr = H / S; a.wr = W / S; a.n = a.hr * a.wr; a.R = S * S;
  if (a.hr > 256 || a.wr + ks - 1 > 256 || a.hr + ks - 1 > 256) return false;
  a.nc = C / 64;
  a.slot = (int)round_up(a.n, 8);
  a.kv_rows = (int)round_up((size_t)topk * a.slot, 64);
  a.q_blocks = (a.n + 15) / 16;
  a.halo_w = a.wr + ks - 1;
  a.halo_h = a.hr + ks - 1;
  a.units = B * a.R;
  a.masked = (a.slot != a.n) || ((topk * a.slot) % 64 != 0);
  const int rb = lepe_row_block(a.hr);
  a.lepe_items = (C / 2) * a.wr * ((a.hr + rb - 1) / rb);
  a.q_chunk = (uint32_t)round_up((size_t)a.q_blocks * 16 * 128, 1024);
  a.kv_chunk = (uint32_t)a.kv_rows * 128u;
  a.h_chunk = (uint32_t)a.halo_w * a.halo_h * 128u;
  a.o_chunk = (uint32_t)a.n * 128u;
  a.tasks = heads * a.q_blocks;
  a.off_k = a.nc * a.q_chunk;
  a.off_v = a.off_k + a.nc * a.kv_chunk;
  a.off_h = a.off_v + a.nc * a.kv_chunk;
  const size_t halo_end = (size_t)a.off_h + (size_t)a.nc * a.h_chunk;
  const size_t o_bytes = round_up((size_t)a.n * C * 4, 1024);
  // O may overwrite the unit's Q/K/V once attention is done with them, unless
  // padded K/V rows must stay zero or a warp would have to hold more than one
  // task's O
  a.alias = !a.masked && a.tasks <= bra::kGroupWarps && o_bytes <= a.off_h;
  if (a.alias) {
    a.off_o = 0;
    a.stage_bytes = (uint32_t)round_up(halo_end, 1024);
  } else {
    a.off_o = (uint32_t)round_up(halo_end, 1024);
    a.stage_bytes = (uint32_t)round_up((size_t)a.off_o + o_bytes, 1024);
  }
  a.tx_bytes = a.nc * (a.o_chunk * (1u + 2u * topk) + a.h_chunk);
  // about three box copies per issuing warp, at most four warps
  const int nbox = a.nc * (2 + 2 * topk);
  a.issue_warps = std::min(4, std::max(1, (nbox + 2) / 3));
  if (topk > 32 || nbox > 32 * a.issue_warps) a.issue_warps = 1;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt(32.0));
  const size_t out_bytes = round_up((size_t)bra::kGroups * 2 * a.nc * a.o_chunk, 1024);
  const size_t w_bytes = round_up((size_t)(ks * ks + 1) * C * 4, 16);
  const size_t bar_bytes = bra::kMaxStages * 8;
  const size_t budget = kMaxSmemPerBlock - 1024;
  const size_t fixed = out_bytes + w_bytes + bar_bytes;
  if (fixed + a.stage_bytes > budget) return false;
  a.stages = (int)std::min<size_t>(bra::kMaxStages, (budget - fixed) / a.stage_bytes);
  if (a.stages > 1) a.stages &= ~1;  // an even count: each group owns half
  a.off_out = (uint32_t)((size_t)a.stages * a.stage_bytes);
  a.off_w = (uint32_t)(a.off_out + out_bytes);
  a.off_bar = (uint32_t)(a.off_w + w_bytes);
  *smem = (size_t)a.off_bar + bar_bytes + 1024;  // slack to align the base to 1024 bytes
  *g = a;
  return *smem <= kMaxSmemPerBlock;
}

// The tensor-memory kernel: bf16, 8 x 8 regions, 64 channels (2 heads of
// 32), at most 4 routed regions (N = 64 topk columns of a tensor-memory
// slot), LePE kernel 1, 3 or 5. Ring depths are the deepest that fit in
// shared memory: K and V rings of 2 (else 1), a halo ring of 3 (else 2).
bool plan_attend_tc(int B, int H, int W, int C, int heads, int S, int topk, int ks,
                    TcGeom *g, size_t *smem) {
  if (C != 64 || heads != 2 || H / S != 8 || W / S != 8 || topk > 4) return false;
  if (ks != 1 && ks != 3 && ks != 5) return false;
  TcGeom a = {};
  a.H = H; a.W = W; a.S = S; a.topk = topk; a.R = S * S;
  a.units = B * a.R;
  a.halo_w = a.halo_h = 8 + ks - 1;
  a.h_bytes = (uint32_t)a.halo_w * a.halo_h * 128u;
  // one key block: P V also forms the row sums (N = 80), so a slot needs 80
  // columns
  a.sum_mma = topk == 1;
  a.slot_cols = a.sum_mma ? 128 : 64;
  while (a.slot_cols < (uint32_t)(64 * topk)) a.slot_cols *= 2;
  a.nslot = std::min(4, (int)(bra::kTcTmemCols / a.slot_cols));
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt(32.0));
  const size_t w_bytes = (size_t)(ks * ks + 1) * 64 * 4;
  const size_t bars = (size_t)bra::kBarCount * 8 + 16;
  const size_t tile = (size_t)topk * 8192;  // K or V tiles of one unit
  struct Depth { int nq, nh, nkv; };
  // Q and K rings equally deep (S needs both), the deepest that fit
  const Depth depths[] = {{4, 2, 4}, {3, 2, 3}, {4, 3, 2}, {4, 2, 2}, {3, 2, 2},
                          {2, 2, 2}, {3, 2, 1}, {2, 2, 1}};
  for (const Depth &dp : depths) {
      const int nkv = dp.nkv, nh = dp.nh;
      a.nq = dp.nq;
      a.nk = a.nv = nkv;
      a.nh = nh;
      a.off_h = (uint32_t)dp.nq * 12288u;
      a.off_k = (uint32_t)round_up((size_t)a.off_h + (size_t)nh * a.h_bytes, 1024);
      a.off_v = (uint32_t)(a.off_k + nkv * tile);
      a.off_ones = (uint32_t)(a.off_v + nkv * tile);
      a.off_p = a.off_ones + (a.sum_mma ? 8192u : 0u);
      a.off_o = a.off_p + 2 * 16384;
      a.off_st = a.off_o + 2 * 16384;
      a.off_w = a.off_st + 2 * 8192;
      a.off_bar = (uint32_t)round_up(a.off_w + w_bytes, 8);
      *smem = (size_t)a.off_bar + bars + 1024;  // slack to align the base to 1024 bytes
      if (*smem <= kMaxSmemPerBlock) {
        *g = a;
        return true;
      }
    }
  return false;
}

// The tcgen05 GEMM (qkv_tc.cuh): K and N multiples of 64 (N / 64 <= 12 for a
// resident W), the output split into tensors of ow channels. W stays resident
// in shared memory when it fits; ring depths are the deepest that fit.
bool plan_linear(int M, int K, int N, int ow, bra::QkvGeom *g, size_t *smem) {
  if (K % 64 || N % 64 || ow % 64 || N % ow || N / ow > 3 || K < 64 || M <= 0) return false;
  bra::QkvGeom a = {};
  a.M = M; a.K = K; a.N = N; a.ow = ow;
  a.ka = K / 64;
  a.nt = N / 64;
  a.tiles = (M + 127) / 128;
  const size_t x_stage = (size_t)a.ka * 16384, w_stage = (size_t)a.ka * 8192;
  const size_t tail = round_up((size_t)N * 4, 16) + bra::kQbCount * 8 + 16;
  struct Cfg { int nx, nw, ns, res; };
  // staging tiles: one to three for each epilogue warpgroup
  constexpr int E = bra::kQkvEpi;
  const Cfg cfgs[] = {{4, a.nt, 3 * E, 1}, {3, a.nt, 3 * E, 1}, {2, a.nt, 3 * E, 1},
                      {2, a.nt, 2 * E, 1}, {2, a.nt, E, 1},     {2, 3, 2 * E, 0},
                      {2, 3, E, 0},        {2, 2, E, 0},        {1, 3, E, 0},
                      {1, 2, E, 0},        {1, a.nt, E, 1},     {1, 1, E, 0}};
  for (const Cfg &c : cfgs) {
    if (c.res && a.nt > 12) continue;
    a.nx = c.nx; a.nw = c.nw; a.ns = c.ns; a.w_resident = c.res;
    a.gw = (c.res && a.nt % 3 == 0) ? 3 : 1;
    a.nacc = a.gw == 3 ? 2 : 4;
    a.off_w = (uint32_t)(c.nx * x_stage);
    a.off_st = (uint32_t)(a.off_w + c.nw * w_stage);
    a.off_b = a.off_st + (uint32_t)c.ns * 16384u;
    a.off_bar = (uint32_t)round_up(a.off_b + (size_t)N * 4, 16);
    *smem = (size_t)a.off_st + (size_t)c.ns * 16384 + tail + 1024;
    if (*smem <= kMaxSmemPerBlock) {
      *g = a;
      return true;
    }
  }
  return false;
}

// Enqueues the GEMM: outputs o[0..N/ow) of [M][ow] each, the residual (the
// layout of the single output) added when given.
int launch_linear(const void *x, const void *w, const float *bias, int M, int K, int N, int ow,
                  void *const *o, const void *res, cudaStream_t s) {
  bra::QkvGeom g;
  size_t smem;
  if (!plan_linear(M, K, N, ow, &g, &smem)) return BRA_ERR_UNSUPPORTED;
  CUtensorMap tx, tw;
  if (!make_map_2d(&tx, x, M, K, 128) || !make_map_2d(&tw, w, N, K, 64)) return BRA_ERR_CUDA;
  (void)cudaGetLastError();
  auto kern = res ? bra::bra_qkv_tc_kernel<true> : bra::bra_qkv_tc_kernel<false>;
  if (allow_smem(reinterpret_cast<const void *>(kern), smem) != cudaSuccess)
    return BRA_ERR_CUDA;
  const unsigned grid = (unsigned)std::min(g.tiles, sm_count());
  const int nout = N / ow;
  kern<<<grid, bra::kQkvThreads, smem, s>>>(
      tx, tw, bias, g, static_cast<__nv_bfloat16 *>(o[0]),
      static_cast<__nv_bfloat16 *>(nout > 1 ? o[1] : o[0]),
      static_cast<__nv_bfloat16 *>(nout > 2 ? o[2] : o[0]),
      static_cast<const __nv_bfloat16 *>(res));
  return cuda_status(cudaGetLastError());
}

// The image-resident kernel: bf16, regions of fewer than 16 tokens (a 16-row
// query block is then partly empty and a region's box copies are under 2 KB),
// and one 64-channel chunk of the whole image's Q, K, V, V halo and f32 O in
// shared memory.
bool plan_attend_image(int H, int W, int C, int heads, int S, int topk, int ks,
                       ImageGeom *g, size_t *smem) {
  if (C % 64 || C / heads != 32) return false;
  ImageGeom a = {};
  a.H = H; a.W = W; a.C = C; a.S = S; a.heads = heads; a.topk = topk;
  a.hr = H / S; a.wr = W / S; a.n = a.hr * a.wr; a.R = S * S;
  if (a.n >= 16) return false;
  a.halo_w = W + ks - 1;
  a.halo_h = H + ks - 1;
  if (a.halo_w > 256 || a.halo_h > 256) return false;  // TMA box limit
  a.nc = C / 64;
  a.nkeys = topk * a.n;
  a.q_blocks = 1;
  const size_t tokens = (size_t)H * W;
  a.tile = (uint32_t)round_up((tokens + 1) * 128, 1024);
  a.off_k = a.tile;
  a.off_v = 2 * a.tile;
  a.off_h = 3 * a.tile;
  a.off_o = (uint32_t)round_up((size_t)a.off_h + (size_t)a.halo_w * a.halo_h * 128, 16);
  a.off_w = (uint32_t)(a.off_o + tokens * 64 * 4);
  a.nkp = (int)round_up((size_t)a.nkeys, 64);
  a.off_tab = (uint32_t)round_up((size_t)a.off_w + (size_t)(ks * ks + 1) * 64 * 4, 16);
  a.off_bar = (uint32_t)round_up((size_t)a.off_tab + (size_t)a.R * a.nkp * 2, 8);
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt(32.0));
  *smem = (size_t)a.off_bar + 8 + 1024;  // slack to align the base to 1024 bytes
  *g = a;
  return *smem <= kMaxSmemPerBlock;
}

// The local form of the image kernel: regions of at most 8 tokens; the
// chunk of the whole image's K (swizzled tile), a zero-bordered V halo with
// 144-byte rows, the LePE weights, the two key tables and a staging area of
// n rows per warp in shared memory (Q is read from global memory, and there
// is no f32 O tile), so that two CTAs share an SM on the stage-3 shape.
// off_v holds the halo-position key table, off_o the staging area.
bool plan_attend_image_local(int H, int W, int C, int heads, int S, int topk, int ks,
                             ImageGeom *g, size_t *smem) {
  if (C % 64 || C / heads != 32) return false;
  ImageGeom a = {};
  a.H = H; a.W = W; a.C = C; a.S = S; a.heads = heads; a.topk = topk;
  a.hr = H / S; a.wr = W / S; a.n = a.hr * a.wr; a.R = S * S;
  if (a.n > 8) return false;
  a.halo_w = W + ks - 1;
  a.halo_h = H + ks - 1;
  if (a.halo_w > 256 || a.halo_h > 256) return false;  // TMA box limit
  a.nc = C / 64;
  a.nkeys = topk * a.n;
  a.q_blocks = 1;
  const size_t tokens = (size_t)H * W;
  const size_t halo = (size_t)a.halo_w * a.halo_h + 1;  // + the zero row
  if (halo > 65535) return false;                       // uint16 key tables
  a.tile = (uint32_t)round_up((tokens + 1) * 128, 1024);
  a.off_k = 0;
  a.off_h = a.tile;
  a.off_w = (uint32_t)round_up((size_t)a.off_h + halo * bra::kHaloPitch, 16);
  a.nkp = (int)round_up((size_t)a.nkeys, 64);
  a.off_tab = (uint32_t)round_up((size_t)a.off_w + (size_t)(ks * ks + 1) * 64 * 4, 16);
  a.off_v = (uint32_t)round_up((size_t)a.off_tab + (size_t)a.R * a.nkp * 2, 16);
  a.off_o = (uint32_t)round_up((size_t)a.off_v + (size_t)a.R * a.nkp * 2, 16);
  a.off_rt = (uint32_t)round_up(
      (size_t)a.off_o + (size_t)bra::kLocalWarps * a.n * bra::kStgStride * 4, 16);
  a.off_bar = (uint32_t)round_up((size_t)a.off_rt + (size_t)(2 * a.R + 16) * 2, 8);
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt(32.0));
  *smem = (size_t)a.off_bar + 8 + 1024;  // slack to align the base to 1024 bytes
  *g = a;
  return *smem <= kMaxSmemPerBlock;
}

// The one-launch forward on the local image kernel's layout: the local
// kernel's shapes with at most 64 regions and C / 64 in {1, 2, 4}; the
// routing's scratch (means, this CTA's affinity rows, the chunk's partial
// affinity) must fit in the V halo's space, and the routing ([R][topk]) and
// a second mbarrier go after the region tables.
bool plan_forward_local(int H, int W, int C, int heads, int S, int topk, int ks,
                        FusedGeom *fg, size_t *smem) {
  ImageGeom a;
  size_t s0;
  if (!plan_attend_image_local(H, W, C, heads, S, topk, ks, &a, &s0)) return false;
  const int G = route_groups(C, BRA_BF16);
  if (!G || a.R > 64 || (a.nc != 1 && a.nc != 2 && a.nc != 4)) return false;
  FusedGeom f = {};
  f.L = 32 / G;
  f.inv_n = 1.0f / static_cast<float>(a.n);
  f.rp = (a.R + 3) / 4 * 4;
  const size_t rows = (size_t)(a.R + a.nc - 1) / a.nc;
  f.off_qm = a.off_h;
  f.off_km = f.off_qm + 64 * f.rp * 4;
  f.off_a = f.off_km + 64 * f.rp * 4;
  f.off_p = (uint32_t)round_up((size_t)f.off_a + rows * a.R * 4, 16);
  const size_t scratch_end = (size_t)f.off_p + (size_t)a.R * a.R * 4;
  if (scratch_end > (size_t)a.off_h + (size_t)a.halo_w * a.halo_h * bra::kHaloPitch)
    return false;
  f.off_ridx = (uint32_t)round_up((size_t)a.off_rt + (size_t)(2 * a.R + 16) * 2, 16);
  a.off_bar = (uint32_t)round_up((size_t)f.off_ridx + (size_t)a.R * topk * 4, 8);
  f.off_bar = a.off_bar;
  f.img = a;
  *smem = (size_t)a.off_bar + 16 + 1024;  // slack to align the base to 1024 bytes
  *fg = f;
  return *smem <= kMaxSmemPerBlock;
}

// The one-launch forward (routing inside the image-resident attend kernel):
// bf16 maps the image kernel takes, at most 64 regions, and channel counts the
// routing kernel supports (C / 64 CTAs in a cluster per image: 1, 2 or 4).
bool plan_forward_image(int H, int W, int C, int heads, int S, int topk, int ks,
                        FusedGeom *fg, size_t *smem) {
  ImageGeom a;
  size_t s0;
  if (!plan_attend_image(H, W, C, heads, S, topk, ks, &a, &s0)) return false;
  const int G = route_groups(C, BRA_BF16);
  if (!G || a.R > 64 || (a.nc != 1 && a.nc != 2 && a.nc != 4)) return false;
  FusedGeom f = {};
  f.L = 32 / G;
  f.inv_n = 1.0f / static_cast<float>(a.n);
  const size_t tokens = (size_t)H * W;
  f.rp = (a.R + 3) / 4 * 4;
  // the routing scratch (means, this CTA's rows of the affinity) shares the
  // area of the f32 O tile, which is written only after the routing
  const size_t rows = (size_t)(a.R + a.nc - 1) / a.nc;
  const size_t routing = (size_t)2 * 64 * f.rp * 4 + rows * a.R * 4;
  f.off_qm = a.off_o;
  f.off_km = f.off_qm + 64 * f.rp * 4;
  f.off_a = f.off_km + 64 * f.rp * 4;
  a.off_w = (uint32_t)round_up((size_t)a.off_o + std::max(tokens * 64 * 4, routing), 16);
  a.off_tab = (uint32_t)round_up((size_t)a.off_w + (size_t)(ks * ks + 1) * 64 * 4, 16);
  f.off_p = (uint32_t)round_up((size_t)a.off_tab + (size_t)a.R * a.nkp * 2, 16);
  f.off_ridx = (uint32_t)round_up((size_t)f.off_p + (size_t)a.R * a.R * 4, 16);
  f.off_tok = (uint32_t)round_up((size_t)f.off_ridx + (size_t)a.R * topk * 4, 16);
  f.off_bar = (uint32_t)round_up((size_t)f.off_tok + (64 + 16) * 2, 8);
  a.off_bar = f.off_bar;
  f.img = a;
  *smem = (size_t)f.off_bar + 16 + 1024;  // slack to align the base to 1024 bytes
  *fg = f;
  return *smem <= kMaxSmemPerBlock;
}

bool plan_attend_f32(int H, int W, int C, int heads, int S, int topk, int ks,
                     AttendF32Geom *g, size_t *smem) {
  if (C % 4 || C / heads > 64) return false;
  AttendF32Geom a = {};
  a.H = H; a.W = W; a.C = C; a.S = S; a.heads = heads; a.topk = topk;
  a.hr = H / S; a.wr = W / S; a.n = a.hr * a.wr; a.R = S * S;
  a.halo_w = a.wr + ks - 1;
  a.halo_h = a.hr + ks - 1;
  a.nk = topk * a.n;
  a.scale = (float)(1.0 / std::sqrt((double)(C / heads)));
  size_t off = (size_t)a.n * C;
  a.off_k = (int)off; off += (size_t)a.nk * (C + 1);
  off = round_up(off, 4);
  a.off_v = (int)off; off += (size_t)a.nk * C;
  a.off_h = (int)off; off += (size_t)a.halo_w * a.halo_h * C;
  a.off_p = (int)off; off += (size_t)(bra::kAttendF32Threads / 32) * a.nk;
  *smem = off * sizeof(float);
  *g = a;
  return *smem <= kMaxSmemPerBlock;
}

template <int KS, int RB, int WR, int HR>
int launch_attend_bf16_kr(const void *q, const void *k, const void *v,
                          const int32_t *idx, int B, const float *w,
                          const float *bias, void *out, const AttendGeom &g,
                          size_t smem, bool pdl, cudaStream_t s) {
  CUtensorMap tq, tk, tv, th, to;
  if (!make_map(&tq, q, B, g.H, g.W, g.C, g.wr, g.hr, true) ||
      !make_map(&tk, k, B, g.H, g.W, g.C, g.wr, g.hr, true) ||
      !make_map(&tv, v, B, g.H, g.W, g.C, g.wr, g.hr, true) ||
      !make_map(&th, v, B, g.H, g.W, g.C, g.halo_w, g.halo_h, false) ||
      !make_map(&to, out, B, g.H, g.W, g.C, g.wr, g.hr, false))
    return BRA_ERR_CUDA;
  auto kern = bra::bra_attend_bf16_kernel<KS, RB, WR, HR>;
  if (allow_smem(reinterpret_cast<const void *>(kern), smem) != cudaSuccess)
    return BRA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min(g.units, sm_count()), 1, 1);
  cfg.blockDim = dim3(bra::kAttendThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, th, to, idx, w, bias, g));
}

template <int KS>
int launch_attend_bf16_ks(const void *q, const void *k, const void *v,
                          const int32_t *idx, int B, const float *w,
                          const float *bias, void *out, const AttendGeom &g,
                          size_t smem, bool pdl, cudaStream_t s) {
  // square regions of the stage shapes get their geometry at compile time
  if constexpr (KS == 5) {
    if (g.wr == g.hr && (g.wr == 8 || g.wr == 4 || g.wr == 2)) {
      switch (g.wr) {
      case 8: return launch_attend_bf16_kr<KS, 8, 8, 8>(q, k, v, idx, B, w, bias, out, g, smem, pdl, s);
      case 4: return launch_attend_bf16_kr<KS, 4, 4, 4>(q, k, v, idx, B, w, bias, out, g, smem, pdl, s);
      default: return launch_attend_bf16_kr<KS, 2, 2, 2>(q, k, v, idx, B, w, bias, out, g, smem, pdl, s);
      }
    }
  }
  switch (lepe_row_block(g.hr)) {
    case 8: return launch_attend_bf16_kr<KS, 8, 0, 0>(q, k, v, idx, B, w, bias, out, g, smem, pdl, s);
    case 4: return launch_attend_bf16_kr<KS, 4, 0, 0>(q, k, v, idx, B, w, bias, out, g, smem, pdl, s);
    case 2: return launch_attend_bf16_kr<KS, 2, 0, 0>(q, k, v, idx, B, w, bias, out, g, smem, pdl, s);
    default: return launch_attend_bf16_kr<KS, 1, 0, 0>(q, k, v, idx, B, w, bias, out, g, smem, pdl, s);
  }
}

template <int KS>
int launch_attend_tc_ks(const void *q, const void *k, const void *v, const int32_t *idx, int B,
                        int C, const float *w, const float *bias, void *out, const TcGeom &g,
                        size_t smem, bool pdl, cudaStream_t s) {
  CUtensorMap tq, tk, tv, th;
  if (!make_map_t(&tq, q, BRA_BF16, B, g.H, g.W, C, 8, 8, true, 32) ||
      !make_map(&tk, k, B, g.H, g.W, C, 8, 8, true) ||
      !make_map(&tv, v, B, g.H, g.W, C, 8, 8, true) ||
      !make_map(&th, v, B, g.H, g.W, C, g.halo_w, g.halo_h, false))
    return BRA_ERR_CUDA;
  auto kern = bra::bra_attend_tc_kernel<KS>;
  if (allow_smem(reinterpret_cast<const void *>(kern), smem) != cudaSuccess)
    return BRA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min(g.units, sm_count()), 1, 1);
  cfg.blockDim = dim3(bra::kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, th, idx, w, bias, g,
                                        static_cast<__nv_bfloat16 *>(out)));
}

template <int KS, int RB>
int launch_attend_image_kr(const void *q, const void *k, const void *v,
                           const int32_t *idx, int B, const float *w,
                           const float *bias, void *out, const ImageGeom &g,
                           size_t smem, bool pdl, cudaStream_t s) {
  CUtensorMap tq, tk, tv, th;
  if (!make_map(&tq, q, B, g.H, g.W, g.C, g.W, g.H, true) ||
      !make_map(&tk, k, B, g.H, g.W, g.C, g.W, g.H, true) ||
      !make_map(&tv, v, B, g.H, g.W, g.C, g.W, g.H, true) ||
      !make_map(&th, v, B, g.H, g.W, g.C, g.halo_w, g.halo_h, false))
    return BRA_ERR_CUDA;
  auto kern = bra::bra_attend_image_kernel<KS, RB>;
  if (allow_smem(reinterpret_cast<const void *>(kern), smem) != cudaSuccess)
    return BRA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((size_t)B * g.nc), 1, 1);
  cfg.blockDim = dim3(bra::kImgThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, th,
                                        static_cast<__nv_bfloat16 *>(out), idx, w, bias, g));
}

template <int KS, int HR, int WR>
int launch_attend_image_local_t(const void *q, const void *k, const void *v,
                                const int32_t *idx, int B, const float *w,
                                const float *bias, void *out, const ImageGeom &g,
                                size_t smem, bool pdl, cudaStream_t s) {
  CUtensorMap tk, tvh;
  // the halo's rows are 72 channels: the chunk's 64 and 8 that pad the row
  // to 144 bytes (past the last channel they read the zero fill)
  if (!make_map(&tk, k, B, g.H, g.W, g.C, g.W, g.H, true) ||
      !make_map_t(&tvh, v, BRA_BF16, B, g.H, g.W, g.C, g.halo_w, g.halo_h, false,
                  bra::kHaloPitch / 2))
    return BRA_ERR_CUDA;
  auto kern = bra::bra_attend_image_local_kernel<KS, HR, WR>;
  if (allow_smem(reinterpret_cast<const void *>(kern), smem) != cudaSuccess)
    return BRA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((size_t)B * g.nc), 1, 1);
  cfg.blockDim = dim3(bra::kLocalThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, tk, tvh,
                                        static_cast<const __nv_bfloat16 *>(q),
                                        static_cast<__nv_bfloat16 *>(out), idx, w, bias, g));
}

// 2 x 2 regions (the stage-3 shape) take the sliding-window LePE, other
// shapes of at most 8 tokens the token-by-token one
template <int KS>
int launch_attend_image_local(const void *q, const void *k, const void *v,
                              const int32_t *idx, int B, const float *w,
                              const float *bias, void *out, const ImageGeom &g,
                              size_t smem, bool pdl, cudaStream_t s) {
  if (g.hr == 2 && g.wr == 2)
    return launch_attend_image_local_t<KS, 2, 2>(q, k, v, idx, B, w, bias, out, g, smem, pdl,
                                                 s);
  return launch_attend_image_local_t<KS, 0, 0>(q, k, v, idx, B, w, bias, out, g, smem, pdl, s);
}

template <int KS>
int launch_attend_image_ks(const void *q, const void *k, const void *v,
                           const int32_t *idx, int B, const float *w,
                           const float *bias, void *out, const ImageGeom &g,
                           size_t smem, bool pdl, cudaStream_t s) {
  // LePE row blocks: 7 rows when they tile the map exactly, else 8
  if (g.H % 7 == 0)
    return launch_attend_image_kr<KS, 7>(q, k, v, idx, B, w, bias, out, g, smem, pdl, s);
  return launch_attend_image_kr<KS, 8>(q, k, v, idx, B, w, bias, out, g, smem, pdl, s);
}

template <int KS, int RB>
int launch_forward_image_kr(const void *q, const void *k, const void *v, int32_t *idx, int B,
                            const float *w, const float *bias, void *out, const FusedGeom &f,
                            size_t smem, cudaStream_t s) {
  const ImageGeom &g = f.img;
  CUtensorMap tq, tk, tv, th;
  if (!make_map(&tq, q, B, g.H, g.W, g.C, g.W, g.H, true) ||
      !make_map(&tk, k, B, g.H, g.W, g.C, g.W, g.H, true) ||
      !make_map(&tv, v, B, g.H, g.W, g.C, g.W, g.H, true) ||
      !make_map(&th, v, B, g.H, g.W, g.C, g.halo_w, g.halo_h, false))
    return BRA_ERR_CUDA;
  auto kern = bra::bra_forward_image_kernel<KS, RB>;
  if (allow_smem(reinterpret_cast<const void *>(kern), smem) != cudaSuccess)
    return BRA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((size_t)B * g.nc), 1, 1);
  cfg.blockDim = dim3(bra::kImgThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = g.nc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, th,
                                        static_cast<__nv_bfloat16 *>(out), idx, w, bias, f));
}

template <int KS, int HR, int WR, int L>
int launch_forward_local_t(const void *q, const void *k, const void *v, int32_t *idx, int B,
                           const float *w, const float *bias, void *out, const FusedGeom &f,
                           size_t smem, cudaStream_t s) {
  const ImageGeom &g = f.img;
  CUtensorMap tk, tvh;
  if (!make_map(&tk, k, B, g.H, g.W, g.C, g.W, g.H, true) ||
      !make_map_t(&tvh, v, BRA_BF16, B, g.H, g.W, g.C, g.halo_w, g.halo_h, false,
                  bra::kHaloPitch / 2))
    return BRA_ERR_CUDA;
  auto kern = bra::bra_forward_local_kernel<KS, HR, WR, L>;
  if (allow_smem(reinterpret_cast<const void *>(kern), smem) != cudaSuccess)
    return BRA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((size_t)B * g.nc), 1, 1);
  cfg.blockDim = dim3(bra::kLocalThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = g.nc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, tk, tvh,
                                        static_cast<const __nv_bfloat16 *>(q),
                                        static_cast<const __nv_bfloat16 *>(k),
                                        static_cast<__nv_bfloat16 *>(out), idx, w, bias, f));
}

template <int KS, int HR, int WR>
int launch_forward_local_l(const void *q, const void *k, const void *v, int32_t *idx, int B,
                           const float *w, const float *bias, void *out, const FusedGeom &f,
                           size_t smem, cudaStream_t s) {
  if (f.L == 1)
    return launch_forward_local_t<KS, HR, WR, 1>(q, k, v, idx, B, w, bias, out, f, smem, s);
  if (f.L == 2)
    return launch_forward_local_t<KS, HR, WR, 2>(q, k, v, idx, B, w, bias, out, f, smem, s);
  return launch_forward_local_t<KS, HR, WR, 4>(q, k, v, idx, B, w, bias, out, f, smem, s);
}

template <int KS>
int launch_forward_local(const void *q, const void *k, const void *v, int32_t *idx, int B,
                         const float *w, const float *bias, void *out, const FusedGeom &f,
                         size_t smem, cudaStream_t s) {
  if (f.img.hr == 2 && f.img.wr == 2)
    return launch_forward_local_l<KS, 2, 2>(q, k, v, idx, B, w, bias, out, f, smem, s);
  return launch_forward_local_l<KS, 0, 0>(q, k, v, idx, B, w, bias, out, f, smem, s);
}

template <int KS>
int launch_forward_image_ks(const void *q, const void *k, const void *v, int32_t *idx, int B,
                            const float *w, const float *bias, void *out, const FusedGeom &f,
                            size_t smem, cudaStream_t s) {
  if (f.img.H % 7 == 0)
    return launch_forward_image_kr<KS, 7>(q, k, v, idx, B, w, bias, out, f, smem, s);
  return launch_forward_image_kr<KS, 8>(q, k, v, idx, B, w, bias, out, f, smem, s);
}

int launch_attend(const void *q, const void *k, const void *v, const int32_t *idx,
                  int B, int H, int W, int C, int heads, int S, int topk,
                  const float *w, const float *bias, int ks, int dtype, void *out,
                  bool pdl, cudaStream_t s);

// Whether all B clusters of the one-launch forward are resident at once on
// the current device (asked once per device and cluster shape). With more
// images the clusters run in waves, each as long as a whole cluster's
// routing, attention and LePE, and the routing kernel plus the attend kernel
// (whose CTAs need no partners) finish sooner.
bool forward_image_one_wave(int B, const FusedGeom &f, size_t smem) {
  struct Entry { int dev, nc; size_t smem; int clusters; };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const int nc = f.img.nc;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry &e : cache)
      if (e.dev == dev && e.nc == nc && e.smem == smem) return B <= e.clusters;
  }
  // every instantiation has the same block shape and shared memory
  const void *kern = reinterpret_cast<const void *>(bra::bra_forward_image_kernel<5, 7>);
  int n = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nc, 1, 1);
  cfg.blockDim = dim3(bra::kImgThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (allow_smem(kern, smem) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess)
    n = 0;
  (void)cudaGetLastError();
  std::lock_guard<std::mutex> lock(mu);
  cache.push_back({dev, nc, smem, n});
  return B <= n;
}

// The forward's launches: one kernel where the shape allows it, else the
// routing kernel and then the attend kernel (programmatic dependent launch).
int launch_forward(const void *q, const void *k, const void *v, int B, int H, int W, int C,
                   int heads, int S, int topk, const float *w, const float *bias, int ks,
                   int dtype, int32_t *idx, void *out, cudaStream_t s) {
  FusedGeom f;
  size_t smem;
  if (dtype == BRA_BF16 && plan_forward_local(H, W, C, heads, S, topk, ks, &f, &smem)) {
    switch (ks) {
      case 1: return launch_forward_local<1>(q, k, v, idx, B, w, bias, out, f, smem, s);
      case 3: return launch_forward_local<3>(q, k, v, idx, B, w, bias, out, f, smem, s);
      case 5: return launch_forward_local<5>(q, k, v, idx, B, w, bias, out, f, smem, s);
      default: return launch_forward_local<7>(q, k, v, idx, B, w, bias, out, f, smem, s);
    }
  }
  if (dtype == BRA_BF16 && plan_forward_image(H, W, C, heads, S, topk, ks, &f, &smem) &&
      forward_image_one_wave(B, f, smem)) {
    switch (ks) {
      case 1: return launch_forward_image_ks<1>(q, k, v, idx, B, w, bias, out, f, smem, s);
      case 3: return launch_forward_image_ks<3>(q, k, v, idx, B, w, bias, out, f, smem, s);
      case 5: return launch_forward_image_ks<5>(q, k, v, idx, B, w, bias, out, f, smem, s);
      default: return launch_forward_image_ks<7>(q, k, v, idx, B, w, bias, out, f, smem, s);
    }
  }
  int rc = launch_route(q, k, B, H, W, C, S, topk, dtype, idx, nullptr, s);
  if (rc) return rc;
  // programmatic dependent launch: the attend grid may start while the route
  // grid drains; it waits for that grid only where it reads the routing index
  return launch_attend(q, k, v, idx, B, H, W, C, heads, S, topk, w, bias, ks, dtype, out,
                       true, s);
}

// Kernels bra_forward launches for a shape (1 or 2).
int forward_launches(int B, int H, int W, int C, int heads, int S, int topk, int ks,
                     int dtype) {
  FusedGeom f;
  size_t smem;
  if (dtype == BRA_BF16 && plan_forward_local(H, W, C, heads, S, topk, ks, &f, &smem))
    return 1;
  return (dtype == BRA_BF16 && plan_forward_image(H, W, C, heads, S, topk, ks, &f, &smem) &&
          forward_image_one_wave(B, f, smem))
             ? 1
             : 2;
}

template <int KS>
int launch_attend_f32_ks(const void *q, const void *k, const void *v,
                         const int32_t *idx, int B, const float *w,
                         const float *bias, void *out, const AttendF32Geom &g,
                         size_t smem, cudaStream_t s) {
  auto kern = bra::bra_attend_f32_kernel<KS>;
  if (allow_smem(reinterpret_cast<const void *>(kern), smem) != cudaSuccess) return BRA_ERR_CUDA;
  const unsigned grid = (unsigned)((size_t)B * g.R);
  kern<<<grid, bra::kAttendF32Threads, smem, s>>>(
      static_cast<const float *>(q), static_cast<const float *>(k),
      static_cast<const float *>(v), idx, w, bias, static_cast<float *>(out), g);
  return cuda_status(cudaGetLastError());
}

int check_attend(const void *q, const void *k, const void *v, const int32_t *idx,
                 int B, int H, int W, int C, int heads, int S, int topk,
                 const float *w, int ks, int dtype, const void *out) {
  int rc = check_map_args(B, H, W, C, S, topk, dtype);
  if (rc) return rc;
  if (heads <= 0 || C % heads) return BRA_ERR_INVALID_ARG;
  if (ks <= 0 || ks % 2 == 0) return BRA_ERR_INVALID_ARG;
  if (B == 0) return BRA_OK;
  if (!q || !k || !v || !idx || !w || !out) return BRA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return BRA_ERR_INVALID_ARG;
  const size_t bytes = (size_t)B * H * W * C * elem_size(dtype);
  if (overlap(out, bytes, q, bytes) || overlap(out, bytes, k, bytes) ||
      overlap(out, bytes, v, bytes))
    return BRA_ERR_INVALID_ARG;
  if (!lepe_ks_supported(ks)) return BRA_ERR_UNSUPPORTED;
  if ((size_t)B * S * S > 0x7fffffffu) return BRA_ERR_UNSUPPORTED;
  size_t smem;
  if (dtype == BRA_BF16) {
    ImageGeom gi;
    AttendGeom g;
    if (!plan_attend_image_local(H, W, C, heads, S, topk, ks, &gi, &smem) &&
        !plan_attend_image(H, W, C, heads, S, topk, ks, &gi, &smem) &&
        !plan_attend_bf16(B, H, W, C, heads, S, topk, ks, &g, &smem))
      return BRA_ERR_UNSUPPORTED;
  } else {
    AttendF32Geom g;
    if (!plan_attend_f32(H, W, C, heads, S, topk, ks, &g, &smem)) return BRA_ERR_UNSUPPORTED;
  }
  return BRA_OK;
}

int launch_attend(const void *q, const void *k, const void *v, const int32_t *idx,
                  int B, int H, int W, int C, int heads, int S, int topk,
                  const float *w, const float *bias, int ks, int dtype, void *out,
                  bool pdl, cudaStream_t s) {
  size_t smem;
  if (dtype == BRA_BF16) {
    ImageGeom gi;
    if (plan_attend_image_local(H, W, C, heads, S, topk, ks, &gi, &smem)) {
      switch (ks) {
        case 1: return launch_attend_image_local<1>(q, k, v, idx, B, w, bias, out, gi, smem, pdl, s);
        case 3: return launch_attend_image_local<3>(q, k, v, idx, B, w, bias, out, gi, smem, pdl, s);
        case 5: return launch_attend_image_local<5>(q, k, v, idx, B, w, bias, out, gi, smem, pdl, s);
        default: return launch_attend_image_local<7>(q, k, v, idx, B, w, bias, out, gi, smem, pdl, s);
      }
    }
    if (plan_attend_image(H, W, C, heads, S, topk, ks, &gi, &smem)) {
      switch (ks) {
        case 1: return launch_attend_image_ks<1>(q, k, v, idx, B, w, bias, out, gi, smem, pdl, s);
        case 3: return launch_attend_image_ks<3>(q, k, v, idx, B, w, bias, out, gi, smem, pdl, s);
        case 5: return launch_attend_image_ks<5>(q, k, v, idx, B, w, bias, out, gi, smem, pdl, s);
        default: return launch_attend_image_ks<7>(q, k, v, idx, B, w, bias, out, gi, smem, pdl, s);
      }
    }
    AttendGeom g;
    plan_attend_bf16(B, H, W, C, heads, S, topk, ks, &g, &smem);
    switch (ks) {
      case 1: return launch_attend_bf16_ks<1>(q, k, v, idx, B, w, bias, out, g, smem, pdl, s);
      case 3: return launch_attend_bf16_ks<3>(q, k, v, idx, B, w, bias, out, g, smem, pdl, s);
      case 5: return launch_attend_bf16_ks<5>(q, k, v, idx, B, w, bias, out, g, smem, pdl, s);
      default: return launch_attend_bf16_ks<7>(q, k, v, idx, B, w, bias, out, g, smem, pdl, s);
    }
  }
  AttendF32Geom g;
  plan_attend_f32(H, W, C, heads, S, topk, ks, &g, &smem);
  switch (ks) {
    case 1: return launch_attend_f32_ks<1>(q, k, v, idx, B, w, bias, out, g, smem, s);
    case 3: return launch_attend_f32_ks<3>(q, k, v, idx, B, w, bias, out, g, smem, s);
    case 5: return launch_attend_f32_ks<5>(q, k, v, idx, B, w, bias, out, g, smem, s);
    default: return launch_attend_f32_ks<7>(q, k, v, idx, B, w, bias, out, g, smem, s);
  }
}

}  // namespace

extern "C" {

int bra_route(const void *q, const void *k, int B, int H, int W, int C, int S,
              int topk, int dtype, int32_t *idx, float *affinity, void *stream) {
  int rc = check_route(q, k, B, H, W, C, S, topk, dtype, idx);
  if (rc || B == 0) return rc;
  (void)cudaGetLastError();
  return launch_route(q, k, B, H, W, C, S, topk, dtype, idx, affinity,
                      static_cast<cudaStream_t>(stream));
}

int bra_attend(const void *q, const void *k, const void *v, const int32_t *idx,
               int B, int H, int W, int C, int heads, int S, int topk,
               const float *lepe_w, const float *lepe_b, int lepe_ks, int dtype,
               void *out, void *stream) {
  int rc = check_attend(q, k, v, idx, B, H, W, C, heads, S, topk, lepe_w, lepe_ks,
                        dtype, out);
  if (rc || B == 0) return rc;
  (void)cudaGetLastError();
  return launch_attend(q, k, v, idx, B, H, W, C, heads, S, topk, lepe_w, lepe_b,
                       lepe_ks, dtype, out, false, static_cast<cudaStream_t>(stream));
}

int bra_forward(const void *q, const void *k, const void *v, int B, int H, int W,
                int C, int heads, int S, int topk, const float *lepe_w,
                const float *lepe_b, int lepe_ks, int dtype,
                int32_t *idx_workspace, void *out, void *stream) {
  int rc = check_route(q, k, B, H, W, C, S, topk, dtype, idx_workspace);
  if (rc) return rc;
  rc = check_attend(q, k, v, idx_workspace, B, H, W, C, heads, S, topk, lepe_w,
                    lepe_ks, dtype, out);
  if (rc || B == 0) return rc;
  const size_t ib = bra_idx_workspace_bytes(B, S, topk);
  const size_t bytes = (size_t)B * H * W * C * elem_size(dtype);
  if (overlap(idx_workspace, ib, out, bytes) || overlap(idx_workspace, ib, q, bytes) ||
      overlap(idx_workspace, ib, k, bytes) || overlap(idx_workspace, ib, v, bytes))
    return BRA_ERR_INVALID_ARG;
  (void)cudaGetLastError();
  return launch_forward(q, k, v, B, H, W, C, heads, S, topk, lepe_w, lepe_b, lepe_ks, dtype,
                        idx_workspace, out, static_cast<cudaStream_t>(stream));
}

int bra_attend_tc(const void *q, const void *k, const void *v, const int32_t *idx, int B,
                  int H, int W, int C, int heads, int S, int topk, const float *lepe_w,
                  const float *lepe_b, int lepe_ks, int dtype, void *out, void *stream) {
  int rc = check_attend(q, k, v, idx, B, H, W, C, heads, S, topk, lepe_w, lepe_ks, dtype, out);
  if (rc || B == 0) return rc;
  TcGeom g;
  size_t smem;
  if (dtype != BRA_BF16 || !plan_attend_tc(B, H, W, C, heads, S, topk, lepe_ks, &g, &smem))
    return BRA_ERR_UNSUPPORTED;
  (void)cudaGetLastError();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (lepe_ks) {
    case 1: return launch_attend_tc_ks<1>(q, k, v, idx, B, C, lepe_w, lepe_b, out, g, smem, false, s);
    case 3: return launch_attend_tc_ks<3>(q, k, v, idx, B, C, lepe_w, lepe_b, out, g, smem, false, s);
    default: return launch_attend_tc_ks<5>(q, k, v, idx, B, C, lepe_w, lepe_b, out, g, smem, false, s);
  }
}

int bra_qkv_project(const void *x, const void *w, const float *bias, long long M, int C,
                    int dtype, void *q, void *k, void *v, void *stream) {
  if (M < 0 || C <= 0) return BRA_ERR_INVALID_ARG;
  if (dtype != BRA_F32 && dtype != BRA_BF16) return BRA_ERR_INVALID_ARG;
  if (M == 0) return BRA_OK;
  if (!x || !w || !q || !k || !v) return BRA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(q) || !aligned16(k) || !aligned16(v))
    return BRA_ERR_INVALID_ARG;
  const size_t bytes = (size_t)M * C * 2;
  const void *outs[3] = {q, k, v};
  for (int i = 0; i < 3; ++i) {
    if (overlap(outs[i], bytes, x, bytes) || overlap(outs[i], bytes, w, (size_t)3 * C * C * 2))
      return BRA_ERR_INVALID_ARG;
    for (int j = 0; j < i; ++j)
      if (overlap(outs[i], bytes, outs[j], bytes)) return BRA_ERR_INVALID_ARG;
  }
  if (dtype != BRA_BF16 || M > 0x7fffffffll - 127 || C > 256) return BRA_ERR_UNSUPPORTED;
  void *qkv[3] = {q, k, v};
  return launch_linear(x, w, bias, (int)M, C, 3 * C, C, qkv, nullptr,
                       static_cast<cudaStream_t>(stream));
}

int bra_linear(const void *x, const void *w, const float *bias, long long M, int K, int N,
               const void *residual, int dtype, void *y, void *stream) {
  if (M < 0 || K <= 0 || N <= 0) return BRA_ERR_INVALID_ARG;
  if (dtype != BRA_F32 && dtype != BRA_BF16) return BRA_ERR_INVALID_ARG;
  if (M == 0) return BRA_OK;
  if (!x || !w || !y) return BRA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (residual && !aligned16(residual)))
    return BRA_ERR_INVALID_ARG;
  const size_t e = elem_size(dtype);
  const size_t xb = (size_t)M * K * e, yb = (size_t)M * N * e;
  if (overlap(y, yb, x, xb) || overlap(y, yb, w, (size_t)N * K * e) ||
      (residual && residual != y && overlap(y, yb, residual, yb)))
    return BRA_ERR_INVALID_ARG;
  if (dtype != BRA_BF16 || M > 0x7fffffffll - 127) return BRA_ERR_UNSUPPORTED;
  void *outs[1] = {y};
  return launch_linear(x, w, bias, (int)M, K, N, N, outs, residual,
                       static_cast<cudaStream_t>(stream));
}

int bra_forward_launches(int B, int H, int W, int C, int heads, int S, int topk, int lepe_ks,
                         int dtype) {
  int rc = check_map_args(B, H, W, C, S, topk, dtype);
  if (rc) return -rc;
  if (heads <= 0 || C % heads || lepe_ks <= 0 || lepe_ks % 2 == 0) return -BRA_ERR_INVALID_ARG;
  if (B == 0) return 0;
  return forward_launches(B, H, W, C, heads, S, topk, lepe_ks, dtype);
}

int bra_layer_norm(const void *x, const float *gamma, const float *beta, long long M, int C,
                   float eps, int dtype, void *y, void *stream) {
  if (M < 0 || C <= 0 || !(eps >= 0.f)) return BRA_ERR_INVALID_ARG;
  if (dtype != BRA_F32 && dtype != BRA_BF16) return BRA_ERR_INVALID_ARG;
  if (M == 0) return BRA_OK;
  if (!x || !y || !aligned16(x) || !aligned16(y)) return BRA_ERR_INVALID_ARG;
  const size_t bytes = (size_t)M * C * elem_size(dtype);
  if (x != y && overlap(x, bytes, y, bytes)) return BRA_ERR_INVALID_ARG;
  if (dtype != BRA_BF16 || (C != 64 && C != 128 && C != 256)) return BRA_ERR_UNSUPPORTED;
  (void)cudaGetLastError();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int G = C / 8;
  const long long per_block = (bra::kLnThreads / 32) * (32 / G);
  const unsigned grid = (unsigned)((M + per_block - 1) / per_block);
  const auto *xi = static_cast<const __nv_bfloat16 *>(x);
  auto *yo = static_cast<__nv_bfloat16 *>(y);
  if (G == 8)
    bra::bra_layer_norm_kernel<8><<<grid, bra::kLnThreads, 0, s>>>(xi, gamma, beta, M, eps, yo);
  else if (G == 16)
    bra::bra_layer_norm_kernel<16><<<grid, bra::kLnThreads, 0, s>>>(xi, gamma, beta, M, eps, yo);
  else
    bra::bra_layer_norm_kernel<32><<<grid, bra::kLnThreads, 0, s>>>(xi, gamma, beta, M, eps, yo);
  return cuda_status(cudaGetLastError());
}

int bra_residual_add(const void *x, const void *r, long long n, int dtype, void *y,
                     void *stream) {
  if (n < 0) return BRA_ERR_INVALID_ARG;
  if (dtype != BRA_F32 && dtype != BRA_BF16) return BRA_ERR_INVALID_ARG;
  if (n == 0) return BRA_OK;
  if (!x || !r || !y || !aligned16(x) || !aligned16(r) || !aligned16(y))
    return BRA_ERR_INVALID_ARG;
  const size_t bytes = (size_t)n * elem_size(dtype);
  if ((x != y && overlap(x, bytes, y, bytes)) || (r != y && overlap(r, bytes, y, bytes)))
    return BRA_ERR_INVALID_ARG;
  if (dtype != BRA_BF16 || n % 8) return BRA_ERR_UNSUPPORTED;
  (void)cudaGetLastError();
  const long long n8 = n / 8;
  const unsigned grid = (unsigned)std::min<long long>((n8 + bra::kLnThreads - 1) / bra::kLnThreads,
                                                      (long long)sm_count() * 8);
  bra::bra_residual_add_kernel<<<grid, bra::kLnThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16 *>(x), static_cast<const __nv_bfloat16 *>(r), n8,
      static_cast<__nv_bfloat16 *>(y));
  return cuda_status(cudaGetLastError());
}

int bra_dwconv_gelu(const void *h, const float *w, const float *bias, int B, int H, int W,
                    int Ch, int dtype, void *y, void *stream) {
  if (B < 0 || H <= 0 || W <= 0 || Ch <= 0) return BRA_ERR_INVALID_ARG;
  if (dtype != BRA_F32 && dtype != BRA_BF16) return BRA_ERR_INVALID_ARG;
  if (B == 0) return BRA_OK;
  if (!h || !w || !y || !aligned16(h) || !aligned16(y)) return BRA_ERR_INVALID_ARG;
  const size_t bytes = (size_t)B * H * W * Ch * elem_size(dtype);
  if (overlap(h, bytes, y, bytes)) return BRA_ERR_INVALID_ARG;
  // a block: all chunks of an 8-token tile row, Ch / 8 x 8 threads
  if (dtype != BRA_BF16 || Ch % 8 || Ch / 8 * bra::kDwTile > bra::kDwMaxThreads)
    return BRA_ERR_UNSUPPORTED;
  const long long tiles = (long long)B * ((H + bra::kDwTile - 1) / bra::kDwTile) *
                          ((W + bra::kDwTile - 1) / bra::kDwTile);
  if (tiles > 0x7fffffffll) return BRA_ERR_UNSUPPORTED;
  (void)cudaGetLastError();
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const unsigned threads = (unsigned)(Ch / 8 * bra::kDwTile);
  // the input tile staged by TMA: one box of all channels up to 256, two of
  // Ch / 2 up to 384 (a box holds at most 256 elements a row)
  const int nb = Ch <= 256 ? 1 : (Ch % 16 == 0 ? 2 : 0);
  CUtensorMap tm;
  if (nb && make_map_t(&tm, h, BRA_BF16, B, H, W, Ch, bra::kDwIn, bra::kDwIn, false, Ch / nb)) {
    // two input buffers and their mbarriers; a persistent grid of as many
    // CTAs as are resident at once
    const size_t smem = (size_t)2 * bra::kDwIn * bra::kDwIn * Ch * 2 + 16 + 128;
    const void *kern = nb == 1 ? reinterpret_cast<const void *>(bra::bra_dwconv_gelu_tma_kernel<1>)
                               : reinterpret_cast<const void *>(bra::bra_dwconv_gelu_tma_kernel<2>);
    if (allow_smem(kern, smem) != cudaSuccess) return BRA_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, (int)threads, smem) !=
            cudaSuccess ||
        per_sm < 1)
      return BRA_ERR_CUDA;
    const unsigned grid = (unsigned)std::min<long long>(tiles, (long long)per_sm * sm_count());
    __nv_bfloat16 *yo = static_cast<__nv_bfloat16 *>(y);
    if (nb == 1)
      bra::bra_dwconv_gelu_tma_kernel<1><<<grid, threads, smem, st>>>(tm, w, bias, B, H, W, Ch,
                                                                       yo);
    else
      bra::bra_dwconv_gelu_tma_kernel<2><<<grid, threads, smem, st>>>(tm, w, bias, B, H, W, Ch,
                                                                       yo);
    return cuda_status(cudaGetLastError());
  }
  bra::bra_dwconv_gelu_kernel<<<(unsigned)tiles, threads, 0, st>>>(
      static_cast<const __nv_bfloat16 *>(h), w, bias, B, H, W, Ch,
      static_cast<__nv_bfloat16 *>(y));
  return cuda_status(cudaGetLastError());
}

size_t bra_block_ffn_workspace_bytes(int B, int H, int W, int C) {
  if (B < 0 || H <= 0 || W <= 0 || C <= 0) return 0;
  // the normalised tokens [M][C], the hidden layer before and after the
  // convolution and GELU [M][3C] each (bf16)
  return (size_t)7 * B * H * W * C * 2;
}

int bra_block_ffn(const void *x, const float *ln_w, const float *ln_b, float eps, const void *w1,
                  const float *b1, const float *conv_w, const float *conv_b, const void *w2,
                  const float *b2, int B, int H, int W, int C, int dtype, void *workspace,
                  void *y, void *stream) {
  if (B < 0 || H <= 0 || W <= 0 || C <= 0 || !(eps >= 0.f)) return BRA_ERR_INVALID_ARG;
  if (dtype != BRA_F32 && dtype != BRA_BF16) return BRA_ERR_INVALID_ARG;
  if (B == 0) return BRA_OK;
  if (!x || !w1 || !conv_w || !w2 || !workspace || !y) return BRA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(workspace) || !aligned16(y)) return BRA_ERR_INVALID_ARG;
  const size_t mc = (size_t)B * H * W * C;
  const size_t bytes = mc * elem_size(dtype);
  const size_t ws = bra_block_ffn_workspace_bytes(B, H, W, C);
  if (overlap(y, bytes, x, bytes) || overlap(y, bytes, workspace, ws) ||
      overlap(x, bytes, workspace, ws))
    return BRA_ERR_INVALID_ARG;
  if (dtype != BRA_BF16) return BRA_ERR_UNSUPPORTED;
  uint8_t *w8 = static_cast<uint8_t *>(workspace);
  void *xn = w8, *hid = w8 + 2 * mc, *act = w8 + 8 * mc;
  const long long M = (long long)B * H * W;
  int rc = bra_layer_norm(x, ln_w, ln_b, M, C, eps, dtype, xn, stream);
  if (rc) return rc;
  rc = bra_linear(xn, w1, b1, M, C, 3 * C, nullptr, dtype, hid, stream);
  if (rc) return rc;
  rc = bra_dwconv_gelu(hid, conv_w, conv_b, B, H, W, 3 * C, dtype, act, stream);
  if (rc) return rc;
  return bra_linear(act, w2, b2, M, 3 * C, C, x, dtype, y, stream);
}

size_t bra_block_attention_workspace_bytes(int B, int H, int W, int C, int S, int topk) {
  if (B < 0 || H <= 0 || W <= 0 || C <= 0 || S <= 0 || topk <= 0) return 0;
  // the normalised tokens, q, k and v (bf16), then the routing index
  return round_up((size_t)4 * B * H * W * C * 2, 256) + bra_idx_workspace_bytes(B, S, topk);
}

int bra_block_attention(const void *x, const float *ln_w, const float *ln_b, float eps,
                        const void *w_qkv, const float *b_qkv, int B, int H, int W, int C,
                        int heads, int S, int topk, const float *lepe_w, const float *lepe_b,
                        int lepe_ks, int dtype, void *workspace, void *y, void *stream) {
  int rc = check_map_args(B, H, W, C, S, topk, dtype);
  if (rc) return rc;
  if (heads <= 0 || C % heads || lepe_ks <= 0 || lepe_ks % 2 == 0 || !(eps >= 0.f))
    return BRA_ERR_INVALID_ARG;
  if (B == 0) return BRA_OK;
  if (!x || !w_qkv || !lepe_w || !workspace || !y) return BRA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_qkv) || !aligned16(workspace) || !aligned16(y))
    return BRA_ERR_INVALID_ARG;
  const size_t mc = (size_t)B * H * W * C;
  const size_t bytes = mc * elem_size(dtype);
  const size_t ws = bra_block_attention_workspace_bytes(B, H, W, C, S, topk);
  if (overlap(y, bytes, x, bytes) || overlap(y, bytes, workspace, ws) ||
      overlap(x, bytes, workspace, ws))
    return BRA_ERR_INVALID_ARG;
  if (dtype != BRA_BF16) return BRA_ERR_UNSUPPORTED;
  uint8_t *w8 = static_cast<uint8_t *>(workspace);
  void *xn = w8, *q = w8 + 2 * mc, *k = w8 + 4 * mc, *v = w8 + 6 * mc;
  int32_t *idx = reinterpret_cast<int32_t *>(w8 + round_up(8 * mc, 256));
  const long long M = (long long)B * H * W;
  rc = bra_layer_norm(x, ln_w, ln_b, M, C, eps, dtype, xn, stream);
  if (rc) return rc;
  rc = bra_qkv_project(xn, w_qkv, b_qkv, M, C, dtype, q, k, v, stream);
  if (rc) return rc;
  rc = bra_forward(q, k, v, B, H, W, C, heads, S, topk, lepe_w, lepe_b, lepe_ks, dtype, idx, y,
                   stream);
  if (rc) return rc;
  return bra_residual_add(x, y, (long long)mc, dtype, y, stream);
}

}  // extern "C"

namespace {

// Shared memory of the attention backward: the region's Q and dout, the
// routed keys' K and V (rows of d + 1 floats), P and dP ([n][nk + 1] each),
// D and the token lists.
bool plan_attend_bwd(int H, int W, int C, int heads, int S, int topk, bra::BwdGeom *g,
                     size_t *smem) {
  if (heads <= 0 || C % heads || C / heads > 64) return false;
  bra::BwdGeom a = {};
  a.H = H; a.W = W; a.C = C; a.S = S; a.heads = heads; a.topk = topk;
  a.hr = H / S; a.wr = W / S; a.n = a.hr * a.wr; a.R = S * S; a.d = C / heads;
  a.nk = topk * a.n;
  a.ds = a.d + 1;
  a.ps = a.nk + 1;
  a.scale = (float)(1.0 / std::sqrt((double)a.d));
  size_t off = (size_t)a.n * a.ds * 4;
  a.off_do = (uint32_t)off; off += (size_t)a.n * a.ds * 4;
  a.off_k = (uint32_t)off; off += (size_t)a.nk * a.ds * 4;
  a.off_v = (uint32_t)off; off += (size_t)a.nk * a.ds * 4;
  a.off_p = (uint32_t)off; off += (size_t)a.n * a.ps * 4;
  a.off_g = (uint32_t)off; off += (size_t)a.n * a.ps * 4;
  a.off_d = (uint32_t)off; off += (size_t)a.n * 4;
  a.off_tok = (uint32_t)round_up(off, 16); off = a.off_tok + (size_t)(a.nk + a.n) * 4;
  *g = a;
  *smem = off;
  return off <= kMaxSmemPerBlock;
}

template <typename T>
int launch_attend_bwd(const void *q, const void *k, const void *v, const int32_t *idx, int B,
                      const float *w, int ks, const void *dout, const bra::BwdGeom &g,
                      size_t smem, float *dq, float *dk, float *dv, float *dw, float *db,
                      cudaStream_t s) {
  // head dimension 32 and 64 keys a query (the stage-1 to stage-3 shapes)
  // fixed at compile time where they hold
  auto kern = g.d == 32 && g.nk == 64 ? bra::bra_attend_bwd_kernel<T, 32, 64>
              : g.d == 32             ? bra::bra_attend_bwd_kernel<T, 32, 0>
                                      : bra::bra_attend_bwd_kernel<T, 0, 0>;
  if (allow_smem(reinterpret_cast<const void *>(kern), smem) != cudaSuccess)
    return BRA_ERR_CUDA;
  const unsigned grid = (unsigned)((size_t)B * g.R * g.heads);
  kern<<<grid, bra::kBwdThreads, smem, s>>>(static_cast<const T *>(q), static_cast<const T *>(k),
                                            static_cast<const T *>(v), idx,
                                            static_cast<const T *>(dout), g, dq, dk, dv);
  int rc = cuda_status(cudaGetLastError());
  if (rc) return rc;
  const unsigned rows = (unsigned)((size_t)B * g.H);
  // a multiple of C threads (several columns of a row at once), or all of
  // the kernel's threads with the channels in turns
  const int NT = ks >= 7 ? bra::lepe_bwd_threads<7>() : bra::lepe_bwd_threads<5>();
  const unsigned nt = (unsigned)(g.C <= NT ? (NT / g.C) * g.C : NT);
  const T *vt = static_cast<const T *>(v), *gt = static_cast<const T *>(dout);
  // the rows staged in shared memory when they fit (C * sizeof(T) a multiple
  // of 16 bytes), else read from global memory
  const size_t staged = (size_t)2 * ks * (g.W + ks - 1) * g.C * sizeof(T);
  const size_t static_part = (size_t)NT * (ks * ks + 1) * 4;
  if ((g.C * sizeof(T)) % 16 == 0 && aligned16(v) && aligned16(dout) &&
      staged + static_part <= kMaxSmemPerBlock) {
    const void *kern = ks == 1   ? reinterpret_cast<const void *>(bra::bra_lepe_bwd_staged_kernel<T, 1>)
                       : ks == 3 ? reinterpret_cast<const void *>(bra::bra_lepe_bwd_staged_kernel<T, 3>)
                       : ks == 5 ? reinterpret_cast<const void *>(bra::bra_lepe_bwd_staged_kernel<T, 5>)
                                 : reinterpret_cast<const void *>(bra::bra_lepe_bwd_staged_kernel<T, 7>);
    // the dynamic part's limit, beside the kernel's static partial sums
    if (staged + static_part > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(kMaxSmemPerBlock - static_part)) != cudaSuccess)
      return BRA_ERR_CUDA;
    switch (ks) {
      case 1:
        bra::bra_lepe_bwd_staged_kernel<T, 1><<<rows, nt, staged, s>>>(vt, w, gt, g.H, g.W, g.C,
                                                                       dv, dw, db);
        break;
      case 3:
        bra::bra_lepe_bwd_staged_kernel<T, 3><<<rows, nt, staged, s>>>(vt, w, gt, g.H, g.W, g.C,
                                                                       dv, dw, db);
        break;
      case 5:
        bra::bra_lepe_bwd_staged_kernel<T, 5><<<rows, nt, staged, s>>>(vt, w, gt, g.H, g.W, g.C,
                                                                       dv, dw, db);
        break;
      default:
        bra::bra_lepe_bwd_staged_kernel<T, 7><<<rows, nt, staged, s>>>(vt, w, gt, g.H, g.W, g.C,
                                                                       dv, dw, db);
        break;
    }
    return cuda_status(cudaGetLastError());
  }
  switch (ks) {
    case 1:
      bra::bra_lepe_bwd_kernel<T, 1><<<rows, nt, 0, s>>>(vt, w, gt, g.H, g.W, g.C, dv, dw, db);
      break;
    case 3:
      bra::bra_lepe_bwd_kernel<T, 3><<<rows, nt, 0, s>>>(vt, w, gt, g.H, g.W, g.C, dv, dw, db);
      break;
    case 5:
      bra::bra_lepe_bwd_kernel<T, 5><<<rows, nt, 0, s>>>(vt, w, gt, g.H, g.W, g.C, dv, dw, db);
      break;
    default:
      bra::bra_lepe_bwd_kernel<T, 7><<<rows, nt, 0, s>>>(vt, w, gt, g.H, g.W, g.C, dv, dw, db);
      break;
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace

extern "C" {

int bra_attend_backward(const void *q, const void *k, const void *v, const int32_t *idx,
                        int B, int H, int W, int C, int heads, int S, int topk,
                        const float *lepe_w, int lepe_ks, const void *dout, int dtype,
                        float *dq, float *dk, float *dv, float *dlepe_w, float *dlepe_b,
                        void *stream) {
  int rc = check_map_args(B, H, W, C, S, topk, dtype);
  if (rc) return rc;
  if (heads <= 0 || C % heads) return BRA_ERR_INVALID_ARG;
  if (lepe_ks <= 0 || lepe_ks % 2 == 0) return BRA_ERR_INVALID_ARG;
  if (B == 0) return BRA_OK;
  if (!q || !k || !v || !idx || !lepe_w || !dout || !dq || !dk || !dv || !dlepe_w)
    return BRA_ERR_INVALID_ARG;
  const size_t in_bytes = (size_t)B * H * W * C * elem_size(dtype);
  const size_t g_bytes = (size_t)B * H * W * C * 4;
  const size_t w_bytes = (size_t)C * lepe_ks * lepe_ks * 4;
  const void *ins[] = {q, k, v, dout};
  float *outs[] = {dq, dk, dv};
  for (int a = 0; a < 3; ++a) {
    float *o = outs[a];
    for (const void *in : ins)
      if (overlap(o, g_bytes, in, in_bytes)) return BRA_ERR_INVALID_ARG;
    for (int a2 = a + 1; a2 < 3; ++a2)
      if (overlap(o, g_bytes, outs[a2], g_bytes)) return BRA_ERR_INVALID_ARG;
    if (overlap(o, g_bytes, dlepe_w, w_bytes)) return BRA_ERR_INVALID_ARG;
    if (dlepe_b && overlap(o, g_bytes, dlepe_b, (size_t)C * 4)) return BRA_ERR_INVALID_ARG;
  }
  if (dlepe_b && overlap(dlepe_w, w_bytes, dlepe_b, (size_t)C * 4)) return BRA_ERR_INVALID_ARG;
  if (!lepe_ks_supported(lepe_ks)) return BRA_ERR_UNSUPPORTED;
  if ((size_t)B * S * S * heads > 0x7fffffffu) return BRA_ERR_UNSUPPORTED;
  bra::BwdGeom g;
  size_t smem;
  if (!plan_attend_bwd(H, W, C, heads, S, topk, &g, &smem)) return BRA_ERR_UNSUPPORTED;
  g.vec4 = g.d % 4 == 0 && aligned16(dq) && aligned16(dk) && aligned16(dv);
  (void)cudaGetLastError();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // dq is written whole; the others are sums
  if (cudaMemsetAsync(dk, 0, g_bytes, s) != cudaSuccess ||
      cudaMemsetAsync(dv, 0, g_bytes, s) != cudaSuccess ||
      cudaMemsetAsync(dlepe_w, 0, w_bytes, s) != cudaSuccess ||
      (dlepe_b && cudaMemsetAsync(dlepe_b, 0, (size_t)C * 4, s) != cudaSuccess))
    return BRA_ERR_CUDA;
  if (dtype == BRA_F32)
    return launch_attend_bwd<float>(q, k, v, idx, B, lepe_w, lepe_ks, dout, g, smem, dq, dk,
                                    dv, dlepe_w, dlepe_b, s);
  return launch_attend_bwd<__nv_bfloat16>(q, k, v, idx, B, lepe_w, lepe_ks, dout, g, smem, dq,
                                          dk, dv, dlepe_w, dlepe_b, s);
}

size_t bra_idx_workspace_bytes(int B, int S, int topk) {
  if (B < 0 || S <= 0 || topk <= 0) return 0;
  return (size_t)B * S * S * topk * sizeof(int32_t);
}

int bra_device_status(void *stream, int clear) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return BRA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, bra::g_status, sizeof(v)) != cudaSuccess)
    return BRA_ERR_CUDA;
  if (clear) {
    const unsigned z = 0;
    if (cudaMemcpyToSymbol(bra::g_status, &z, sizeof(z)) != cudaSuccess)
      return BRA_ERR_CUDA;
  }
  if (v & bra::kStatusTimeout) return BRA_ERR_TIMEOUT;
  if (v & bra::kStatusBadIndex) return BRA_ERR_INVALID_ARG;
  return BRA_OK;
}

const char *bra_status_string(int status) {
  switch (status) {
    case BRA_OK: return "ok";
    case BRA_ERR_INVALID_ARG: return "invalid argument";
    case BRA_ERR_UNSUPPORTED: return "unsupported shape";
    case BRA_ERR_CUDA: return "CUDA error";
    case BRA_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

int bra_abi_version(void) { return 103; }

int bra_check_wait_timeout(uint64_t limit_ns, void *stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000ull) return BRA_ERR_INVALID_ARG;
  (void)cudaGetLastError();
  bra::bra_wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns);
  return cuda_status(cudaGetLastError());
}

}  // extern "C"

// ------------------------------------------------- allocation-free forward
// bra_forward_static keeps the routing index in this file-scope device array
// instead of a caller-supplied workspace. Every GPU that loads the library
// holds it (BRA_STATIC_IDX_MAX_ENTRIES int32, 1 MiB) until the process exits.
namespace {

__device__ __align__(256) int32_t g_static_idx[BRA_STATIC_IDX_MAX_ENTRIES];

// Device address of g_static_idx, looked up once per device. In host code the
// array's name is only a host-side stand-in, so kernels must be given this
// address instead.
int32_t *static_idx_address() {
  constexpr int kMaxDevices = 64;
  static int32_t *addr[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_idx) != cudaSuccess || !p) return nullptr;
    addr[dev] = static_cast<int32_t *>(p);
  }
  return addr[dev];
}

}  // namespace

extern "C" int bra_forward_static(const void *q, const void *k, const void *v, int B,
                                  int H, int W, int C, int heads, int S, int topk,
                                  const float *lepe_w, const float *lepe_b,
                                  int lepe_ks, int dtype, void *out, void *stream) {
  if (B > 0 && S > 0 && topk > 0 &&
      (long long)B * S * S * topk > (long long)BRA_STATIC_IDX_MAX_ENTRIES)
    return BRA_ERR_UNSUPPORTED;
  // argument checks first, against a stand-in workspace pointer that cannot
  // overlap a caller buffer's check (the real address is only known on the
  // device); nothing is launched unless they pass
  int rc = check_route(q, k, B, H, W, C, S, topk, dtype,
                       reinterpret_cast<const int32_t *>(q));
  if (rc) return rc;
  rc = check_attend(q, k, v, reinterpret_cast<const int32_t *>(q), B, H, W, C, heads, S,
                    topk, lepe_w, lepe_ks, dtype, out);
  if (rc || B == 0) return rc;
  int32_t *idx = static_idx_address();
  if (!idx) return BRA_ERR_CUDA;
  (void)cudaGetLastError();
  return launch_forward(q, k, v, B, H, W, C, heads, S, topk, lepe_w, lepe_b, lepe_ks, dtype,
                        idx, out, static_cast<cudaStream_t>(stream));
}

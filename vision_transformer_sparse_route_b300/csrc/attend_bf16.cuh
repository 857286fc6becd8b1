// attend_bf16.cuh -- fused routed attention + LePE for bf16 maps on sm_103a.
//
// For one query region i of image b (a "unit"), with routing I = idx[b, i, :]:
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
// Persistent, one CTA per SM, walking the units blockIdx.x, blockIdx.x +
// gridDim.x, ... through a ring of shared-memory stages. A unit's stage
// receives, by TMA box copies, the Q tile, the routed regions' K and V tiles
// (the gather exists only in shared memory) and the V halo (region plus ks/2
// border; TMA's zero fill outside the image is the conv's zero padding).
//
// The CTA's 16 warps form two groups of 8 that take alternate units, so that
// one group's attention (tensor cores, exponentials) overlaps the other
// group's LePE (fp32 FMAs). For its unit a group runs
//   attention  one warp per (head, 16 query rows): S = Q K^T with mma.sync
//              m16n8k16 (bf16 in, f32 accumulate) over 64 keys at a time, an
//              online softmax whose exponentials are taken two at a time in
//              bf16 (they feed the bf16 P V product directly), O += P V, and
//              the row sums as an MMA of the same bf16 P against ones; the
//              normalised O (f32) goes back into the stage;
//   LePE       one thread per (channel pair, column, block of rows): the
//              depthwise stencil from the halo with packed f32x2 FMAs, plus
//              O, rounded once to bf16 into
//              the group's output staging tile;
// then the group's first warp refills the stage with the copies of the unit
// `stages` iterations ahead (its routing read by that warp while the unit was
// computed; one lane per box, one instruction for all boxes), while its last
// warp sends the staging tile out with a TMA store. A box copy holds up the
// thread that issues it for a long time (about a microsecond per instruction
// on the stage-1 shape), so each of these sits on a different warp.
#pragma once

#include "ptx.cuh"

namespace bra {

constexpr int kGroupWarps = 8;
constexpr int kGroups = 2;
constexpr int kGroupThreads = 32 * kGroupWarps;
constexpr int kAttendThreads = kGroups * kGroupThreads;
constexpr int kMaxStages = 6;

struct AttendGeom {
  int H, W, C, S, heads, topk;
  int hr, wr, n, R;
  int nc;         // 64-channel chunks, C / 64
  int slot;       // key rows per routed region in K/V slots (n rounded to 8)
  int kv_rows;    // rows of one K or V chunk buffer (topk * slot rounded to 64)
  int q_blocks;   // 16-row query blocks per region
  int tasks;      // heads * q_blocks attention tasks per unit
  int halo_w, halo_h;
  int units;      // B * S * S
  int stages;     // pipeline depth
  int masked;     // keys need masking (padded slots or a partial 64-key block)
  int alias;      // O overwrites the unit's Q/K/V once attention is done
  int issue_warps;  // warps of a group that issue a refill's box copies
  int lepe_items; // (C / 2) * wr * ceil(hr / RB)
  uint32_t q_chunk, kv_chunk, h_chunk, o_chunk;  // bytes per chunk buffer
  uint32_t off_k, off_v, off_h;  // within a stage
  uint32_t off_o;                // f32 O tile, within a stage
  uint32_t stage_bytes, tx_bytes;
  uint32_t off_out;              // output staging tiles [groups][2][nc * o_chunk]
  uint32_t off_w, off_bar;       // from the 1024-aligned base
  float scale_log2;              // d^-1/2 * log2(e)
};

__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Waits for the grids this launch depends on (programmatic dependent launch);
// a no-op when launched without that attribute.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Waits until at most N committed bulk stores still read shared memory.
template <int N>
__device__ __forceinline__ void tma_store_wait_read_n() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Word offset of O element (t, c) in the f32 O tile [n][C]: the column is
// XORed with 8 * (t mod 4), so that the eight rows one MMA fragment store
// touches fall in different banks.
__device__ __forceinline__ int o_index(int C, int t, int c) {
  return t * C + (c ^ ((t & 3) << 3));
}

// max of three floats in one instruction
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 2^x of a bf16 pair: packs (lo, hi) to bf16 (round to nearest even) and
// takes the hardware's bf16 exp2 of both halves; the result is the bf16 pair
// that multiplies V.
__device__ __forceinline__ uint32_t exp2_bf16x2(float lo, float hi) {
  uint32_t x, e;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(x) : "f"(hi), "f"(lo));
  asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(e) : "r"(x));
  return e;
}

// ------------------------------------------------------------- attention
// One attention task: 16 query rows (block qb) of head h for the unit whose
// tiles sit at q_base / k_base / v_base. Leaves the normalised O rows
// (row0 = qb*16 + lane/4 and row0 + 8, channels h*32 + a*8 + 2*(lane%4))
// in o.
template <bool MASKED>
__device__ __forceinline__ void attention_task(const AttendGeom &g, int h,
                                               int qb, uint32_t q_base,
                                               uint32_t k_base, uint32_t v_base,
                                               float (&o)[4][4], int lane) {
  const int cb = (h & 1) * 4;  // first 16-byte column of the head in its chunk
  const int nslots = g.topk * g.slot;
  // Per-lane byte offsets of the ldmatrix rows. Key blocks start at multiples
  // of 8 rows, so a row's swizzle (row mod 8) is the lane's own: within a
  // block only the block's base moves.
  const int l7 = lane & 7;
  const uint32_t k_off = l7 * 128 + (((cb + (lane >> 3)) ^ l7) << 4);
  const uint32_t v_row = l7 + ((lane >> 3) & 1) * 8;
  const uint32_t v_off0 = v_row * 128 + (((cb + (lane >> 4)) ^ l7) << 4);
  const uint32_t v_off1 = v_row * 128 + (((cb + 2 + (lane >> 4)) ^ l7) << 4);
  uint32_t qa[2][4];
#pragma unroll
  for (int ks = 0; ks < 2; ++ks)
    ldsm_x4(q_base + swz128(qb * 16 + (lane & 15), cb + ks * 2 + (lane >> 4)),
            qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);

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

  for (int kb = 0; kb < nslots; kb += 64) {
    const uint32_t kblk = k_base + kb * 128 + k_off;
    float s[8][4];
#pragma unroll
    for (int jt = 0; jt < 8; ++jt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[jt][e] = 0.f;
      if (!MASKED || kb + jt * 8 < nslots) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kblk + jt * 1024, b0, b1, b2, b3);
        mma_bf16_16816(s[jt], qa[0], b0, b1);
        mma_bf16_16816(s[jt], qa[1], b2, b3);
      }
    }
    if (MASKED) {
#pragma unroll
      for (int jt = 0; jt < 8; ++jt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = kb + jt * 8 + 2 * (lane & 3) + (e & 1);
          if (key >= nslots || (key % g.slot) >= g.n) s[jt][e] = -INFINITY;
        }
    }
    // row maxima (rows lane/4 and lane/4 + 8), three values per instruction
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
    float2 nb[2];  // -(new running max), in log2 units, per row
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
    // P = 2^(S * scale * log2 e - max), as bf16 pairs
    uint32_t p[8][2];
#pragma unroll
    for (int jt = 0; jt < 8; ++jt) {
      const float2 x0 = __ffma2_rn(make_float2(s[jt][0], s[jt][1]), sc2, nb[0]);
      const float2 x1 = __ffma2_rn(make_float2(s[jt][2], s[jt][3]), sc2, nb[1]);
      p[jt][0] = exp2_bf16x2(x0.x, x0.y);
      p[jt][1] = exp2_bf16x2(x1.x, x1.y);
    }
    const uint32_t vblk = v_base + kb * 128;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (!MASKED || kb + t * 16 < nslots) {
        const uint32_t pa[4] = {p[2 * t][0], p[2 * t][1], p[2 * t + 1][0],
                                p[2 * t + 1][1]};
        uint32_t r0, r1, r2, r3;
        ldsm_x4_trans(vblk + t * 2048 + v_off0, r0, r1, r2, r3);
        mma_bf16_16816(o[0], pa, r0, r1);
        mma_bf16_16816(o[1], pa, r2, r3);
        ldsm_x4_trans(vblk + t * 2048 + v_off1, r0, r1, r2, r3);
        mma_bf16_16816(o[2], pa, r0, r1);
        mma_bf16_16816(o[3], pa, r2, r3);
        mma_bf16_16816(l4, pa, ones, ones);  // row sums of the bf16 P
      }
    }
  }
  const float inv0 = 1.f / l4[0], inv1 = 1.f / l4[2];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    o[a][0] *= inv0; o[a][1] *= inv0;
    o[a][2] *= inv1; o[a][3] *= inv1;
  }
}

// Writes one task's O rows into the f32 O tile.
__device__ __forceinline__ void store_o(const AttendGeom &g, int h, int qb,
                                        const float (&o)[4][4], float *so, int lane) {
  const int row0 = qb * 16 + (lane >> 2);
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int ch = h * 32 + a * 8 + 2 * (lane & 3);
    if (row0 < g.n)
      *reinterpret_cast<float2 *>(so + o_index(g.C, row0, ch)) = make_float2(o[a][0], o[a][1]);
    if (row0 + 8 < g.n)
      *reinterpret_cast<float2 *>(so + o_index(g.C, row0 + 8, ch)) =
          make_float2(o[a][2], o[a][3]);
  }
}

// ------------------------------------------------------------------ LePE
// LePE of rows ry0 .. ry0+RB-1, column x, channels c, c+1 of one unit, plus
// the attention output from so; bf16 result into the (unswizzled) output
// tile ob. wgt holds the pair's KS*KS weights, bias the pair's bias. WR and
// HR, when non-zero, are the region's width and height known at compile time
// (then every halo offset is an immediate); zero means read them from g.
template <int KS, int RB, int WR, int HR>
__device__ __forceinline__ void lepe_item(const AttendGeom &g, const uint8_t *hb,
                                          const float *so, uint8_t *ob, int c,
                                          int x, int ry0, const float2 (&wgt)[KS * KS],
                                          float2 bias) {
  const int wr = WR ? WR : g.wr, hr = HR ? HR : g.hr;
  const int halo_w = wr + KS - 1, halo_h = hr + KS - 1;
  const int cc = c >> 6, cw = (c & 63) * 2;
  float2 acc[RB];
#pragma unroll
  for (int r = 0; r < RB; ++r) acc[r] = bias;
  const uint8_t *col = hb + cc * g.h_chunk + ((size_t)ry0 * halo_w + x) * 128 + cw;
#pragma unroll
  for (int yy = 0; yy < RB + KS - 1; ++yy) {
    if ((HR && HR % RB == 0) || ry0 + yy < halo_h) {
      const uint8_t *rp = col + yy * halo_w * 128;
#pragma unroll
      for (int w = 0; w < KS; ++w) {
        const uint32_t t2 = *reinterpret_cast<const uint32_t *>(rp + w * 128);
        // the two bf16 as floats, by byte permutes (integer pipe, leaving the
        // FMA pipe to the stencil)
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
    if ((HR && HR % RB == 0) || row < hr) {
      const int t = row * wr + x;
      const float2 ov = *reinterpret_cast<const float2 *>(so + o_index(g.C, t, c));
      const float2 sum = __fadd2_rn(acc[r], ov);
      *reinterpret_cast<uint32_t *>(ob + cc * g.o_chunk + t * 128 + cw) =
          pack_bf16x2(sum.x, sum.y);
    }
  }
}

template <int KS>
__device__ __forceinline__ void load_pair_weights(const float *sw, int C, int c,
                                                  float2 (&wgt)[KS * KS],
                                                  float2 &bias) {
#pragma unroll
  for (int e = 0; e < KS * KS; ++e)
    wgt[e] = *reinterpret_cast<const float2 *>(sw + e * C + c);
  bias = *reinterpret_cast<const float2 *>(sw + KS * KS * C + c);
}

// --------------------------------------------------------------- copies
// Issues the TMA copies of unit u into stage st, completing on bar: the Q
// tile, the K and V tiles of the unit's routed regions and the V halo. Run by
// warp `part` of nw warps. jl holds routed region number `lane` of the unit
// (read ahead by the caller) for lane < topk. When the unit has at most 32 nw
// boxes and at most 32 routed regions, lane l of warp `part` computes the
// operands of box l nw + part and one instruction a warp issues them (a box
// copy costs its issuing thread far more than the instruction, so boxes from
// one thread go out one after another); otherwise lane 0 of warp 0 issues
// every box, reading regions beyond 32 from idx. Warp 0 posts the expected
// byte count; copies of the other warps that complete before it only take
// the barrier's transaction count below zero for a while, and the phase
// cannot complete before warp 0's arrival.
template <int KS>
__device__ __forceinline__ void issue_unit(const AttendGeom &g, const CUtensorMap *tm_q,
                                           const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                                           const CUtensorMap *tm_vh, const int32_t *idx,
                                           int jl, uint8_t *st, uint64_t *bar, int u,
                                           int lane, int part = 0, int nw = 1) {
  constexpr int PAD = KS / 2;
  const int b = u / g.R, i = u % g.R;
  const int y0 = (i / g.S) * g.hr, x0 = (i % g.S) * g.wr;
  if (lane == 0 && part == 0) mbar_arrive_expect_tx(bar, g.tx_bytes);
  __syncwarp();
  const int nbox = g.nc * (2 + 2 * g.topk);
  if (nbox <= 32 * nw && g.topk <= 32) {
    const int l = lane * nw + part;
    // box l: chunk l % nc of Q (l / nc == 0), the halo (1), then K and V of
    // routed region m alternately (2 + 2m, 3 + 2m)
    const int cc = l % g.nc, r = l / g.nc;
    const int m = r >= 2 ? min((r - 2) >> 1, g.topk - 1) : 0;
    const int j = __shfl_sync(0xffffffffu, jl, m);
    const CUtensorMap *map = tm_q;
    uint8_t *dst = st + cc * g.q_chunk;
    int cx = x0, cy = y0;
    if (r == 1) {
      map = tm_vh;
      dst = st + g.off_h + cc * g.h_chunk;
      cx = x0 - PAD;
      cy = y0 - PAD;
    } else if (r >= 2) {
      const bool is_v = (r - 2) & 1;
      map = is_v ? tm_v : tm_k;
      dst = st + (is_v ? g.off_v : g.off_k) + cc * g.kv_chunk + m * g.slot * 128u;
      if (j < 0 || j >= g.R) {  // out of range: read zeros, flag it
        if (l < nbox) atomicOr(&g_status, kStatusBadIndex);
        cx = 0;
        cy = g.H;  // a box wholly below the image is all fill (zeros)
      } else {
        cx = (j % g.S) * g.wr;
        cy = (j / g.S) * g.hr;
      }
    }
    if (l < nbox) tma_load_4d(dst, map, bar, cc * 64, cx, cy, b);
    return;
  }
  if (part != 0) return;
  if (lane == 0) {
    for (int cc = 0; cc < g.nc; ++cc)
      tma_load_4d(st + cc * g.q_chunk, tm_q, bar, cc * 64, x0, y0, b);
  }
  const int32_t *ri = idx + (size_t)u * g.topk;
  for (int m0 = 0; m0 < g.topk; m0 += 32) {
    const int jw = m0 == 0 ? jl : (m0 + lane < g.topk ? __ldg(ri + m0 + lane) : 0);
    const int mn = min(32, g.topk - m0);
    for (int e = 0; e < mn; ++e) {
      const int j = __shfl_sync(0xffffffffu, jw, e);
      if (lane == 0) {
        const int m = m0 + e;
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
          tma_load_4d(st + g.off_k + off, tm_k, bar, cc * 64, xj, yj, b);
          tma_load_4d(st + g.off_v + off, tm_v, bar, cc * 64, xj, yj, b);
        }
      }
    }
  }
  if (lane == 0)
    for (int cc = 0; cc < g.nc; ++cc)
      tma_load_4d(st + g.off_h + cc * g.h_chunk, tm_vh, bar, cc * 64, x0 - PAD, y0 - PAD, b);
}

// Routed region number `lane` of unit u (lane < min(topk, 32)), else 0.
__device__ __forceinline__ int read_route_lane(const AttendGeom &g, const int32_t *idx,
                                               int u, int lane) {
  return lane < g.topk ? __ldg(idx + (size_t)u * g.topk + lane) : 0;
}

// ------------------------------------------------------------------ kernel
template <int KS, int RB, int WR, int HR>
__global__ void __launch_bounds__(kAttendThreads, 1)
    bra_attend_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_vh,
                           const __grid_constant__ CUtensorMap tm_o,
                           const int32_t *__restrict__ idx,
                           const float *__restrict__ lepe_w,
                           const float *__restrict__ lepe_b, AttendGeom g) {
  extern __shared__ uint8_t attend_smem_raw[];
  // 1024-byte aligned base, derived from the shared array by an offset so
  // that every access through it stays a shared-memory access
  uint8_t *smem = attend_smem_raw + ((1024u - (smem_u32(attend_smem_raw) & 1023u)) & 1023u);
  uint8_t *stage0 = smem;                                 // [stages][stage_bytes]
  float *sw = reinterpret_cast<float *>(smem + g.off_w);  // [KS*KS][C], bias [C]
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + g.off_bar);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = warp / kGroupWarps, gw = warp % kGroupWarps;
  const int gt = tid % kGroupThreads;
  const int bar_id = 1 + grp;  // the group's named barrier
  const int nslots = g.topk * g.slot;
  const uint32_t out_tile = g.nc * g.o_chunk;

  if (tid == 0) {
    for (int s = 0; s < g.stages; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  // LePE weights, tap-major so that a warp reads 32 consecutive channel pairs
  for (int e = tid; e < g.C * KS * KS; e += kAttendThreads) {
    const int tap = e / g.C, c = e % g.C;
    sw[e] = __ldg(lepe_w + (size_t)c * KS * KS + tap);
  }
  for (int c = tid; c < g.C; c += kAttendThreads)
    sw[KS * KS * g.C + c] = lepe_b ? __ldg(lepe_b + c) : 0.f;
  if (g.masked) {
    // Rows of the K/V slots that no copy writes (region slots padded to 8
    // rows, the buffer tail) hold zeros for the whole kernel: P is zero there
    // but 0 * NaN is not. (With masking, O never overlaps K/V.)
    for (int e = tid; e < g.stages * 2 * g.nc * g.kv_rows * 8; e += kAttendThreads) {
      const int c16 = e & 7, row = (e >> 3) % g.kv_rows;
      const int buf = (e >> 3) / g.kv_rows;  // stage * 2nc + tensor * nc + chunk
      const int st = buf / (2 * g.nc), tb = buf % (2 * g.nc);
      if (row >= nslots || (row % g.slot) >= g.n) {
        uint8_t *base = stage0 + st * g.stage_bytes +
                        (tb < g.nc ? g.off_k : g.off_v) + (tb % g.nc) * g.kv_chunk;
        *reinterpret_cast<uint4 *>(base + row * 128 + c16 * 16) = make_uint4(0, 0, 0, 0);
      }
    }
  }
  __syncthreads();

  if (warp == 0) {
    // first copies: the units of the first `stages` iterations
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      prefetch_tensormap(&tm_vh);
    }
    grid_dependency_wait();  // the routing index comes from the previous grid
    for (int it = 0; it < g.stages; ++it) {
      const int u = blockIdx.x + it * gridDim.x;
      if (u >= g.units) break;
      const int jl = read_route_lane(g, idx, u, lane);
      issue_unit<KS>(g, &tm_q, &tm_k, &tm_v, &tm_vh, idx, jl, stage0 + it * g.stage_bytes,
                     &full[it], u, lane);
    }
  }

  const int pairs = g.C / 2;

  // Each group owns the stages s with s % groups == grp (the stage count is
  // even when both groups run), so a group only ever waits for the next phase
  // of its own stages' barriers. With one stage, the second group idles.
  const int groups = g.stages >= 2 ? kGroups : 1;
  int k = 0;  // this group's iteration count
  for (int it = grp; grp < groups; it += groups, ++k) {
    const int u = blockIdx.x + it * gridDim.x;
    if (u >= g.units) break;
    const int s = it % g.stages;
    const int un = u + g.stages * gridDim.x;  // the unit this stage is refilled with
    int jl = 0;
    if (gw < g.issue_warps) {
      grid_dependency_wait();
      if (un < g.units) jl = read_route_lane(g, idx, un, lane);  // lands while we work
    }
    mbar_wait(&full[s], (it / g.stages) & 1);
    uint8_t *st = stage0 + s * g.stage_bytes;
    float *so = reinterpret_cast<float *>(st + g.off_o);

    // ---- attention
    if (g.alias) {
      // at most one task per warp: O stays in registers until every warp of
      // the group has stopped reading this unit's Q/K/V
      float o[4][4];
      const int task = gw, h = task % g.heads, qb = task / g.heads;
      if (task < g.tasks) {
        const int cc = h >> 1;
        const uint32_t qb_ = smem_u32(st + cc * g.q_chunk);
        const uint32_t kb_ = smem_u32(st + g.off_k + cc * g.kv_chunk);
        const uint32_t vb_ = smem_u32(st + g.off_v + cc * g.kv_chunk);
        attention_task<false>(g, h, qb, qb_, kb_, vb_, o, lane);
      }
      named_sync(bar_id, kGroupThreads);
      if (task < g.tasks) store_o(g, h, qb, o, so, lane);
    } else {
      for (int task = gw; task < g.tasks; task += kGroupWarps) {
        const int h = task % g.heads, qb = task / g.heads;
        const int cc = h >> 1;
        const uint32_t qb_ = smem_u32(st + cc * g.q_chunk);
        const uint32_t kb_ = smem_u32(st + g.off_k + cc * g.kv_chunk);
        const uint32_t vb_ = smem_u32(st + g.off_v + cc * g.kv_chunk);
        float o[4][4];
        if (g.masked)
          attention_task<true>(g, h, qb, qb_, kb_, vb_, o, lane);
        else
          attention_task<false>(g, h, qb, qb_, kb_, vb_, o, lane);
        store_o(g, h, qb, o, so, lane);
      }
    }
    named_sync(bar_id, kGroupThreads);  // O complete; the staging tile is free

    // ---- LePE + O -> bf16 staging tile
    uint8_t *ob = smem + g.off_out + (grp * 2 + (k & 1)) * out_tile;
    const uint8_t *hb = st + g.off_h;
    for (int item = gt; item < g.lepe_items; item += kGroupThreads) {
      const int cp = item % pairs, rest = item / pairs;
      const int x = rest % (WR ? WR : g.wr), ry0 = (rest / (WR ? WR : g.wr)) * RB;
      // the pair's weights, from shared memory each time (registers are
      // needed by the attention code in between)
      float2 wgt[KS * KS], bias;
      load_pair_weights<KS>(sw, g.C, 2 * cp, wgt, bias);
      lepe_item<KS, RB, WR, HR>(g, hb, so, ob, 2 * cp, x, ry0, wgt, bias);
    }
    fence_async_shared();  // staging tile (generic writes) before the TMA store
    named_sync(bar_id, kGroupThreads);

    // the stage is no longer read: the group's first warp refills it while
    // its last warp sends the output out (lane cc: channel chunk cc)
    if (gw < g.issue_warps && un < g.units)
      issue_unit<KS>(g, &tm_q, &tm_k, &tm_v, &tm_vh, idx, jl, st, &full[s], un, lane, gw, g.issue_warps);
    if (gw == kGroupWarps - 1 && lane < g.nc) {
      const int b = u / g.R, i = u % g.R;
      const int y0 = (i / g.S) * g.hr, x0 = (i % g.S) * g.wr;
      tma_store_4d(&tm_o, ob + lane * g.o_chunk, lane * 64, x0, y0, b);
      tma_store_commit();
      // the group's other staging tile (written next) must have been read
      tma_store_wait_read_n<1>();
    }
  }
  if (grp < groups && gw == kGroupWarps - 1 && lane < g.nc) tma_store_wait_read();
  if (tid == 0) settle_after_timeout();
}

}  // namespace bra

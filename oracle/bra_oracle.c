/*
 * bra_oracle.c -- CPU oracle for the forward pass of Bi-Level Routing
 * Attention (BRA), the attention of BiFormer.
 *
 * TEST INFRASTRUCTURE. This is the plain, slow, double-precision definition
 * the CUDA library is checked against. Only the test suite, the smoke check and
 * the CPU-baseline leg of the benchmark load it; the library never does, and
 * this file shares no code, header or table with the CUDA sources.
 *
 * Sources (web pages about BiFormer; each function cites the passage it
 * follows):
 *   [P1] "CVPR2023：BiFormer中的双层路由注意力机制解析" (cybasar.com),
 *        §2 (region-level routing idea) and §3 (implementation steps).
 *   [P2] "从静态到动态：BRA双层路由注意力如何革新视觉Transformer的计算范式"
 *        (snabindia.com), §2 (region mean pooling), §4 (TopkRouting, LePE).
 *   [P4] "Biformer注意力机制的原理及数学公式推导" (csdn), the local-window
 *        attention formula softmax(Q K^T / sqrt(d_k)) V.
 *   [P5] "BiFormer: Vision Transformer mit Bi-Level-Routing-Attention"
 *        (hyper.ai, arXiv 2303.08810 abstract): token-to-token attention over
 *        the union of the routed regions.
 *
 * Readings where the pages leave a step open (all stated in the design notes):
 *   - Regions are numbered row-major on the S x S grid and tokens row-major
 *     inside a region, which is what [P1] §3's reshape to [S^2, HW/S^2, C]
 *     produces. H and W must be multiples of S.
 *   - Routing uses all C channels (one routing per image shared by the heads),
 *     as [P1] §3 gives q_r the shape [S^2, C]. The affinity is unscaled (a
 *     positive scale does not change the order).
 *   - Top-k: largest values first, ties to the lowest region index.
 *   - Head h owns channels [h*d, (h+1)*d), d = C / heads; the attention scale
 *     is d^-1/2 (the key dimension of [P4]'s formula).
 *   - One softmax per query over all k*n routed keys jointly ([P1] §3's k_g
 *     has k*HW/S^2 keys per region and the softmax runs over the last axis).
 *   - LePE is the depthwise (groups = C) cross-correlation of V with a
 *     ks x ks kernel and a bias, zero-padded by ks/2 at the image border
 *     ([P2] §4's nn.Conv2d(dim, dim, ks, stride 1, padding ks//2,
 *     groups=dim)), added to the attention output ([P1] §3 `out += lce(v)`).
 *     No residual and no output projection.
 *
 *   - The Q/K/V projections of [P1] §3 (`q = self.q_proj(x)`, `k_proj`,
 *     `v_proj`) are per-token linear maps with a bias (PyTorch nn.Linear's
 *     default), given as one weight [3C][C] (rows 0..C-1 for q, C..2C-1 for
 *     k, 2C..3C-1 for v) and one bias [3C].
 *   - The block around BRA ("p3" below: "BiFormer架构核心思想解析" §3.1,
 *     `x = x + self.bra(self.norm1(x))`) normalises each token with
 *     nn.LayerNorm(dim): over its C channels, biased variance, eps = 1e-5
 *     (PyTorch's default), then a per-channel scale and shift.
 *   - Its ConvFFN (p3 §3.1 "ConvFFN: a feed-forward network with a 3x3
 *     depthwise convolution"; p1 §4: a two-layer MLP of ratio 3) is read as
 *     fc2(GELU(dwconv3x3(fc1(x)))): fc1 = Linear(C, 3C), a depthwise 3x3
 *     convolution with bias and zero padding 1 in the 3C-channel hidden
 *     layer, the exact (erf) GELU of nn.GELU, fc2 = Linear(3C, C).
 *
 *   - The backward of attend holds the routing fixed: [P2] §4's TopkRouting
 *     with diff_routing=False passes no gradient to the routing, so the
 *     index is a constant of the attention and only q, k, v and the LePE's
 *     weight and bias receive gradients.
 *
 * All tensors are contiguous channels-last [B, H, W, C] arrays of double.
 * Functions return 0 on success and 1 on an invalid argument.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1

typedef struct {
  int B, H, W, C, S;
  int R;      /* regions per image, S*S */
  int hr, wr; /* region height and width in tokens */
  int n;      /* tokens per region */
} geom;

static int make_geom(int B, int H, int W, int C, int S, geom *g) {
  if (B < 0 || H <= 0 || W <= 0 || C <= 0 || S <= 0) return ORACLE_EINVAL;
  if (H % S || W % S) return ORACLE_EINVAL;
  g->B = B; g->H = H; g->W = W; g->C = C; g->S = S;
  g->R = S * S;
  g->hr = H / S;
  g->wr = W / S;
  g->n = g->hr * g->wr;
  return ORACLE_OK;
}

/* Region partition, [P1] §3: token t of region r (row-major grid of S x S
 * regions, row-major tokens inside a region) sits at image row y, column x. */
static void region_token(const geom *g, int r, int t, int *y, int *x) {
  int ry = r / g->S, rx = r % g->S;
  *y = ry * g->hr + t / g->wr;
  *x = rx * g->wr + t % g->wr;
}

static size_t offset_of(const geom *g, int b, int y, int x) {
  return (((size_t)b * g->H + y) * g->W + x) * (size_t)g->C;
}

/* ---------------------------------------------------------------------------
 * Step 1: region-level mean of a token map ([P1] §3 `q.mean(dim=1)`; [P2] §2
 * pools each region by its average). out is [B, S*S, C].
 */
int oracle_region_means(const double *x, int B, int H, int W, int C, int S,
                        double *out) {
  geom g;
  if (!x || !out || make_geom(B, H, W, C, S, &g)) return ORACLE_EINVAL;
  for (int b = 0; b < B; ++b)
    for (int r = 0; r < g.R; ++r)
      for (int c = 0; c < C; ++c) {
        double sum = 0.0;
        for (int t = 0; t < g.n; ++t) {
          int y, xx;
          region_token(&g, r, t, &y, &xx);
          sum += x[offset_of(&g, b, y, xx) + c];
        }
        out[((size_t)b * g.R + r) * C + c] = sum / g.n;
      }
  return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * Step 2: region affinity A_r = q_r k_r^T over all C channels ([P1] §3;
 * [P2] §4 TopkRouting's attn_logit, without the positive scale). A is
 * [B, S*S, S*S].
 */
int oracle_affinity(const double *q, const double *k, int B, int H, int W,
                    int C, int S, double *A) {
  geom g;
  if (!q || !k || !A || make_geom(B, H, W, C, S, &g)) return ORACLE_EINVAL;
  size_t nm = (size_t)B * g.R * C;
  double *qm = malloc(nm * sizeof(double));
  double *km = malloc(nm * sizeof(double));
  if (!qm || !km) { free(qm); free(km); return ORACLE_EINVAL; }
  oracle_region_means(q, B, H, W, C, S, qm);
  oracle_region_means(k, B, H, W, C, S, km);
  for (int b = 0; b < B; ++b)
    for (int i = 0; i < g.R; ++i)
      for (int j = 0; j < g.R; ++j) {
        const double *qi = qm + ((size_t)b * g.R + i) * C;
        const double *kj = km + ((size_t)b * g.R + j) * C;
        double dot = 0.0;
        for (int c = 0; c < C; ++c) dot += qi[c] * kj[c];
        A[((size_t)b * g.R + i) * g.R + j] = dot;
      }
  free(qm);
  free(km);
  return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * Step 3: per-row top-k of the affinity ([P1] §3 `torch.topk(A_r, k).indices`;
 * [P2] §4). Largest first; among equal values the lowest column wins. A is
 * [rows, R]; idx is [rows, topk].
 */
int oracle_topk(const double *A, int rows, int R, int topk, int32_t *idx) {
  if (!A || !idx || rows < 0 || R <= 0 || topk <= 0 || topk > R)
    return ORACLE_EINVAL;
  unsigned char *taken = malloc((size_t)R);
  if (!taken) return ORACLE_EINVAL;
  for (int i = 0; i < rows; ++i) {
    const double *row = A + (size_t)i * R;
    memset(taken, 0, (size_t)R);
    for (int m = 0; m < topk; ++m) {
      int best = -1;
      for (int j = 0; j < R; ++j) {
        if (taken[j]) continue;
        if (best < 0 || row[j] > row[best]) best = j; /* strict: ties keep lower j */
      }
      taken[best] = 1;
      idx[(size_t)i * topk + m] = best;
    }
  }
  free(taken);
  return ORACLE_OK;
}

/* Routing = steps 1-3. idx is [B, S*S, topk]; A (optional) is [B, S*S, S*S]. */
int oracle_route(const double *q, const double *k, int B, int H, int W, int C,
                 int S, int topk, int32_t *idx, double *A_out) {
  geom g;
  if (!q || !k || !idx || make_geom(B, H, W, C, S, &g)) return ORACLE_EINVAL;
  if (topk <= 0 || topk > g.R) return ORACLE_EINVAL;
  size_t na = (size_t)B * g.R * g.R;
  double *A = A_out ? A_out : malloc((na ? na : 1) * sizeof(double));
  if (!A) return ORACLE_EINVAL;
  int rc = oracle_affinity(q, k, B, H, W, C, S, A);
  if (!rc) rc = oracle_topk(A, B * g.R, g.R, topk, idx);
  if (!A_out) free(A);
  return rc;
}

/* ---------------------------------------------------------------------------
 * Step 4: token-to-token attention over the routed regions ([P1] §3: gather
 * k and v of the k routed regions, attn = softmax(q k_g^T * scale), out =
 * attn v_g; [P5]: attention over the union of the routed regions; [P4]: scale
 * 1/sqrt(d_k)). The gathered keys are never stored here either: each query
 * walks the routed regions directly.
 */
typedef struct {
  const double *q, *k, *v;
  const int32_t *idx;
  geom g;
  int heads, topk;
  double *out;
  int status;
} attn_job;

/* Logits, probabilities and output of one query (b, region i, slot t, head h).
 * probs / keys (optional) receive the k*n probabilities and the flat token
 * index y*W + x of each key, in routed order. */
static int attend_one(const attn_job *J, int b, int i, int t, int h,
                      double *logit, double *probs, int32_t *keys,
                      double *out_vec) {
  const geom *g = &J->g;
  int d = g->C / J->heads;
  double scale = 1.0 / sqrt((double)d);
  int y, x;
  region_token(g, i, t, &y, &x);
  const double *qv = J->q + offset_of(g, b, y, x) + (size_t)h * d;
  int nk = J->topk * g->n;
  for (int m = 0; m < J->topk; ++m) {
    int j = J->idx[((size_t)b * g->R + i) * J->topk + m];
    if (j < 0 || j >= g->R) return ORACLE_EINVAL;
    for (int s = 0; s < g->n; ++s) {
      int yk, xk;
      region_token(g, j, s, &yk, &xk);
      const double *kv = J->k + offset_of(g, b, yk, xk) + (size_t)h * d;
      double dot = 0.0;
      for (int e = 0; e < d; ++e) dot += qv[e] * kv[e];
      logit[m * g->n + s] = dot * scale;
      if (keys) keys[m * g->n + s] = yk * g->W + xk;
    }
  }
  /* softmax over all nk keys jointly: subtract the max, exponentiate, divide */
  double mx = logit[0];
  for (int a = 1; a < nk; ++a) if (logit[a] > mx) mx = logit[a];
  double sum = 0.0;
  for (int a = 0; a < nk; ++a) { logit[a] = exp(logit[a] - mx); sum += logit[a]; }
  for (int a = 0; a < nk; ++a) logit[a] /= sum;
  if (probs) memcpy(probs, logit, (size_t)nk * sizeof(double));
  if (out_vec) {
    for (int e = 0; e < d; ++e) out_vec[e] = 0.0;
    for (int m = 0; m < J->topk; ++m) {
      int j = J->idx[((size_t)b * g->R + i) * J->topk + m];
      for (int s = 0; s < g->n; ++s) {
        int yk, xk;
        region_token(g, j, s, &yk, &xk);
        const double *vv = J->v + offset_of(g, b, yk, xk) + (size_t)h * d;
        double p = logit[m * g->n + s];
        for (int e = 0; e < d; ++e) out_vec[e] += p * vv[e];
      }
    }
  }
  return ORACLE_OK;
}

typedef struct {
  attn_job *job;
  int tid, nthreads;
} attn_worker;

static void *attn_thread(void *arg) {
  attn_worker *w = (attn_worker *)arg;
  attn_job *J = w->job;
  const geom *g = &J->g;
  int d = g->C / J->heads;
  double *logit = malloc((size_t)J->topk * g->n * sizeof(double));
  if (!logit) { J->status = ORACLE_EINVAL; return NULL; }
  long units = (long)g->B * g->R;
  for (long u = w->tid; u < units; u += w->nthreads) {
    int b = (int)(u / g->R), i = (int)(u % g->R);
    for (int t = 0; t < g->n; ++t) {
      int y, x;
      region_token(g, i, t, &y, &x);
      for (int h = 0; h < J->heads; ++h) {
        double *o = J->out + offset_of(g, b, y, x) + (size_t)h * d;
        if (attend_one(J, b, i, t, h, logit, NULL, NULL, o))
          J->status = ORACLE_EINVAL;
      }
    }
  }
  free(logit);
  return NULL;
}

static int run_threads(void *(*fn)(void *), attn_job *job, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  attn_worker *ws = malloc(sizeof(attn_worker) * (size_t)nthreads);
  pthread_t *th = malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!ws || !th) { free(ws); free(th); return ORACLE_EINVAL; }
  for (int t = 0; t < nthreads; ++t) {
    ws[t].job = job; ws[t].tid = t; ws[t].nthreads = nthreads;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, fn, &ws[t]);
  fn(&ws[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(ws);
  free(th);
  return ORACLE_OK;
}

static int attn_args_ok(const double *q, const double *k, const double *v,
                        const int32_t *idx, int B, int H, int W, int C,
                        int heads, int S, int topk, geom *g) {
  if (!q || !k || !v || !idx || make_geom(B, H, W, C, S, g)) return 0;
  if (heads <= 0 || C % heads) return 0;
  if (topk <= 0 || topk > g->R) return 0;
  return 1;
}

/* Attention part only: out[B, H, W, C] = routed softmax attention. */
int oracle_routed_attention(const double *q, const double *k, const double *v,
                            const int32_t *idx, int B, int H, int W, int C,
                            int heads, int S, int topk, double *out,
                            int nthreads) {
  attn_job J;
  if (!out || !attn_args_ok(q, k, v, idx, B, H, W, C, heads, S, topk, &J.g))
    return ORACLE_EINVAL;
  J.q = q; J.k = k; J.v = v; J.idx = idx;
  J.heads = heads; J.topk = topk; J.out = out; J.status = ORACLE_OK;
  if (run_threads(attn_thread, &J, nthreads)) return ORACLE_EINVAL;
  return J.status;
}

/* Probabilities of one query: probs[topk*n], keys[topk*n] (flat y*W + x),
 * out_vec[d] (optional). Used by the softmax-sum and order checks. */
int oracle_query_probs(const double *q, const double *k, const double *v,
                       const int32_t *idx, int B, int H, int W, int C,
                       int heads, int S, int topk, int b, int y, int x, int h,
                       double *probs, int32_t *keys, double *out_vec) {
  attn_job J;
  if (!probs || !attn_args_ok(q, k, v, idx, B, H, W, C, heads, S, topk, &J.g))
    return ORACLE_EINVAL;
  if (b < 0 || b >= B || y < 0 || y >= H || x < 0 || x >= W || h < 0 ||
      h >= heads)
    return ORACLE_EINVAL;
  J.q = q; J.k = k; J.v = v; J.idx = idx;
  J.heads = heads; J.topk = topk; J.out = NULL; J.status = ORACLE_OK;
  const geom *g = &J.g;
  int i = (y / g->hr) * g->S + x / g->wr;
  int t = (y % g->hr) * g->wr + x % g->wr;
  double *logit = malloc((size_t)topk * g->n * sizeof(double));
  if (!logit) return ORACLE_EINVAL;
  int rc = attend_one(&J, b, i, t, h, logit, probs, keys, out_vec);
  free(logit);
  return rc;
}

/* ---------------------------------------------------------------------------
 * Step 5: LePE ([P2] §4: nn.Conv2d(dim, dim, kernel_size=ks, stride=1,
 * padding=ks//2, groups=dim) applied to V; bias included as nn.Conv2d's
 * default). Cross-correlation, zero padding at the image border.
 * w is [C, ks, ks], bias [C] or NULL (zero). out is [B, H, W, C].
 */
int oracle_lepe(const double *v, int B, int H, int W, int C, const double *w,
                const double *bias, int ks, double *out) {
  if (!v || !w || !out || B < 0 || H <= 0 || W <= 0 || C <= 0) return ORACLE_EINVAL;
  if (ks <= 0 || ks % 2 == 0) return ORACLE_EINVAL;
  int pad = ks / 2;
  for (int b = 0; b < B; ++b)
    for (int y = 0; y < H; ++y)
      for (int x = 0; x < W; ++x)
        for (int c = 0; c < C; ++c) {
          double acc = bias ? bias[c] : 0.0;
          for (int u = 0; u < ks; ++u)
            for (int s = 0; s < ks; ++s) {
              int yy = y + u - pad, xx = x + s - pad;
              if (yy < 0 || yy >= H || xx < 0 || xx >= W) continue;
              acc += w[((size_t)c * ks + u) * ks + s] *
                     v[(((size_t)b * H + yy) * W + xx) * C + c];
            }
          out[(((size_t)b * H + y) * W + x) * C + c] = acc;
        }
  return ORACLE_OK;
}

/* Attend = step 4 + step 5 (out = attention + LePE(v)), given the routing. */
int oracle_attend(const double *q, const double *k, const double *v,
                  const int32_t *idx, int B, int H, int W, int C, int heads,
                  int S, int topk, const double *w, const double *bias, int ks,
                  double *out, int nthreads) {
  geom g;
  if (!out || !w || !attn_args_ok(q, k, v, idx, B, H, W, C, heads, S, topk, &g))
    return ORACLE_EINVAL;
  size_t total = (size_t)B * H * W * C;
  double *lepe = malloc((total ? total : 1) * sizeof(double));
  if (!lepe) return ORACLE_EINVAL;
  int rc = oracle_routed_attention(q, k, v, idx, B, H, W, C, heads, S, topk,
                                   out, nthreads);
  if (!rc) rc = oracle_lepe(v, B, H, W, C, w, bias, ks, lepe);
  if (!rc)
    for (size_t e = 0; e < total; ++e) out[e] += lepe[e];
  free(lepe);
  return rc;
}

/* The whole forward: routing (steps 1-3), then attend (steps 4-5). */
int oracle_forward(const double *q, const double *k, const double *v, int B,
                   int H, int W, int C, int heads, int S, int topk,
                   const double *w, const double *bias, int ks, int32_t *idx,
                   double *out, int nthreads) {
  int rc = oracle_route(q, k, B, H, W, C, S, topk, idx, NULL);
  if (rc) return rc;
  return oracle_attend(q, k, v, idx, B, H, W, C, heads, S, topk, w, bias, ks,
                       out, nthreads);
}

/*
 * [P1] §3 "线性投影获取Q,K,V": q = x W_q^T + b_q, k = x W_k^T + b_k,
 * v = x W_v^T + b_v for every token (the projections act on each token alone,
 * so the region reshape before them changes nothing). x is [M][C] (M tokens),
 * w is [3C][C] in the nn.Linear [out][in] layout, bias is [3C] or NULL (zero);
 * q, k and v are [M][C].
 */
int oracle_qkv_project(const double *x, int M, int C, const double *w, const double *bias,
                       double *q, double *k, double *v) {
  if (!x || !w || !q || !k || !v || M < 0 || C <= 0) return ORACLE_EINVAL;
  double *outs[3] = {q, k, v};
  for (int m = 0; m < M; ++m)
    for (int t = 0; t < 3; ++t)
      for (int j = 0; j < C; ++j) {
        const double *wr = w + ((size_t)t * C + j) * C;
        double acc = bias ? bias[(size_t)t * C + j] : 0.0;
        for (int c = 0; c < C; ++c) acc += x[(size_t)m * C + c] * wr[c];
        outs[t][(size_t)m * C + j] = acc;
      }
  return ORACLE_OK;
}

/*
 * p3 ("BiFormer架构核心思想解析") §3.1, `self.norm1 = nn.LayerNorm(dim)`:
 * y[m][c] = (x[m][c] - mean_m) / sqrt(var_m + eps) * gamma[c] + beta[c],
 * with mean_m and var_m (biased: divided by C) over the C channels of token m.
 * gamma and beta may be NULL (1 and 0).
 */
int oracle_layer_norm(const double *x, int M, int C, const double *gamma,
                      const double *beta, double eps, double *y) {
  if (!x || !y || M < 0 || C <= 0 || !(eps >= 0.0)) return ORACLE_EINVAL;
  for (int m = 0; m < M; ++m) {
    const double *xr = x + (size_t)m * C;
    double mean = 0.0;
    for (int c = 0; c < C; ++c) mean += xr[c];
    mean /= C;
    double var = 0.0;
    for (int c = 0; c < C; ++c) var += (xr[c] - mean) * (xr[c] - mean);
    var /= C;
    const double rstd = 1.0 / sqrt(var + eps);
    for (int c = 0; c < C; ++c)
      y[(size_t)m * C + c] = (xr[c] - mean) * rstd * (gamma ? gamma[c] : 1.0) +
                             (beta ? beta[c] : 0.0);
  }
  return ORACLE_OK;
}

/*
 * A linear layer (nn.Linear): y[m][n] = sum_k x[m][k] w[n][k] + bias[n]
 * (bias may be NULL); x [M][K], w [N][K], y [M][N]. Used for the ConvFFN's
 * fc1 and fc2 (p3 §3.1, p1 §4).
 */
int oracle_linear(const double *x, int M, int K, const double *w, int N, const double *bias,
                  double *y) {
  if (!x || !w || !y || M < 0 || K <= 0 || N <= 0) return ORACLE_EINVAL;
  for (int m = 0; m < M; ++m)
    for (int n = 0; n < N; ++n) {
      double acc = bias ? bias[n] : 0.0;
      const double *wr = w + (size_t)n * K;
      for (int k = 0; k < K; ++k) acc += x[(size_t)m * K + k] * wr[k];
      y[(size_t)m * N + n] = acc;
    }
  return ORACLE_OK;
}

/* nn.GELU (exact form): x * (1 + erf(x / sqrt 2)) / 2, element by element. */
int oracle_gelu(const double *x, size_t n, double *y) {
  if (!x || !y) return ORACLE_EINVAL;
  for (size_t i = 0; i < n; ++i) y[i] = 0.5 * x[i] * (1.0 + erf(x[i] / sqrt(2.0)));
  return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * Backward of attend (out = attention + LePE(v), the routing fixed; see the
 * readings above). dout is dL/dout. For one query (its row of the softmax P
 * over the k*n routed keys, its attention output O, D = dout . O):
 *   dv[key] += P[key] dout                         (O = sum P v)
 *   dS[key]  = P[key] (dout . v[key] - D)          (softmax)
 *   dq      += scale dS[key] k[key],   dk[key] += scale dS[key] q
 * and for the LePE (cross-correlation, zero padding):
 *   dv[y][x][c] += sum_{u,s} w[c][u][s] dout[y - u + pad][x - s + pad][c]
 *   dw[c][u][s]  = sum_{b,y,x} dout[y][x][c] v[y + u - pad][x + s - pad][c]
 *   db[c]        = sum_{b,y,x} dout[y][x][c]
 * (terms whose position falls outside the image are absent). dq, dk, dv are
 * [B, H, W, C]; dw [C, ks, ks]; db [C] or NULL. All outputs are overwritten.
 */
int oracle_attend_backward(const double *q, const double *k, const double *v,
                           const int32_t *idx, int B, int H, int W, int C, int heads,
                           int S, int topk, const double *w, int ks, const double *dout,
                           double *dq, double *dk, double *dv, double *dw, double *db) {
  geom g;
  if (!w || !dout || !dq || !dk || !dv || !dw ||
      !attn_args_ok(q, k, v, idx, B, H, W, C, heads, S, topk, &g))
    return ORACLE_EINVAL;
  if (ks <= 0 || ks % 2 == 0) return ORACLE_EINVAL;
  size_t total = (size_t)B * H * W * C;
  memset(dq, 0, total * sizeof(double));
  memset(dk, 0, total * sizeof(double));
  memset(dv, 0, total * sizeof(double));
  memset(dw, 0, (size_t)C * ks * ks * sizeof(double));
  if (db) memset(db, 0, (size_t)C * sizeof(double));
  attn_job J = {q, k, v, idx, g, heads, topk, NULL, 0};
  int d = C / heads, nk = topk * g.n;
  double scale = 1.0 / sqrt((double)d);
  double *logit = malloc((size_t)nk * sizeof(double));
  double *probs = malloc((size_t)nk * sizeof(double));
  int32_t *keys = malloc((size_t)nk * sizeof(int32_t));
  double *o = malloc((size_t)d * sizeof(double));
  int rc = (logit && probs && keys && o) ? ORACLE_OK : ORACLE_EINVAL;
  for (int b = 0; b < B && !rc; ++b)
    for (int i = 0; i < g.R && !rc; ++i)
      for (int t = 0; t < g.n && !rc; ++t)
        for (int h = 0; h < heads && !rc; ++h) {
          rc = attend_one(&J, b, i, t, h, logit, probs, keys, o);
          if (rc) break;
          int y, x;
          region_token(&g, i, t, &y, &x);
          size_t qo = offset_of(&g, b, y, x) + (size_t)h * d;
          const double *go = dout + qo;
          double D = 0.0;
          for (int e = 0; e < d; ++e) D += go[e] * o[e];
          for (int a = 0; a < nk; ++a) {
            size_t ko = ((size_t)b * H * W + keys[a]) * C + (size_t)h * d;
            double dp = 0.0;
            for (int e = 0; e < d; ++e) dp += go[e] * v[ko + e];
            double ds = probs[a] * (dp - D);
            for (int e = 0; e < d; ++e) {
              dv[ko + e] += probs[a] * go[e];
              dq[qo + e] += scale * ds * k[ko + e];
              dk[ko + e] += scale * ds * q[qo + e];
            }
          }
        }
  free(logit);
  free(probs);
  free(keys);
  free(o);
  if (rc) return rc;
  int pad = ks / 2;
  for (int b = 0; b < B; ++b)
    for (int y = 0; y < H; ++y)
      for (int x = 0; x < W; ++x)
        for (int c = 0; c < C; ++c) {
          double go = dout[(((size_t)b * H + y) * W + x) * C + c];
          if (db) db[c] += go;
          for (int u = 0; u < ks; ++u)
            for (int s2 = 0; s2 < ks; ++s2) {
              int yy = y + u - pad, xx = x + s2 - pad;
              if (yy < 0 || yy >= H || xx < 0 || xx >= W) continue;
              size_t vo = (((size_t)b * H + yy) * W + xx) * C + c;
              dw[((size_t)c * ks + u) * ks + s2] += go * v[vo];
              dv[vo] += w[((size_t)c * ks + u) * ks + s2] * go;
            }
        }
  return ORACLE_OK;
}

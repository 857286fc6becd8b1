/*
 * bra.h -- C ABI of the Bi-Level Routing Attention (BRA) forward for B300
 * (sm_103a). BRA is the attention of BiFormer.
 *
 * Sources of the operations (web pages about BiFormer):
 *   "CVPR2023：BiFormer中的双层路由注意力机制解析" (cybasar.com), §2-§3:
 *       region partition, region-mean Q/K, region affinity, top-k routing,
 *       gather of the routed K/V, softmax attention, out += lce(v).
 *   "从静态到动态：BRA双层路由注意力如何革新视觉Transformer的计算范式"
 *       (snabindia.com), §2 (mean pooling per region), §4 (TopkRouting,
 *       LePE as a depthwise nn.Conv2d with padding ks//2, groups = dim).
 *   "BiFormer: Vision Transformer mit Bi-Level-Routing-Attention"
 *       (hyper.ai abstract of arXiv 2303.08810): token-to-token attention
 *       over the union of the routed regions.
 *
 * Conventions shared by every entry point
 *   Layout     q, k, v and out are contiguous channels-last [B, H, W, C]
 *              arrays in DEVICE memory, of type float32 (BRA_F32) or bfloat16
 *              (BRA_BF16); out has the type of q. Regions are the S x S grid
 *              numbered row-major; region r covers rows (r / S) * H/S ... and
 *              columns (r % S) * W/S ... . Head h owns channels
 *              [h * d, (h + 1) * d), d = C / heads.
 *   LePE       lepe_w is float32 [C, ks, ks] (device), lepe_b float32 [C]
 *              (device) or NULL for no bias. Zero padding at the image border.
 *   Routing    idx is int32 [B, S*S, topk] (device): for each query region the
 *              topk regions of largest affinity, largest first, ties to the
 *              lowest region index. The affinity is mean(q_r) . mean(k_r)
 *              over all C channels, computed in float32.
 *   Ownership  The caller allocates and owns every buffer. No entry point
 *              allocates, frees or synchronises: all work is enqueued on
 *              `stream` (a cudaStream_t; NULL is the legacy default stream).
 *   Errors     Arguments are checked before anything is enqueued; on a
 *              non-zero return nothing was launched. A launch failure returns
 *              BRA_ERR_CUDA. Faults that happen on the device surface at the
 *              caller's next synchronisation. Device-side checks (a wait that
 *              gave up, a routing index out of range) set a status word read
 *              by bra_device_status(). Nothing throws across the ABI.
 *   Aliasing   out must not overlap q, k or v.
 *   Threads    Except for bra_forward_static, the library keeps no per-call
 *              state: calls on different streams may run concurrently.
 *              bra_forward_static keeps its routing index in one fixed
 *              array per device, so its calls must not overlap on the GPU.
 *   Empty      B == 0 is valid and enqueues nothing.
 */
#ifndef BRA_H_
#define BRA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum bra_status {
  BRA_OK = 0,
  BRA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment, aliasing */
  BRA_ERR_UNSUPPORTED = 2, /* valid BRA, but a shape this build does not run */
  BRA_ERR_CUDA = 3,        /* a CUDA call or launch failed */
  BRA_ERR_TIMEOUT = 4      /* a device-side wait gave up (bra_device_status) */
};

enum bra_dtype { BRA_F32 = 0, BRA_BF16 = 1 };

/*
 * bra_route -- region-level routing (steps "q_r = q.mean", "A_r = q_r k_r^T",
 * "I_r = topk(A_r)" of the cybasar page §3; TopkRouting of the snabindia page
 * §4).
 *   q, k      [B, H, W, C] device, dtype
 *   B..C, S   map size and region grid; H and W must be multiples of S
 *   topk      1 <= topk <= S*S
 *   idx       out: int32 [B, S*S, topk] device
 *   affinity  out (optional, may be NULL): float32 [B, S*S, S*S] device, the
 *             unscaled region affinity the selection was taken on
 * Supported: S*S <= 1024, B <= 65535, and C * element size a power of two
 * from 16 to 512 bytes (bf16: C in {8, 16, ..., 256}; f32: C in {4, ..., 128});
 * otherwise BRA_ERR_UNSUPPORTED.
 */
int bra_route(const void *q, const void *k, int B, int H, int W, int C, int S,
              int topk, int dtype, int32_t *idx, float *affinity, void *stream);

/*
 * bra_attend -- token-to-token attention over the routed regions plus LePE
 * (steps "k_g = gather(k, I_r)", "attn = softmax(q k_g^T * scale)",
 * "out = attn v_g", "out += lce(v)" of the cybasar page §3; the LePE conv of
 * the snabindia page §4). The gathered K/V are never written to memory.
 *   q, k, v   [B, H, W, C] device, dtype
 *   idx       int32 [B, S*S, topk] device, values in [0, S*S) (an index out of
 *             range reads zeros and sets the device status word)
 *   heads     C % heads == 0; scale is (C/heads)^-1/2
 *   lepe_w/b  see above; lepe_ks odd, 1..7
 *   out       [B, H, W, C] device, dtype of q
 * Supported: bf16 with C % 64 == 0 and d == 32; f32 with C % 4 == 0 and
 * d <= 64; shared-memory footprint within the per-block limit. Otherwise
 * BRA_ERR_UNSUPPORTED. bf16 maps whose regions hold fewer than 16 tokens and
 * whose whole image fits in shared memory one 64-channel chunk at a time
 * (about 250 tokens) run an image-resident kernel (regions of at most 8
 * tokens its local form: K and a zero-bordered V halo in shared memory, two
 * CTAs to an SM); the others a persistent kernel over query regions. The
 * choice depends on the shape only.
 */
int bra_attend(const void *q, const void *k, const void *v, const int32_t *idx,
               int B, int H, int W, int C, int heads, int S, int topk,
               const float *lepe_w, const float *lepe_b, int lepe_ks, int dtype,
               void *out, void *stream);

/*
 * bra_attend_tc -- bra_attend computed with the 5th-generation tensor cores
 * (tcgen05.mma, accumulators in tensor memory) for maps of 8 x 8 regions with
 * C = 64 (2 heads of 32), topk <= 4 and lepe_ks 1, 3 or 5: S = Q K^T for both
 * heads at once against a block-diagonal Q operand (M = 128), P V block by
 * block, the softmax and LePE on separate warps. Arguments, layout and errors
 * as bra_attend; other shapes return BRA_ERR_UNSUPPORTED. The result equals
 * bra_attend's within the bf16 tolerance (the exponentials and row sums are
 * formed in the same precision; the order of additions differs). On the
 * B300 this variant is measured as fast as bra_attend on the stage-1 shape
 * alone but slower inside the forward and on the 512 x 512 shape, so
 * bra_forward does not use it.
 */
int bra_attend_tc(const void *q, const void *k, const void *v, const int32_t *idx, int B,
                  int H, int W, int C, int heads, int S, int topk, const float *lepe_w,
                  const float *lepe_b, int lepe_ks, int dtype, void *out, void *stream);

/*
 * bra_forward -- the whole forward: the routing of bra_route, then the
 * attention of bra_attend, on one stream.
 *   idx_workspace  device buffer of bra_idx_workspace_bytes(B, S, topk)
 *                  bytes; receives the routing index, the same bit for bit
 *                  as bra_route's.
 * Other arguments as above. bf16 maps with at most 64 regions and C in {64,
 * 128, 256} that the image-resident attend kernel takes run as one kernel
 * with the routing computed inside it (one cluster of C / 64 CTAs per
 * image): always for regions of at most 8 tokens, and for regions of 9 to 15
 * tokens when every image's cluster is resident at once on the device. Other
 * problems run the routing kernel and then the attend kernel.
 */
int bra_forward(const void *q, const void *k, const void *v, int B, int H,
                int W, int C, int heads, int S, int topk, const float *lepe_w,
                const float *lepe_b, int lepe_ks, int dtype,
                int32_t *idx_workspace, void *out, void *stream);

/*
 * bra_forward_static -- bra_forward for callers that cannot allocate device
 * memory. It has no counterpart on the pages: it exists for callers that are
 * handed only their input and output buffers and may not call cudaMalloc,
 * such as a plugin inside an inference engine that owns the whole device
 * memory budget, or a latency-critical loop where cudaMalloc's implicit
 * synchronisation is not acceptable. The routing index lives in a fixed
 * array inside the library (BRA_STATIC_IDX_MAX_ENTRIES int32 = 1 MiB per
 * GPU, held until the process exits) instead of a caller workspace; nothing
 * is allocated, freed or synchronised.
 *   Arguments    as bra_forward, without idx_workspace.
 *   Limit        B * S*S * topk <= BRA_STATIC_IDX_MAX_ENTRIES, otherwise
 *                BRA_ERR_UNSUPPORTED and nothing is launched.
 *   First call   the first call on each device looks up the array's device
 *                address (cudaGetSymbolAddress) with that device current;
 *                make that first call before any stream capture.
 *   Sharing      every call on a device uses the same array: calls that
 *                overlap on the GPU (on different streams, or from several
 *                threads) race on it. Serialise them, or use bra_forward
 *                with a workspace per stream. Each call overwrites the index
 *                it reads, so no clearing is needed between calls.
 *   The index is not returned; use bra_route for it.
 */
#define BRA_STATIC_IDX_MAX_ENTRIES (1 << 18)
int bra_forward_static(const void *q, const void *k, const void *v, int B,
                       int H, int W, int C, int heads, int S, int topk,
                       const float *lepe_w, const float *lepe_b, int lepe_ks,
                       int dtype, void *out, void *stream);

/*
 * bra_qkv_project -- the linear projections in front of BRA ("q =
 * self.q_proj(x)", "k = self.k_proj(x)", "v = self.v_proj(x)" of the cybasar
 * page §3), per token, on the tensor cores:
 *   q[m][j] = sum_c x[m][c] w[j][c] + bias[j]
 *   k[m][j] = sum_c x[m][c] w[C + j][c] + bias[C + j]
 *   v[m][j] = sum_c x[m][c] w[2C + j][c] + bias[2C + j]
 * with f32 accumulation and one rounding to bf16.
 *   x        [M][C] device bf16 (e.g. a channels-last [B, H, W, C] map,
 *            M = B H W)
 *   w        [3C][C] device bf16, the [out][in] layout of a linear layer
 *   bias     [3C] device float32, or NULL for none
 *   q, k, v  out: [M][C] device bf16 each (the inputs of bra_forward)
 * Supported: bf16, C a multiple of 64 from 64 to 256; otherwise
 * BRA_ERR_UNSUPPORTED. Pointers 16-byte aligned, outputs disjoint from each
 * other and from the inputs (else BRA_ERR_INVALID_ARG). M == 0 enqueues
 * nothing.
 */
int bra_qkv_project(const void *x, const void *w, const float *bias, long long M, int C,
                    int dtype, void *q, void *k, void *v, void *stream);

/*
 * bra_layer_norm -- the LayerNorm of the BiFormer block ("self.norm1 =
 * nn.LayerNorm(dim)" of the page "BiFormer架构核心思想解析" §3.1) over the C
 * channels of every token:
 *   y[m][c] = (x[m][c] - mean_m) / sqrt(var_m + eps) * gamma[c] + beta[c]
 * with the biased variance; float32 arithmetic, one rounding to bf16.
 *   x, y     [M][C] device bf16 (y may be x: in place)
 *   gamma, beta  [C] device float32, or NULL for 1 and 0
 * Supported: bf16 with C in {64, 128, 256}; otherwise BRA_ERR_UNSUPPORTED.
 * eps < 0, a NULL or unaligned (16-byte) x or y, or y partly overlapping x:
 * BRA_ERR_INVALID_ARG. M == 0 enqueues nothing.
 */
int bra_layer_norm(const void *x, const float *gamma, const float *beta, long long M, int C,
                   float eps, int dtype, void *y, void *stream);

/*
 * bra_residual_add -- y = x + r element by element (the residual of the
 * same block, "x = x + self.bra(...)"), the float32 sum rounded once to bf16.
 *   x, r, y  n elements each, device bf16; y may be x or r.
 * Supported: bf16 with n a multiple of 8; otherwise BRA_ERR_UNSUPPORTED.
 * NULL or unaligned pointers, or y partly overlapping x or r:
 * BRA_ERR_INVALID_ARG.
 */
int bra_residual_add(const void *x, const void *r, long long n, int dtype, void *y,
                     void *stream);

/*
 * bra_linear -- a linear layer (nn.Linear) on the tensor cores, the kernel of
 * bra_qkv_project with one output: y[m][n] = sum_k x[m][k] w[n][k] + bias[n]
 * (+ residual[m][n] when residual is not NULL), f32 accumulation, one
 * rounding to bf16. The ConvFFN's fc1 and fc2 (page "BiFormer架构核心思想解析"
 * §3.1; the cybasar page §4: ratio 3).
 *   x [M][K], w [N][K] device bf16; bias [N] device float32 or NULL;
 *   residual [M][N] device bf16 or NULL (it may be y); y [M][N] device bf16.
 * Supported: bf16, K and N multiples of 64 whose tiles fit in shared memory
 * (K up to 384 with N = 64 or 128; K up to 256 with N up to 768); otherwise
 * BRA_ERR_UNSUPPORTED. NULL or unaligned (16-byte) pointers, y overlapping x
 * or w, or partly overlapping residual: BRA_ERR_INVALID_ARG.
 */
int bra_linear(const void *x, const void *w, const float *bias, long long M, int K, int N,
               const void *residual, int dtype, void *y, void *stream);

/*
 * bra_dwconv_gelu -- the hidden layer of the ConvFFN: y = GELU(dwconv3x3(h)),
 * the depthwise 3 x 3 cross-correlation with a bias and zero padding 1 at the
 * image border (the LePE's operation with a 3 x 3 kernel), then GELU in its
 * exact form x (1 + erf(x / sqrt 2)) / 2; float32 arithmetic, one rounding.
 *   h, y      [B, H, W, Ch] device bf16 (disjoint)
 *   w         [Ch, 3, 3] device float32; bias [Ch] device float32 or NULL
 * Supported: bf16, Ch a multiple of 8 up to 384 (the hidden layer of
 * C = 64 or 128; a block holds all channels of an 8-token tile row);
 * otherwise BRA_ERR_UNSUPPORTED.
 */
int bra_dwconv_gelu(const void *h, const float *w, const float *bias, int B, int H, int W,
                    int Ch, int dtype, void *y, void *stream);

/*
 * bra_attend_backward -- the gradients of bra_attend's output (routed
 * attention + LePE) with the routing held fixed: TopkRouting with
 * diff_routing=False (the snabindia page §4) passes no gradient to the
 * routing, so idx is a constant. Given dout = dL/dout, with P a query's
 * softmax over its k*n routed keys, O its attention output, D = dout . O and
 * scale = (C/heads)^-1/2:
 *   dv[key] += P dout;  dS = P (dout . v[key] - D);
 *   dq += scale dS k[key];  dk[key] += scale dS q;
 *   dv += the LePE's transpose applied to dout;
 *   dlepe_w[c][u][s] = sum_{b,y,x} dout[y][x][c] v[y+u-ks/2][x+s-ks/2][c];
 *   dlepe_b[c] = sum_{b,y,x} dout[y][x][c].
 *   q, k, v, dout  [B, H, W, C] device, dtype; idx, heads, S, topk, lepe_w,
 *                  lepe_ks as bra_attend (the forward's bias does not enter)
 *   dq, dk, dv     out: float32 [B, H, W, C] device, overwritten
 *   dlepe_w        out: float32 [C, lepe_ks, lepe_ks] device, overwritten
 *   dlepe_b        out (optional, may be NULL): float32 [C] device
 * Arithmetic is float32; dk, dv and the LePE gradients are summed with
 * atomic adds, so their last bits may differ from run to run. An index out
 * of range reads zero keys (as bra_attend does), sends them no gradient and
 * sets the device status word. Supported: C / heads <= 64 and a
 * per-block shared-memory footprint of about 4 (2 n + 2 topk n)(C / heads + 1)
 * + 8 n (topk n + 1) bytes within the limit (n = tokens per region);
 * otherwise BRA_ERR_UNSUPPORTED. Outputs must not overlap the inputs or one
 * another.
 */
int bra_attend_backward(const void *q, const void *k, const void *v, const int32_t *idx,
                        int B, int H, int W, int C, int heads, int S, int topk,
                        const float *lepe_w, int lepe_ks, const void *dout, int dtype,
                        float *dq, float *dk, float *dv, float *dlepe_w, float *dlepe_b,
                        void *stream);

/* Bytes of the workspace bra_block_ffn needs; 0 on invalid sizes. */
size_t bra_block_ffn_workspace_bytes(int B, int H, int W, int C);

/*
 * bra_block_ffn -- the ConvFFN branch of the BiFormer block (page
 * "BiFormer架构核心思想解析" §3.1 "x = x + self.ffn(self.norm2(x))"):
 *   y = x + fc2(GELU(dwconv3x3(fc1(norm2(x)))))
 * with fc1 [3C][C] (w1, b1), the convolution [3C, 3, 3] (conv_w, conv_b) and
 * fc2 [C][3C] (w2, b2). The pages name a two-layer MLP of ratio 3 with a 3 x 3
 * depthwise convolution; this library reads the convolution as sitting in
 * the hidden layer before the activation, and the activation as nn.GELU.
 * It enqueues bra_layer_norm, bra_linear, bra_dwconv_gelu and bra_linear
 * (with x as the residual).
 *   x, y      [B, H, W, C] device bf16 (disjoint)
 *   workspace device buffer of bra_block_ffn_workspace_bytes(...) bytes
 * Supported: bf16 and the shapes of its steps (C = 64 or 128); errors as
 * those steps'.
 */
int bra_block_ffn(const void *x, const float *ln_w, const float *ln_b, float eps, const void *w1,
                  const float *b1, const float *conv_w, const float *conv_b, const void *w2,
                  const float *b2, int B, int H, int W, int C, int dtype, void *workspace,
                  void *y, void *stream);

/* Bytes of the workspace bra_block_attention needs; 0 on invalid sizes. */
size_t bra_block_attention_workspace_bytes(int B, int H, int W, int C, int S, int topk);

/*
 * bra_block_attention -- the attention branch of the BiFormer block (page
 * "BiFormer架构核心思想解析" §3.1): y = x + bra(norm1(x)), where bra is the
 * Q/K/V projections of the cybasar page §3 followed by bra_forward (routing,
 * routed attention and LePE; the pages give BRA no output projection). It
 * enqueues bra_layer_norm, bra_qkv_project, bra_forward and
 * bra_residual_add on the stream.
 *   x         [B, H, W, C] device bf16, the block input
 *   ln_w, ln_b  LayerNorm scale and shift, [C] float32 (or NULL), eps as in
 *             bra_layer_norm
 *   w_qkv, b_qkv  as w and bias of bra_qkv_project
 *   lepe_*    as in bra_attend
 *   workspace device buffer of bra_block_attention_workspace_bytes(...) bytes
 *             (16-byte aligned): the normalised tokens, q, k, v and the
 *             routing index
 *   y         out: [B, H, W, C] device bf16, disjoint from x and workspace
 * Supported: bf16 and the shapes of its four steps; errors as those steps'.
 */
int bra_block_attention(const void *x, const float *ln_w, const float *ln_b, float eps,
                        const void *w_qkv, const float *b_qkv, int B, int H, int W, int C,
                        int heads, int S, int topk, const float *lepe_w, const float *lepe_b,
                        int lepe_ks, int dtype, void *workspace, void *y, void *stream);

/*
 * bra_forward_launches -- how many kernels bra_forward (and
 * bra_forward_static) enqueue for this problem on the current device: 1 or 2,
 * 0 for B == 0, or minus a status code for invalid sizes. Nothing is
 * enqueued (it may query the device's occupancy once).
 */
int bra_forward_launches(int B, int H, int W, int C, int heads, int S, int topk, int lepe_ks,
                         int dtype);

/* Bytes of the routing index [B, S*S, topk] int32; 0 on invalid sizes. */
size_t bra_idx_workspace_bytes(int B, int S, int topk);

/*
 * bra_device_status -- synchronise `stream`, then read the device status word
 * that kernels set on the current device. Returns BRA_OK, BRA_ERR_TIMEOUT (a
 * bounded wait gave up), BRA_ERR_INVALID_ARG (a routing index was out of
 * range) or BRA_ERR_CUDA (the synchronisation itself failed). With clear != 0
 * the word is reset to zero afterwards.
 */
int bra_device_status(void *stream, int clear);

/* Static text for a status code. */
const char *bra_status_string(int status);

/* Version of this ABI (major * 100 + minor). */
int bra_abi_version(void);

/*
 * bra_check_wait_timeout -- exercises the device-side failure path without a
 * fault: enqueues one small kernel whose bounded mbarrier wait can never
 * complete (it expects bytes that no copy delivers). The wait gives up after
 * limit_ns nanoseconds of the GPU's global timer, sets the timeout bit of the
 * device status word and the kernel returns; bra_device_status then reports
 * BRA_ERR_TIMEOUT (clear the word before further work: after a timeout,
 * later waits that do not succeed at once return without waiting).
 *   limit_ns  1000 .. 1e9, otherwise BRA_ERR_INVALID_ARG and nothing is
 *             enqueued.
 * No page describes it; it tests this library's own error reporting.
 */
int bra_check_wait_timeout(uint64_t limit_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* BRA_H_ */

/*
 * dpp.h -- C ABI of the displaced-patch-parallelism hot path (libdpp.so).
 *
 * Displaced patch parallelism ("DistriFusion: Distributed Parallel Inference
 * for High-Resolution Diffusion Models", reader's notes, Introduction
 * para. 4 and Related Work / Parallelism): an image latent is cut into P
 * horizontal bands ("patches"), one per device.  At a displaced denoising
 * step each band computes its own rows from fresh activations and takes the
 * other bands' activations from the previous step (the stale buffer), so
 * the exchange between devices can overlap compute.  The first step is
 * synchronous (stale == fresh).  The layer wrappers are a 3x3 convolution
 * (DistriConv2dPP), GroupNorm (DistriGroupNorm) and self/cross attention
 * (DistriSelfAttentionPP, DistriCrossAttentionPP); the exchange is an
 * all_gather of each band's rows concatenated along the height axis
 * ("DistriFusion开发者必读：分布式UNet架构设计与模块拆分实现详解", sections
 * 卷积层拆分, 归一化层拆分, 注意力机制拆分, 分布式通信与同步机制).
 *
 * This library runs all P bands on ONE GPU: band p is a "virtual device"
 * inside each batched launch, and the all_gather becomes an in-HBM refresh
 * of the stale buffer, normally written by the producing kernel itself.
 * Every displaced op computes, for band p, the ordinary full-image layer
 * applied to the composite image Z_p (fresh rows R_p = [p*H/P, (p+1)*H/P),
 * stale rows elsewhere), restricted to R_p.
 *
 * Conventions for every entry point:
 *   - Memory: all tensor pointers are DEVICE pointers owned by the caller,
 *     16-byte aligned, dense (no strides).  The library never allocates
 *     device memory and keeps no state between calls except the per-device
 *     entries listed under Devices below, a launch counter and the
 *     optional profiling events of dpp_set_attn_core_events().  TMA tensor
 *     maps are encoded on the host at every call, so nothing is keyed by a
 *     pointer that the caller may free.  Workspace, where needed, is passed
 *     in by the caller; its size comes from the matching *_workspace_bytes()
 *     query.
 *   - Layout: activations NHWC [B, H, W, C] (torch channels_last); attention
 *     tokens [B, N, C] with N = H*W and token n = h*W + w, so band p owns
 *     the contiguous tokens [p*N/P, (p+1)*N/P).  Channel c of an attention
 *     layer belongs to head c / head_dim.
 *   - Types: DPP_BF16 = bf16 storage, fp32 accumulation and softmax;
 *     DPP_F32 = fp32 storage and arithmetic (SIMT path, no TF32).
 *     Biases, GroupNorm affine and statistics are always fp32.  Attention
 *     layers of type DPP_BF16 keep their K/V state (and their internal Q
 *     and O) in fp16: same tensor-core rate as bf16 with an 11-bit
 *     significand, which keeps the layer's chained roundings inside the
 *     bf16 error bound; bf16 intermediates alone exceed it.
 *   - Streams: every call is asynchronous on `stream` (a cudaStream_t;
 *     NULL = legacy default stream).
 *   - Errors: argument checks run on the host before anything is launched
 *     and return a dpp_status with no side effect.  A failed launch returns
 *     DPP_ERR_CUDA.  Kernels that wait on barriers give up after a bounded
 *     time and record DPP_ERR_TIMEOUT in a device status word read by
 *     dpp_device_status(); an attention layer of type DPP_BF16 whose Q, K
 *     or V leaves the fp16 range records DPP_ERR_RANGE there.
 *   - Devices: the library keeps, per device, the address of its device
 *     status word and of the static GroupNorm scratch, the shared-memory
 *     limits it has set on its kernels and the GroupNorm launch's occupancy.  These belong to the device's
 *     primary context: do not use the library across cudaDeviceReset
 *     (reload the library in a new process instead).
 *   - Synchronous step: passing NULL as the stale input (stale_prev,
 *     stats_prev, kv_prev) means "all bands are fresh" -- the synchronous
 *     first step, which is exactly the unpartitioned full-image layer.
 *   - Stale inputs and the *_next outputs that refresh them must not
 *     overlap (DPP_ERR_ALIAS): band q's refresh would otherwise overwrite
 *     data band p still reads in the same launch.
 */
#ifndef DPP_H_
#define DPP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *dpp_stream;

typedef enum {
  DPP_OK = 0,
  DPP_ERR_INVALID_ARG = 1, /* null pointer, bad size, H % P != 0, ... */
  DPP_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. head_dim != 64) */
  DPP_ERR_ALIAS = 3,       /* a stale input overlaps the buffer refreshing it */
  DPP_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required */
  DPP_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed */
  DPP_ERR_TIMEOUT = 6,     /* a bounded device-side wait gave up */
  DPP_ERR_ALIGN = 7,       /* a pointer is not 16-byte aligned */
  DPP_ERR_RANGE = 8        /* a value exceeded the fp16 range of an attention state
                              (|Q|, |K| or |V| > 65504 in a bf16 layer); reported
                              through the device status word */
} dpp_status;

typedef enum { DPP_F32 = 0, DPP_BF16 = 1 } dpp_dtype;

/* Where a band's conv reads the input rows just outside the band (its halo):
 *   DPP_HALO_STALE  displaced patch parallelism: from stale_prev (the
 *                   previous step), or fresh for the synchronous step;
 *   DPP_HALO_FRESH  the conv_in flag of the conv wrapper (is_first_layer):
 *                   the input latent is identical on every device, so the
 *                   halo is fresh and stale_prev is ignored;
 *   DPP_HALO_ZERO   naive patch parallelism (every band an image of its own,
 *                   zero-padded at its edges: the seam baseline of the
 *                   DistriFusion notes, Introduction para. 3). */
typedef enum { DPP_HALO_STALE = 0, DPP_HALO_FRESH = 1, DPP_HALO_ZERO = 2 } dpp_halo;

/* 3x3 conv, stride 1, zero padding 1, C_in -> C_out; halo: a dpp_halo.
 * accumulate != 0: y += the conv's result (y is read first: the residual
 * addition of a ResNet block, done in place on the residual). */
typedef struct {
  int B, H, W, C_in, C_out, P;
  dpp_dtype dtype;
  int halo;
  int accumulate;
} dpp_conv_desc;

/* Activation applied after a GroupNorm's affine. */
typedef enum { DPP_ACT_NONE = 0, DPP_ACT_SILU = 1 } dpp_act;

/* GroupNorm over [B, H, W, C] with G groups of C/G consecutive channels.
 * band_local != 0: naive patch parallelism -- each band's statistics over
 * its own rows only (stats_prev is ignored).
 * act: a dpp_act applied to the output (DPP_ACT_SILU: y * sigmoid(y), the
 * GroupNorm -> SiLU of a ResNet block); the statistics are those of x. */
typedef struct {
  int B, H, W, C, G, P;
  float eps;
  dpp_dtype dtype;
  int band_local;
  int act;
} dpp_gn_desc;

/* Attention over an H x W token grid (N = H*W), C = heads * head_dim.
 * n_ctx / c_ctx: text-context length and width (cross-attention only).
 * band_local != 0 (self-attention): naive patch parallelism -- a band's
 * queries attend over its own tokens only (kv_prev is ignored).
 * accumulate != 0: y += the attention's output (y is read first: the
 * residual addition of a transformer block, in place on the residual). */
typedef struct {
  int B, H, W, C, heads, head_dim, P;
  int n_ctx, c_ctx;
  dpp_dtype dtype;
  int band_local;
  int accumulate;
} dpp_attn_desc;

/* LayerNorm over the C channels of each of T tokens. */
typedef struct {
  int T, C;
  float eps;
  dpp_dtype dtype;
} dpp_ln_desc;

/* y[M, N] = x[M, K] w^T + bias (torch Linear, w [N, K]).
 * epilogue DPP_EPI_GEGLU: w is [2N, K] and bias [2N]; with h = x w^T + bias,
 * y = h[:, :N] * GELU(h[:, N:]) (exact erf GELU: the gated feed-forward of a
 * transformer block).  accumulate != 0: y += the result (y read first). */
typedef enum { DPP_EPI_NONE = 0, DPP_EPI_GEGLU = 1 } dpp_epilogue;
typedef struct {
  int M, K, N;
  dpp_dtype dtype;
  int epilogue;
  int accumulate;
} dpp_linear_desc;

/* ---------------------------------------------------------------------------
 * dpp_conv3x3 -- DistriConv2dPP (section 卷积层拆分 of the DistriFusion
 * developer guide; displaced semantics from the reader's notes, Introduction
 * para. 4).
 *   y[b,h,w,o] = bias[o] + sum_{i,dy,dx} w[o,dy,dx,i] * Z_p[b,h+dy-1,w+dx-1,i]
 * for h in band p, Z_p = x on the band's rows and stale_prev elsewhere
 * (only the rows just above and below the band are read from stale_prev),
 * zero outside the image.
 *   x, stale_prev, y : [B, H, W, C_in/C_out] NHWC, desc->dtype.
 *                      stale_prev == NULL or == x: synchronous step.
 *   w                : [C_out, 3, 3, C_in] (torch [C_out, C_in, 3, 3] in
 *                      channels_last memory), desc->dtype.
 *   bias             : [C_out] fp32 or NULL.
 * Requires H % P == 0, C_in and C_out multiples of 8 (bf16) / 4 (f32),
 * halo one of the dpp_halo values.  With DPP_HALO_ZERO the rows outside
 * the band read as zero (naive patches); with DPP_HALO_FRESH as x.
 * y must not overlap x or stale_prev.
 * ------------------------------------------------------------------------- */
dpp_status dpp_conv3x3(const dpp_conv_desc *desc, const void *x, const void *stale_prev,
                       const void *w, const float *bias, void *y, dpp_stream stream);

/* ---------------------------------------------------------------------------
 * dpp_groupnorm -- DistriGroupNorm (section 归一化层拆分 of the DistriFusion
 * developer guide).  Per band p, batch b, group g:
 *   s1 = sum over band p of x  +  sum_{q != p} stats_prev[q,b,g,0]
 *   s2 = likewise for x^2,  n = H*W*C/G,  mean = s1/n,
 *   var = max(s2/n - mean^2, 0) (biased),
 *   y = (x - mean) / sqrt(var + eps) * gamma[c] + beta[c]   on band p's rows.
 * The band's fresh partials (sum x, sum x^2) are written to stats_next[p]
 * in the same call: that write is the refresh of the GroupNorm state.
 *   x, y        : [B, H, W, C] NHWC, desc->dtype; y may equal x (in place).
 *   stats_prev  : [P, B, G, 2] fp32, the previous step's stats_next, or NULL
 *                 for the synchronous step (statistics of x alone).
 *   stats_next  : [P, B, G, 2] fp32 output; must not overlap stats_prev.
 *   gamma, beta : [C] fp32, both NULL for no affine.
 *   ws          : dpp_groupnorm_workspace_bytes(desc) bytes of device memory,
 *                 any contents (the call clears the counters it holds).
 *                 Calls sharing a workspace must not overlap on the GPU.
 * The kernel is a cooperative launch (all its CTAs resident at once), so
 * it waits for the whole device when other work occupies it.
 * Requires H % P == 0, C % G == 0, C a multiple of 8 (bf16) / 4 (f32).
 * ------------------------------------------------------------------------- */
dpp_status dpp_groupnorm(const dpp_gn_desc *desc, const void *x, const float *stats_prev,
                         float *stats_next, const float *gamma, const float *beta, void *y,
                         void *ws, size_t ws_bytes, dpp_stream stream);
size_t dpp_groupnorm_workspace_bytes(const dpp_gn_desc *desc);

/* ---------------------------------------------------------------------------
 * dpp_groupnorm_static -- dpp_groupnorm without a workspace argument.  The
 * pages have no counterpart: this entry point exists for callers that cannot
 * allocate device memory -- plugins running inside a host program that owns
 * the whole device-memory budget (an inference server's pre-planned arena, a
 * framework layer API that hands out no workspace), or code that must not
 * call cudaMalloc on a hot path because it may synchronise the device.
 * Arguments and results are those of dpp_groupnorm; its scratch lives in a
 * static device array of DPP_GN_STATIC_SCRATCH_BYTES that every GPU loading
 * the library holds until the process exits.  It allocates nothing.
 *   - Returns DPP_ERR_WORKSPACE when dpp_groupnorm_workspace_bytes(desc)
 *     exceeds DPP_GN_STATIC_SCRATCH_BYTES (512 bytes per batch x band
 *     unit with G = 32 groups: about 2000 units).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls share the array and it keeps the last call's contents
 *     (each call clears the counters it needs before use): calls whose
 *     kernels overlap on the GPU (several streams or host threads) race on
 *     it.
 * ------------------------------------------------------------------------- */
#define DPP_GN_STATIC_SCRATCH_BYTES (1u << 20)
dpp_status dpp_groupnorm_static(const dpp_gn_desc *desc, const void *x,
                                const float *stats_prev, float *stats_next,
                                const float *gamma, const float *beta, void *y,
                                dpp_stream stream);

/* ---------------------------------------------------------------------------
 * dpp_conv3x3_gn + dpp_groupnorm_apply -- the conv followed by the displaced
 * GroupNorm of its output (the ResNet block's conv -> GroupNorm of the U-Net
 * the DistriFusion developer guide partitions, sections 卷积层拆分 and
 * 归一化层拆分), with the GroupNorm's fresh partial sums produced by the
 * conv's epilogue instead of a pass of their own.  Results equal
 * dpp_conv3x3 followed by dpp_groupnorm on the same inputs (up to the
 * order of floating-point additions).
 *
 * dpp_conv3x3_gn: dpp_conv3x3, and in the same call
 *   gn_sums[p,b,g] = (sum y, sum y^2) over band p of image b and the
 *                    C_out/G channels of group g, of y as stored.
 *   gn_sums : [P, B, G, 2] fp64 device memory, overwritten.
 *   Requires the bf16 tensor-core conv (DPP_ERR_UNSUPPORTED otherwise) and
 *   C_out % G == 0.
 *
 * dpp_groupnorm_apply: dpp_groupnorm given gn_sums of x; one pass over x.
 *   Band p's statistics are gn_sums[p] plus stats_prev[q] for q != p
 *   (NULL stats_prev: all bands' gn_sums -- the synchronous step);
 *   stats_next[p] = gn_sums[p] rounded to fp32 (the refresh of the state).
 *   Other arguments and rules as dpp_groupnorm; no workspace; G <= 1024.
 * ------------------------------------------------------------------------- */
dpp_status dpp_conv3x3_gn(const dpp_conv_desc *desc, const void *x, const void *stale_prev,
                          const void *w, const float *bias, void *y, int G, double *gn_sums,
                          dpp_stream stream);
dpp_status dpp_groupnorm_apply(const dpp_gn_desc *desc, const void *x, const float *stats_prev,
                               const double *gn_sums, float *stats_next, const float *gamma,
                               const float *beta, void *y, dpp_stream stream);

/* ---------------------------------------------------------------------------
 * dpp_groupnorm_sums + dpp_groupnorm_affine + dpp_conv3x3_norm -- the
 * ResNet block's GroupNorm -> SiLU -> conv (DistriFusion developer guide,
 * sections 归一化层拆分 and 卷积层拆分) with the normalised tensor never
 * stored: the GroupNorm is reduced to one scale and shift per band, image
 * and channel, and the conv applies them (and the SiLU) to its input as it
 * loads it.  Results equal dpp_groupnorm (act) followed by dpp_conv3x3 on
 * the normalised tensor, up to floating-point rounding, when the conv's
 * stale_prev is the previous step's un-normalised input and affine_prev
 * the previous step's affine (then the halo rows are normalised exactly as
 * the previous step's GroupNorm normalised them).
 *
 * dpp_groupnorm_sums: gn_sums[p,b,g] = (sum x, sum x^2) over band p of
 *   image b and the C/G channels of group g (what dpp_conv3x3_gn produces
 *   for its output), for an input no conv summed.  One read of x.
 *   gn_sums : [P, B, G, 2] fp64 device memory, overwritten.  G <= 1024 and
 *             C <= 4096 (bf16) / 2048 (fp32), else DPP_ERR_UNSUPPORTED.
 *   The sums are bit-reproducible (fixed reduction order).
 *
 * dpp_groupnorm_affine: per band p, image b, channel c in group g,
 *   affine[p,b,c] = (a, s),  a = gamma[c] / sqrt(var + eps),
 *                            s = beta[c] - mean * a,
 *   with mean and var of band p's statistics as dpp_groupnorm_apply forms
 *   them (gn_sums[p] plus stats_prev[q] for q != p; NULL stats_prev: every
 *   band's gn_sums, the synchronous step; band_local: band p's alone).
 *   stats_next[p] = gn_sums[p] in fp32 (the refresh of the GroupNorm
 *   state), or NULL to skip it.  desc->act is not used (the conv applies it).
 *   affine : [P, B, C, 2] fp32 (scale, shift interleaved), overwritten.
 *
 * dpp_conv3x3_norm: dpp_conv3x3 (+ dpp_conv3x3_gn's sums when gn_sums is
 *   not NULL) of the tensor Z' with
 *     Z'[b,h,w,c] = act(Z[b,h,w,c] * a[q,b,c] + s[q,b,c]),  q = h / (H/P),
 *   where (a, s) is affine for the rows of band p and for fresh halo rows,
 *   and affine_prev (the previous step's) for halo rows read from
 *   stale_prev; image padding and the zero halo (DPP_HALO_ZERO) stay zero.
 *   act: DPP_ACT_NONE or DPP_ACT_SILU (x * sigmoid(x), evaluated as
 *   h + h tanh(h), h = x/2, with a hardware tanh of about 2^-11 relative
 *   error, below the bf16 rounding of the normalised value).
 *   affine, affine_prev : [P, B, C_in, 2] fp32 from dpp_groupnorm_affine;
 *                         affine_prev may be NULL when no halo row is read
 *                         from stale_prev (stale_prev NULL or == x, or a
 *                         fresh or zero halo).
 *   Requires the bf16 tensor-core conv (DPP_ERR_UNSUPPORTED otherwise);
 *   other arguments and rules as dpp_conv3x3_gn.  Only the halo rows of
 *   stale_prev are read (see dpp_refresh_halo).
 * ------------------------------------------------------------------------- */
dpp_status dpp_groupnorm_sums(const dpp_gn_desc *desc, const void *x, double *gn_sums,
                              dpp_stream stream);
dpp_status dpp_groupnorm_affine(const dpp_gn_desc *desc, const double *gn_sums,
                                const float *stats_prev, float *stats_next, const float *gamma,
                                const float *beta, float *affine, dpp_stream stream);
dpp_status dpp_conv3x3_norm(const dpp_conv_desc *desc, const void *x, const void *stale_prev,
                            const float *affine, const float *affine_prev, int act,
                            const void *w, const float *bias, void *y, int G, double *gn_sums,
                            dpp_stream stream);

/* ---------------------------------------------------------------------------
 * dpp_self_attn -- DistriSelfAttentionPP (section 注意力机制拆分 of the
 * DistriFusion developer guide, attn1).  For band p:
 *   Q = x[band p] wq^T;  K/V rows of band p's tokens are x[band p] wk^T /
 *   x[band p] wv^T (fresh), all other rows come from kv_prev (stale);
 *   O = softmax(Q K^T / sqrt(head_dim)) V per head;  y[band p] = O wo^T.
 * The fresh K/V of every token are written to kv_next by the projection
 * kernel itself: that write is the refresh of the attention state.
 *   x, y     : [B, N, C] tokens, desc->dtype.
 *   wq..wo   : [C, C] torch Linear [out, in], desc->dtype, no bias.
 *   kv_prev  : [B, N, 2, C] (K then V per token) from the previous step,
 *              or NULL for the synchronous step.  fp16 for DPP_BF16
 *              layers, fp32 for DPP_F32 layers.
 *   kv_next  : [B, N, 2, C] output, same type; must not overlap kv_prev.
 *   ws       : dpp_self_attn_workspace_bytes(desc) bytes (Q and O).
 * Requires head_dim == 64, H % P == 0, C == heads * 64.
 * DPP_BF16 layers hold Q, K, V and O in fp16: if a projected value exceeds
 * 65504 the call still completes, and DPP_ERR_RANGE is recorded in the
 * device status word (dpp_device_status); the output is then not valid.
 * ------------------------------------------------------------------------- */
dpp_status dpp_self_attn(const dpp_attn_desc *desc, const void *x, const void *wq,
                         const void *wk, const void *wv, const void *wo,
                         const void *kv_prev, void *kv_next, void *y, void *ws,
                         size_t ws_bytes, dpp_stream stream);
size_t dpp_self_attn_workspace_bytes(const dpp_attn_desc *desc);

/* ---------------------------------------------------------------------------
 * dpp_cross_attn -- DistriCrossAttentionPP (attn2).  The text context is
 * replicated on every device, so no stale state enters:
 *   Q = x wq^T, K = ctx wk^T, V = ctx wv^T,
 *   y = softmax(Q K^T / sqrt(head_dim)) V wo^T.
 *   x, y   : [B, N, C];  ctx : [B, n_ctx, c_ctx];  desc->dtype.
 *   wq, wo : [C, C];  wk, wv : [C, c_ctx].
 *   ws     : dpp_cross_attn_workspace_bytes(desc) bytes.
 * Requires head_dim == 64, c_ctx a multiple of 8.
 * ------------------------------------------------------------------------- */
dpp_status dpp_cross_attn(const dpp_attn_desc *desc, const void *x, const void *ctx,
                          const void *wq, const void *wk, const void *wv, const void *wo,
                          void *y, void *ws, size_t ws_bytes, dpp_stream stream);
size_t dpp_cross_attn_workspace_bytes(const dpp_attn_desc *desc);

/* ---------------------------------------------------------------------------
 * dpp_cross_attn_kv + dpp_cross_attn_cached -- dpp_cross_attn in two parts,
 * so that the context's K and V are projected once per prompt (the text
 * context is the same at every denoising step) instead of once per call:
 *   dpp_cross_attn_kv:     kv_ctx[b, t, 0, :] = ctx[b, t] wk^T,
 *                          kv_ctx[b, t, 1, :] = ctx[b, t] wv^T.
 *   dpp_cross_attn_cached: y = softmax((x wq^T) K^T / sqrt(head_dim)) V wo^T
 *                          with K, V from kv_ctx.
 *   kv_ctx : [B, n_ctx, 2, C] (K then V per context token), fp16 for
 *            DPP_BF16 layers, fp32 for DPP_F32 layers; written by
 *            dpp_cross_attn_kv, read by dpp_cross_attn_cached.
 *   ws     : dpp_cross_attn_cached_workspace_bytes(desc) bytes (Q and O).
 * The pair computes exactly what dpp_cross_attn computes (same kernels in
 * the same order), which is itself the two calls back to back.
 * ------------------------------------------------------------------------- */
dpp_status dpp_cross_attn_kv(const dpp_attn_desc *desc, const void *ctx, const void *wk,
                             const void *wv, void *kv_ctx, dpp_stream stream);
dpp_status dpp_cross_attn_cached(const dpp_attn_desc *desc, const void *x, const void *kv_ctx,
                                 const void *wq, const void *wo, void *y, void *ws,
                                 size_t ws_bytes, dpp_stream stream);
size_t dpp_cross_attn_cached_workspace_bytes(const dpp_attn_desc *desc);

/* ---------------------------------------------------------------------------
 * dpp_cfg_combine -- classifier-free-guidance combine and the denoising
 * discrepancy of the Hydiff summaries (gist.science, "基于条件的数据划分"
 * and "自适应并行切换"; Avetisyan, "Адаптивное переключение"):
 *   out[i] = eps_u[i] + scale * (eps_c[i] - eps_u[i])
 *   sums3  = { sum|eps_c - eps_u|, sum|eps_u|, sum|eps_c| }   (fp64)
 * rel-MAE = sums3[0] / sums3[1].  The reduction order is fixed, so sums3 is
 * bit-reproducible for a given n.
 *   eps_u, eps_c, out : n fp32 (out may equal eps_u or eps_c).
 *   sums3             : 3 doubles of device memory, or NULL.
 *   ws                : dpp_cfg_workspace_bytes(n) bytes.  Its first 16
 *                       bytes are a completion counter that must be zero
 *                       before the first call (e.g. cudaMemset); every call
 *                       that completes leaves it zero again.  Calls that
 *                       share a workspace must not overlap on the GPU.
 * ------------------------------------------------------------------------- */
dpp_status dpp_cfg_combine(const float *eps_u, const float *eps_c, float scale, size_t n,
                           float *out, double *sums3, void *ws, size_t ws_bytes,
                           dpp_stream stream);
size_t dpp_cfg_workspace_bytes(size_t n);

/* ---------------------------------------------------------------------------
 * dpp_refresh_stale -- the all_gather of the gathered-buffer exchange
 * (section 分布式通信与同步机制 of the DistriFusion developer guide):
 * bands are concatenated along the height axis.  The tensor is viewed as
 * [outer][rows][row_bytes]; band p owns rows [p*rows/P, (p+1)*rows/P) of
 * every outer slice.  For every p whose bit is set in patch_mask the band is
 * copied bit-exactly from fresh to stale; other bands are left untouched.
 *   NHWC activations : outer = B, rows = H, row_bytes = W*C*elem
 *   K/V state        : outer = B, rows = N, row_bytes = 2*C*elem
 *   GroupNorm stats  : outer = 1, rows = P, row_bytes = B*G*2*4
 * Requires rows % P == 0, 1 <= P <= 64, row_bytes % 16 == 0; fresh and
 * stale must not overlap.
 * ------------------------------------------------------------------------- */
dpp_status dpp_refresh_stale(const void *fresh, void *stale, size_t outer, size_t rows,
                             size_t row_bytes, int P, uint64_t patch_mask, dpp_stream stream);

/* ---------------------------------------------------------------------------
 * dpp_refresh_halo -- the part of the all_gather (same section) that a
 * displaced 3x3 conv reads: at every band boundary the last row of the band
 * above and the first row of the band below, copied bit-exactly from fresh
 * to stale; every other row of stale is left untouched.  For a conv input
 * that is overwritten later in the step (the residual stream), this keeps
 * the rows the next step reads as halo at 2 (P - 1) rows per outer slice.
 *   View and requirements as dpp_refresh_stale (outer = B, rows = H,
 *   row_bytes = W*C*elem for NHWC); P = 1 copies nothing;
 *   outer * 2 * (P - 1) <= 65535.
 * ------------------------------------------------------------------------- */
dpp_status dpp_refresh_halo(const void *fresh, void *stale, size_t outer, size_t rows,
                            size_t row_bytes, int P, dpp_stream stream);

/* ---------------------------------------------------------------------------
 * Per-token layers of the U-Net's transformer blocks.  The DistriFusion
 * developer guide (sections 卷积层拆分, 注意力机制拆分, 归一化层拆分) replaces
 * only the convolutions, the attention layers and the GroupNorms; the layers
 * below act on one token at a time, so a band computes them on its own rows
 * with no stale state.
 *
 * dpp_layernorm: y[t, c] = (x[t, c] - mean_t) / sqrt(var_t + eps) * gamma[c]
 *   + beta[c], mean and biased variance over the C channels of token t.
 *   x, y : [T, C] desc->dtype (bf16 or fp32); y may equal x.
 *   gamma, beta : [C] fp32, both NULL for no affine.
 *   Requires C a multiple of 8 (bf16) / 4 (fp32), C <= 8192.
 *
 * dpp_linear: see dpp_linear_desc.  x [M, K], y [M, N] bf16; w [N, K] (or
 *   [2N, K] for DPP_EPI_GEGLU) bf16; bias fp32 or NULL.  Tensor cores;
 *   requires DPP_BF16, K a multiple of 8, N a multiple of 64 (of 128 with
 *   DPP_EPI_GEGLU); y must not overlap x or w.  DPP_ERR_UNSUPPORTED for
 *   other types.
 * ------------------------------------------------------------------------- */
dpp_status dpp_layernorm(const dpp_ln_desc *desc, const void *x, const float *gamma,
                         const float *beta, void *y, dpp_stream stream);
dpp_status dpp_linear(const dpp_linear_desc *desc, const void *x, const void *w,
                      const float *bias, void *y, dpp_stream stream);

/* ---------------------------------------------------------------------------
 * dpp_wait_selftest -- exercises one of the library's bounded device waits
 * against an event that never comes, so that failure detection can be
 * tested without a fault: the kernel waits its limit (1 s), records
 * DPP_ERR_TIMEOUT in the status word (read it with dpp_device_status) and
 * returns; the context stays usable.
 *   kind 0: the acquire-poll wait on a unit counter (the cooperative
 *           GroupNorm's); scratch = 16 bytes of device memory holding zeros,
 *           which nothing advances.
 *   kind 1: the mbarrier wait of the tensor-core kernels; scratch unused.
 * Returns DPP_OK once the kernel is launched; it runs for about a second.
 * ------------------------------------------------------------------------- */
dpp_status dpp_wait_selftest(int kind, void *scratch, dpp_stream stream);

/* ---------------------------------------------------------------------------
 * dpp_workspace_bytes -- the workspace any entry point needs, by op: the
 * per-op queries above behind one call.  desc points to the op's descriptor
 * (dpp_gn_desc for DPP_OP_GROUPNORM, dpp_attn_desc for the attention ops,
 * a size_t element count for DPP_OP_CFG_COMBINE).  Ops that need no
 * workspace (conv, refresh, LayerNorm, linear, the one-pass GroupNorm)
 * return 0; an invalid descriptor or op returns 0 as well.
 * ------------------------------------------------------------------------- */
typedef enum {
  DPP_OP_CONV3X3 = 0,
  DPP_OP_GROUPNORM = 1,
  DPP_OP_SELF_ATTN = 2,
  DPP_OP_CROSS_ATTN = 3,
  DPP_OP_CFG_COMBINE = 4,
  DPP_OP_REFRESH_STALE = 5
} dpp_op;
size_t dpp_workspace_bytes(int op, const void *desc);

/* ---------------------------------------------------------------------------
 * Adaptive parallelism switching (the Hydiff summaries: gist.science,
 * section 自适应并行切换; Avetisyan, "Адаптивное переключение").  Host-side
 * state machine over the per-step denoising discrepancy d (rel-MAE of the
 * conditional vs the unconditional noise estimate: sums3[0] / sums3[1] of
 * dpp_cfg_combine).  Three stages: warm-up (serial) until tau1, where the
 * decline of d flattens; parallel until tau2, where d starts rising; fully
 * connecting (serial) to the end.  The pages fix no thresholds:
 *   tau1: for `patience` consecutive steps the relative drop
 *         (d_prev - d) / d_prev is below flat_tol (a rise counts as flat);
 *   tau2: for `patience` consecutive steps d exceeds the lowest d of the
 *         parallel stage by more than the fraction rise_tol.
 * dpp_switch_update feeds one step's d and returns the stage the next step
 * runs in; NaN or negative d changes nothing.  Host only: no GPU work, no
 * allocation, no global state.
 * ------------------------------------------------------------------------- */
enum { DPP_STAGE_WARMUP = 0, DPP_STAGE_PARALLEL = 1, DPP_STAGE_FULLY_CONNECTING = 2 };
typedef struct {
  double flat_tol, rise_tol;
  int patience;
  int stage;   /* DPP_STAGE_* */
  int run;     /* consecutive steps the current stage's exit condition has held */
  int steps;   /* steps observed */
  double prev; /* last d */
  double min_d; /* lowest d in the parallel stage */
} dpp_switch_state;
void dpp_switch_init(dpp_switch_state *state, double flat_tol, double rise_tol, int patience);
int dpp_switch_update(dpp_switch_state *state, double d);

/* Reads and clears the device status word written by bounded waits
 * (DPP_ERR_TIMEOUT) and by the fp16 range check of bf16 attention layers
 * (DPP_ERR_RANGE); DPP_OK when neither happened since the last read.
 * Synchronises `stream`. */
dpp_status dpp_device_status(dpp_stream stream);

/* SHA-256 (hex) of the sources and compiler flags this library was built
 * from; the build rebuilds a library whose hash differs from its sources. */
const char *dpp_source_hash(void);

/* Number of kernels this library has launched in this process (monotonic).
 * Calls rejected by argument checks launch nothing and leave it unchanged. */
uint64_t dpp_launch_count(void);

/* Profiling hook.  When start and stop are both non-NULL (cudaEvent_t
 * values), every later dpp_self_attn / dpp_cross_attn call records `start`
 * on its stream immediately before launching its attention-core kernel and
 * `stop` immediately after; pass NULL, NULL to turn it off.  Process-global
 * and not thread-safe: meant for a benchmark timing that one kernel live. */
void dpp_set_attn_core_events(void *start, void *stop);

/* Human-readable name of a status code (static storage). */
const char *dpp_status_string(dpp_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int dpp_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DPP_H_ */

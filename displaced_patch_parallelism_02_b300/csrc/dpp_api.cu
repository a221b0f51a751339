// C-ABI entry points of libdpp.so (declared in include/dpp.h).
//
// Every entry point validates its arguments on the host -- before any CUDA
// call -- and returns a dpp_status without launching anything when they are
// wrong.  The library allocates no device memory: workspaces come from the
// caller, sized by the *_workspace_bytes() queries.
#include <atomic>
#include <cstdio>
#include <cstring>

#include "dpp_internal.h"

namespace dpp {

__device__ int g_device_status;

int *device_status_ptr() {
  static int *cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cache[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    cache[dev] = reinterpret_cast<int *>(p);
  }
  return cache[dev];
}

}  // namespace dpp

using namespace dpp;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

size_t elem_size(dpp_dtype t) { return t == DPP_BF16 ? 2 : 4; }

bool dtype_ok(dpp_dtype t) { return t == DPP_F32 || t == DPP_BF16; }

// channel granularity of the 16-byte vector paths
int chan_quantum(dpp_dtype t) { return t == DPP_BF16 ? 8 : 4; }

dpp_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DPP_OK : DPP_ERR_CUDA; }

constexpr long long kMaxElems = (1ll << 31) - 1;

dpp_status check_conv(const dpp_conv_desc *d, const void *x, const void *stale, const void *w,
                      const float *bias, const void *y) {
  if (!d || !x || !w || !y) return DPP_ERR_INVALID_ARG;
  if (!dtype_ok(d->dtype)) return DPP_ERR_INVALID_ARG;
  if (d->B < 1 || d->H < 1 || d->W < 1 || d->C_in < 1 || d->C_out < 1 || d->P < 1)
    return DPP_ERR_INVALID_ARG;
  if (d->H % d->P != 0) return DPP_ERR_INVALID_ARG;
  if (d->halo < DPP_HALO_STALE || d->halo > DPP_HALO_ZERO) return DPP_ERR_INVALID_ARG;
  const int q = chan_quantum(d->dtype);
  if (d->C_in % q || d->C_out % q) return DPP_ERR_INVALID_ARG;
  const long long pix = (long long)d->B * d->H * d->W;
  if (pix * d->C_in > kMaxElems || pix * d->C_out > kMaxElems) return DPP_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (stale && !aligned16(stale)) ||
      (bias && !aligned16(bias)))
    return DPP_ERR_ALIGN;
  const size_t es = elem_size(d->dtype);
  const size_t nx = (size_t)pix * d->C_in * es, ny = (size_t)pix * d->C_out * es;
  if (overlap(y, ny, x, nx) || overlap(y, ny, stale, nx) ||
      overlap(y, ny, w, (size_t)d->C_out * 9 * d->C_in * es))
    return DPP_ERR_ALIAS;
  return DPP_OK;
}

dpp_status check_gn(const dpp_gn_desc *d) {
  if (!d || !dtype_ok(d->dtype)) return DPP_ERR_INVALID_ARG;
  if (d->B < 1 || d->H < 1 || d->W < 1 || d->C < 1 || d->G < 1 || d->P < 1)
    return DPP_ERR_INVALID_ARG;
  if (d->H % d->P != 0 || d->C % d->G != 0) return DPP_ERR_INVALID_ARG;
  if (!(d->eps >= 0.f)) return DPP_ERR_INVALID_ARG;
  const int q = chan_quantum(d->dtype);
  if (d->C % q) return DPP_ERR_INVALID_ARG;
  if (d->C / q > 1024) return DPP_ERR_UNSUPPORTED;
  if ((long long)d->B * d->H * d->W * d->C > kMaxElems) return DPP_ERR_UNSUPPORTED;
  return DPP_OK;
}

dpp_status check_attn(const dpp_attn_desc *d, bool cross) {
  if (!d || !dtype_ok(d->dtype)) return DPP_ERR_INVALID_ARG;
  if (d->B < 1 || d->H < 1 || d->W < 1 || d->C < 1 || d->heads < 1 || d->P < 1)
    return DPP_ERR_INVALID_ARG;
  if (d->head_dim != 64) return DPP_ERR_UNSUPPORTED;
  if (d->C != d->heads * d->head_dim) return DPP_ERR_INVALID_ARG;
  if (d->H % d->P != 0) return DPP_ERR_INVALID_ARG;
  if (cross) {
    if (d->n_ctx < 1 || d->c_ctx < 1) return DPP_ERR_INVALID_ARG;
    if (d->c_ctx % 8) return DPP_ERR_INVALID_ARG;
  }
  const long long N = (long long)d->H * d->W;
  if ((long long)d->B * N * 3 * d->C > kMaxElems) return DPP_ERR_UNSUPPORTED;
  return DPP_OK;
}

size_t attn_tokens(const dpp_attn_desc &d) { return (size_t)d.B * d.H * d.W; }

// Bytes of the context K/V [B, n_ctx, 2, C] in the attention state type.
size_t ctx_kv_bytes(const dpp_attn_desc &d) {
  return (size_t)d.B * d.n_ctx * 2 * d.C * elem_bytes(inter_elem(d.dtype));
}


std::atomic<uint64_t> g_launches{0};
cudaEvent_t g_core_start = nullptr, g_core_stop = nullptr;

// Counts the kernels of a launcher call that returned cudaSuccess.
cudaError_t counted(cudaError_t e, int kernels) {
  if (e == cudaSuccess) g_launches += (uint64_t)kernels;
  return e;
}

// Projection GEMM: the tcgen05 kernel when the shape and types allow it
// (16-bit operands), the SIMT kernel otherwise (fp32 layers).
cudaError_t gemm(const GemmArgs &g, cudaStream_t s) {
  if (gemm_tc_supported(g)) return counted(launch_gemm_tc(g, device_status_ptr(), s), 1);
  return counted(launch_gemm_simt(g, s), 1);
}

// Bytes of the fp16 copy of Wo a bf16 attention layer keeps in its workspace
// (the output projection's two operands must share one 16-bit type).
size_t wo16_bytes(const dpp_attn_desc &d) {
  return d.dtype == DPP_BF16 ? align_up((size_t)d.C * d.C * 2, 256) : 0;
}

// The first projection of a bf16 attention layer (QKV, or cross-attention's
// Q) also makes the fp16 copy of wo the output projection needs, as a side
// task of the GEMM's epilogue warps: one launch fewer per call.  Returns
// whether the copy was attached (the tensor-core GEMM runs this shape).
bool attach_wo16(GemmArgs &g, const dpp_attn_desc &d, const void *wo, void *wo16) {
  if (d.dtype != DPP_BF16) return false;
  g.cast_src = wo;
  g.cast_dst = wo16;
  g.cast_n = (size_t)d.C * d.C;
  if (gemm_tc_supported(g)) return true;
  g.cast_src = nullptr;
  g.cast_dst = nullptr;
  g.cast_n = 0;
  return false;
}

// Output projection y = O wo^T; for bf16 layers wo is cast to fp16 into
// `wo16` (unless the first projection already did) so both operands are fp16.
cudaError_t out_proj(const dpp_attn_desc &d, const void *o, const void *wo, void *wo16, void *y,
                     int M, cudaStream_t s, bool wo16_ready) {
  const Elem te = inter_elem(d.dtype), tl = layer_elem(d.dtype);
  const int C = d.C;
  const void *w = wo;
  Elem tw = tl;
  if (d.dtype == DPP_BF16) {
    if (!wo16_ready) {
      cudaError_t e = counted(launch_cast_bf16_f16(wo, wo16, (size_t)C * C, s), 1);
      if (e != cudaSuccess) return e;
    }
    w = wo16;
    tw = E_F16;
  }
  GemmArgs op{o, {w, nullptr, nullptr}, C, M, C, C, y, C, C, nullptr, 0, te, tw, tl};
  op.accumulate = d.accumulate ? 1 : 0;  // y += O wo^T: the block's residual addition
  return gemm(op, s);
}

// Launches the attention core, bracketed by the profiling events when set.
cudaError_t attn_core(const AttnArgs &a, cudaStream_t s) {
  if (g_core_start && g_core_stop) cudaEventRecord(g_core_start, s);
  cudaError_t e = xattn_tc_supported(a)  ? counted(launch_xattn_tc(a, device_status_ptr(), s), 1)
                  : attn_tc_supported(a) ? counted(launch_attn_tc(a, device_status_ptr(), s), 1)
                                         : counted(launch_attn_simt(a, s), 1);
  if (g_core_start && g_core_stop) cudaEventRecord(g_core_stop, s);
  return e;
}

}  // namespace

extern "C" {

const char *dpp_status_string(dpp_status s) {
  switch (s) {
    case DPP_OK: return "DPP_OK";
    case DPP_ERR_INVALID_ARG: return "DPP_ERR_INVALID_ARG";
    case DPP_ERR_UNSUPPORTED: return "DPP_ERR_UNSUPPORTED";
    case DPP_ERR_ALIAS: return "DPP_ERR_ALIAS";
    case DPP_ERR_WORKSPACE: return "DPP_ERR_WORKSPACE";
    case DPP_ERR_CUDA: return "DPP_ERR_CUDA";
    case DPP_ERR_TIMEOUT: return "DPP_ERR_TIMEOUT";
    case DPP_ERR_ALIGN: return "DPP_ERR_ALIGN";
    case DPP_ERR_RANGE: return "DPP_ERR_RANGE";
  }
  return "DPP_ERR_UNKNOWN";
}

int dpp_version(void) { return 100; }

#ifndef DPP_SOURCE_SHA256
#define DPP_SOURCE_SHA256 "unknown"
#endif
const char *dpp_source_hash(void) { return DPP_SOURCE_SHA256; }

uint64_t dpp_launch_count(void) { return g_launches.load(); }

void dpp_set_attn_core_events(void *start, void *stop) {
  g_core_start = (cudaEvent_t)start;
  g_core_stop = (cudaEvent_t)stop;
}

dpp_status dpp_device_status(dpp_stream stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DPP_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return DPP_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return DPP_ERR_CUDA;
  return (dpp_status)v;
}

// ------------------------------------------------------------------ refresh
dpp_status dpp_refresh_stale(const void *fresh, void *stale, size_t outer, size_t rows,
                             size_t row_bytes, int P, uint64_t patch_mask, dpp_stream stream) {
  if (!fresh || !stale) return DPP_ERR_INVALID_ARG;
  if (P < 1 || P > 64 || rows == 0 || outer == 0 || rows % (size_t)P) return DPP_ERR_INVALID_ARG;
  if (row_bytes == 0 || row_bytes % 16) return DPP_ERR_INVALID_ARG;
  if (!aligned16(fresh) || !aligned16(stale)) return DPP_ERR_ALIGN;
  const size_t total = outer * rows * row_bytes;
  if (total / outer / rows != row_bytes) return DPP_ERR_INVALID_ARG;  // overflow
  if (overlap(fresh, total, stale, total)) return DPP_ERR_ALIAS;
  if (P < 64) patch_mask &= (1ull << P) - 1;
  if (patch_mask == 0) return DPP_OK;
  return from_cuda(counted(launch_refresh(fresh, stale, outer, rows, row_bytes, P, patch_mask,
                                          (cudaStream_t)stream), 1));
}

dpp_status dpp_refresh_halo(const void *fresh, void *stale, size_t outer, size_t rows,
                            size_t row_bytes, int P, dpp_stream stream) {
  if (!fresh || !stale) return DPP_ERR_INVALID_ARG;
  if (P < 1 || rows == 0 || outer == 0 || rows % (size_t)P) return DPP_ERR_INVALID_ARG;
  if (row_bytes == 0 || row_bytes % 16) return DPP_ERR_INVALID_ARG;
  if (!aligned16(fresh) || !aligned16(stale)) return DPP_ERR_ALIGN;
  const size_t total = outer * rows * row_bytes;
  if (total / outer / rows != row_bytes) return DPP_ERR_INVALID_ARG;  // overflow
  if (overlap(fresh, total, stale, total)) return DPP_ERR_ALIAS;
  if (P == 1) return DPP_OK;  // one band: no halo
  if (outer * 2 * (size_t)(P - 1) > 65535) return DPP_ERR_UNSUPPORTED;
  return from_cuda(counted(
      launch_refresh_halo(fresh, stale, outer, rows, row_bytes, P, (cudaStream_t)stream), 1));
}

// ---------------------------------------------------------------------- CFG
size_t dpp_cfg_workspace_bytes(size_t n) { return 16 + cfg_blocks(n) * 3 * sizeof(double); }

dpp_status dpp_cfg_combine(const float *eps_u, const float *eps_c, float scale, size_t n,
                           float *out, double *sums3, void *ws, size_t ws_bytes,
                           dpp_stream stream) {
  if (n > 0 && (!eps_u || !eps_c || !out)) return DPP_ERR_INVALID_ARG;
  if (n > ((size_t)1 << 40)) return DPP_ERR_UNSUPPORTED;
  if (!aligned16(eps_u) || !aligned16(eps_c) || !aligned16(out) ||
      (sums3 && ((uintptr_t)sums3 & 7u)))
    return DPP_ERR_ALIGN;
  const size_t nb = n * sizeof(float);
  if ((out != eps_u && overlap(out, nb, eps_u, nb)) || (out != eps_c && overlap(out, nb, eps_c, nb)))
    return DPP_ERR_ALIAS;
  if (sums3) {
    if (!ws || ws_bytes < dpp_cfg_workspace_bytes(n)) return DPP_ERR_WORKSPACE;
    if (!aligned16(ws)) return DPP_ERR_ALIGN;
    if (overlap(ws, ws_bytes, sums3, 3 * sizeof(double))) return DPP_ERR_ALIAS;
  }
  return from_cuda(
      counted(launch_cfg(eps_u, eps_c, scale, n, out, sums3, ws, (cudaStream_t)stream), 1));
}

// ---------------------------------------------------------------- groupnorm
size_t dpp_groupnorm_workspace_bytes(const dpp_gn_desc *d) {
  if (check_gn(d) != DPP_OK) return 0;
  return gn_workspace(*d);
}

dpp_status dpp_groupnorm(const dpp_gn_desc *d, const void *x, const float *stats_prev,
                         float *stats_next, const float *gamma, const float *beta, void *y,
                         void *ws, size_t ws_bytes, dpp_stream stream) {
  dpp_status st = check_gn(d);
  if (st != DPP_OK) return st;
  if (!x || !y || !stats_next) return DPP_ERR_INVALID_ARG;
  if ((gamma == nullptr) != (beta == nullptr)) return DPP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(stats_next) ||
      (stats_prev && !aligned16(stats_prev)))
    return DPP_ERR_ALIGN;
  const size_t need = gn_workspace(*d);
  if (!ws || ws_bytes < need) return DPP_ERR_WORKSPACE;
  if (!aligned16(ws)) return DPP_ERR_ALIGN;
  const size_t nx = (size_t)d->B * d->H * d->W * d->C * elem_size(d->dtype);
  const size_t ns = (size_t)d->P * d->B * d->G * 2 * sizeof(float);
  if (y != x && overlap(y, nx, x, nx)) return DPP_ERR_ALIAS;
  if (overlap(stats_prev, ns, stats_next, ns)) return DPP_ERR_ALIAS;
  if (overlap(ws, need, x, nx) || overlap(ws, need, y, nx) || overlap(ws, need, stats_next, ns) ||
      overlap(stats_next, ns, y, nx))
    return DPP_ERR_ALIAS;
  return from_cuda(counted(launch_groupnorm(*d, x, stats_prev, stats_next, gamma, beta, y, ws,
                                            (cudaStream_t)stream), 2));
}

dpp_status dpp_groupnorm_static(const dpp_gn_desc *d, const void *x, const float *stats_prev,
                                float *stats_next, const float *gamma, const float *beta,
                                void *y, dpp_stream stream) {
  dpp_status st = check_gn(d);
  if (st != DPP_OK) return st;
  if (!x || !y || !stats_next) return DPP_ERR_INVALID_ARG;
  if ((gamma == nullptr) != (beta == nullptr)) return DPP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(stats_next) ||
      (stats_prev && !aligned16(stats_prev)))
    return DPP_ERR_ALIGN;
  if (gn_workspace(*d) > kGnStaticScratchBytes) return DPP_ERR_WORKSPACE;
  const size_t nx = (size_t)d->B * d->H * d->W * d->C * elem_size(d->dtype);
  const size_t ns = (size_t)d->P * d->B * d->G * 2 * sizeof(float);
  if (y != x && overlap(y, nx, x, nx)) return DPP_ERR_ALIAS;
  if (overlap(stats_prev, ns, stats_next, ns) || overlap(stats_next, ns, y, nx))
    return DPP_ERR_ALIAS;
  return from_cuda(counted(launch_groupnorm_static(*d, x, stats_prev, stats_next, gamma, beta,
                                                   y, (cudaStream_t)stream), 2));
}

// --------------------------------------------------------------------- conv
dpp_status dpp_conv3x3(const dpp_conv_desc *d, const void *x, const void *stale_prev,
                       const void *w, const float *bias, void *y, dpp_stream stream) {
  dpp_status st = check_conv(d, x, stale_prev, w, bias, y);
  if (st != DPP_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (conv_tc_supported(*d))  // bf16: tensor cores; fp32: the SIMT kernel
    return from_cuda(
        counted(launch_conv_tc(*d, x, stale_prev, w, bias, y, device_status_ptr(), s), 1));
  return from_cuda(counted(launch_conv_simt(*d, x, stale_prev, w, bias, y, s), 1));
}

// ------------------------------------------- conv + GroupNorm, fused sums
dpp_status dpp_conv3x3_gn(const dpp_conv_desc *d, const void *x, const void *stale_prev,
                          const void *w, const float *bias, void *y, int G, double *gn_sums,
                          dpp_stream stream) {
  dpp_status st = check_conv(d, x, stale_prev, w, bias, y);
  if (st != DPP_OK) return st;
  if (!gn_sums || G < 1 || d->C_out % G) return DPP_ERR_INVALID_ARG;
  if (!conv_tc_supported(*d)) return DPP_ERR_UNSUPPORTED;
  if (!aligned16(gn_sums)) return DPP_ERR_ALIGN;
  const size_t es = elem_size(d->dtype);
  const long long pix = (long long)d->B * d->H * d->W;
  const size_t ns = (size_t)d->P * d->B * G * 2 * sizeof(double);
  if (overlap(gn_sums, ns, y, (size_t)pix * d->C_out * es) ||
      overlap(gn_sums, ns, x, (size_t)pix * d->C_in * es) ||
      overlap(gn_sums, ns, stale_prev, (size_t)pix * d->C_in * es) ||
      overlap(gn_sums, ns, w, (size_t)d->C_out * 9 * d->C_in * es) ||
      overlap(gn_sums, ns, bias, (size_t)d->C_out * sizeof(float)))
    return DPP_ERR_ALIAS;
  return from_cuda(counted(launch_conv_tc(*d, x, stale_prev, w, bias, y, device_status_ptr(),
                                          (cudaStream_t)stream, gn_sums, G),
                           2));
}

dpp_status dpp_groupnorm_apply(const dpp_gn_desc *d, const void *x, const float *stats_prev,
                               const double *gn_sums, float *stats_next, const float *gamma,
                               const float *beta, void *y, dpp_stream stream) {
  dpp_status st = check_gn(d);
  if (st != DPP_OK) return st;
  if (!x || !y || !stats_next || !gn_sums) return DPP_ERR_INVALID_ARG;
  if ((gamma == nullptr) != (beta == nullptr)) return DPP_ERR_INVALID_ARG;
  if (d->G > 1024) return DPP_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(y) || !aligned16(stats_next) || !aligned16(gn_sums) ||
      (stats_prev && !aligned16(stats_prev)))
    return DPP_ERR_ALIGN;
  const size_t nx = (size_t)d->B * d->H * d->W * d->C * elem_size(d->dtype);
  const size_t ns = (size_t)d->P * d->B * d->G * 2 * sizeof(float);
  if (y != x && overlap(y, nx, x, nx)) return DPP_ERR_ALIAS;
  if (overlap(stats_prev, ns, stats_next, ns) || overlap(stats_next, ns, y, nx) ||
      overlap(stats_next, ns, gn_sums, 2 * ns) || overlap(y, nx, gn_sums, 2 * ns))
    return DPP_ERR_ALIAS;
  return from_cuda(counted(launch_groupnorm_apply(*d, x, stats_prev, gn_sums, stats_next, gamma,
                                                  beta, y, (cudaStream_t)stream),
                           1));
}

// ------------------------------- GroupNorm -> SiLU applied on the conv's load
dpp_status dpp_groupnorm_sums(const dpp_gn_desc *d, const void *x, double *gn_sums,
                              dpp_stream stream) {
  dpp_status st = check_gn(d);
  if (st != DPP_OK) return st;
  if (!x || !gn_sums) return DPP_ERR_INVALID_ARG;
  if (d->G > 1024 || d->C / chan_quantum(d->dtype) > 512) return DPP_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(gn_sums)) return DPP_ERR_ALIGN;
  const size_t nx = (size_t)d->B * d->H * d->W * d->C * elem_size(d->dtype);
  if (overlap(gn_sums, (size_t)d->P * d->B * d->G * 2 * sizeof(double), x, nx))
    return DPP_ERR_ALIAS;
  return from_cuda(counted(launch_groupnorm_sums(*d, x, gn_sums, (cudaStream_t)stream), 2));
}

dpp_status dpp_groupnorm_affine(const dpp_gn_desc *d, const double *gn_sums,
                                const float *stats_prev, float *stats_next, const float *gamma,
                                const float *beta, float *affine, dpp_stream stream) {
  dpp_status st = check_gn(d);
  if (st != DPP_OK) return st;
  if (!gn_sums || !affine) return DPP_ERR_INVALID_ARG;
  if ((gamma == nullptr) != (beta == nullptr)) return DPP_ERR_INVALID_ARG;
  if (d->G > 1024) return DPP_ERR_UNSUPPORTED;
  if (!aligned16(gn_sums) || !aligned16(affine) || (stats_next && !aligned16(stats_next)) ||
      (stats_prev && !aligned16(stats_prev)))
    return DPP_ERR_ALIGN;
  const size_t ns = (size_t)d->P * d->B * d->G * 2 * sizeof(float);
  const size_t na = (size_t)d->P * d->B * d->C * 2 * sizeof(float);
  if (overlap(affine, na, gn_sums, 2 * ns) || overlap(affine, na, stats_prev, ns) ||
      overlap(affine, na, stats_next, ns) || overlap(affine, na, gamma, d->C * sizeof(float)) ||
      overlap(affine, na, beta, d->C * sizeof(float)) || overlap(stats_next, ns, gn_sums, 2 * ns) ||
      overlap(stats_next, ns, stats_prev, ns))
    return DPP_ERR_ALIAS;
  return from_cuda(counted(launch_groupnorm_affine(*d, gn_sums, stats_prev, stats_next, gamma,
                                                   beta, affine, (cudaStream_t)stream),
                           1));
}

dpp_status dpp_conv3x3_norm(const dpp_conv_desc *d, const void *x, const void *stale_prev,
                            const float *affine, const float *affine_prev, int act,
                            const void *w, const float *bias, void *y, int G, double *gn_sums,
                            dpp_stream stream) {
  dpp_status st = check_conv(d, x, stale_prev, w, bias, y);
  if (st != DPP_OK) return st;
  if (!affine || (act != DPP_ACT_NONE && act != DPP_ACT_SILU)) return DPP_ERR_INVALID_ARG;
  const bool use_stale = stale_prev && stale_prev != x && d->halo == DPP_HALO_STALE;
  if (use_stale && !affine_prev) return DPP_ERR_INVALID_ARG;
  if (gn_sums && (G < 1 || d->C_out % G)) return DPP_ERR_INVALID_ARG;
  if (!conv_tc_supported(*d)) return DPP_ERR_UNSUPPORTED;
  if (!aligned16(affine) || (affine_prev && !aligned16(affine_prev)) ||
      (gn_sums && !aligned16(gn_sums)))
    return DPP_ERR_ALIGN;
  const size_t es = elem_size(d->dtype);
  const long long pix = (long long)d->B * d->H * d->W;
  const size_t ny = (size_t)pix * d->C_out * es;
  const size_t na = (size_t)d->P * d->B * d->C_in * 2 * sizeof(float);
  if (overlap(y, ny, affine, na) || (use_stale && overlap(y, ny, affine_prev, na)))
    return DPP_ERR_ALIAS;
  if (gn_sums) {
    const size_t ns = (size_t)d->P * d->B * G * 2 * sizeof(double);
    if (overlap(gn_sums, ns, y, ny) || overlap(gn_sums, ns, x, (size_t)pix * d->C_in * es) ||
        overlap(gn_sums, ns, stale_prev, (size_t)pix * d->C_in * es) ||
        overlap(gn_sums, ns, w, (size_t)d->C_out * 9 * d->C_in * es) ||
        overlap(gn_sums, ns, bias, (size_t)d->C_out * sizeof(float)) ||
        overlap(gn_sums, ns, affine, na) || (use_stale && overlap(gn_sums, ns, affine_prev, na)))
      return DPP_ERR_ALIAS;
  }
  return from_cuda(counted(
      launch_conv_norm_tc(*d, x, stale_prev, affine, use_stale ? affine_prev : nullptr, act, w,
                          bias, y, device_status_ptr(), (cudaStream_t)stream, gn_sums, G),
      gn_sums ? 2 : 1));
}

// ---------------------------------------------------------------- attention
size_t dpp_self_attn_workspace_bytes(const dpp_attn_desc *d) {
  if (check_attn(d, false) != DPP_OK) return 0;
  const size_t n = attn_tokens(*d) * d->C * elem_bytes(inter_elem(d->dtype));
  return 2 * align_up(n, 256) + wo16_bytes(*d);  // Q, O, fp16 Wo
}

size_t dpp_cross_attn_workspace_bytes(const dpp_attn_desc *d) {
  if (check_attn(d, true) != DPP_OK) return 0;
  // the cached call's Q, O and fp16 Wo, then the context K/V
  return dpp_cross_attn_cached_workspace_bytes(d) + align_up(ctx_kv_bytes(*d), 256);
}

dpp_status dpp_self_attn(const dpp_attn_desc *d, const void *x, const void *wq, const void *wk,
                         const void *wv, const void *wo, const void *kv_prev, void *kv_next,
                         void *y, void *ws, size_t ws_bytes, dpp_stream stream) {
  dpp_status st = check_attn(d, false);
  if (st != DPP_OK) return st;
  if (!x || !wq || !wk || !wv || !wo || !kv_next || !y) return DPP_ERR_INVALID_ARG;
  const void *ptrs[] = {x, wq, wk, wv, wo, kv_next, y, ws};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return DPP_ERR_ALIGN;
  if (kv_prev && !aligned16(kv_prev)) return DPP_ERR_ALIGN;
  const size_t need = dpp_self_attn_workspace_bytes(d);
  if (!ws || ws_bytes < need) return DPP_ERR_WORKSPACE;
  const size_t es = elem_size(d->dtype);
  const Elem te = inter_elem(d->dtype), tl = layer_elem(d->dtype);
  const size_t nt = attn_tokens(*d);
  const size_t nx = nt * d->C * es, nkv = nt * 2 * d->C * elem_bytes(te);
  const size_t nq = nt * d->C * elem_bytes(te);
  if (overlap(kv_prev, nkv, kv_next, nkv)) return DPP_ERR_ALIAS;
  if (overlap(y, nx, kv_next, nkv) || overlap(y, nx, kv_prev, nkv) || overlap(ws, need, y, nx) ||
      overlap(ws, need, x, nx) || overlap(ws, need, kv_next, nkv) ||
      overlap(ws, need, kv_prev, nkv) || overlap(x, nx, kv_next, nkv))
    return DPP_ERR_ALIAS;
  if (y != x && overlap(y, nx, x, nx)) return DPP_ERR_ALIAS;
  cudaStream_t s = (cudaStream_t)stream;
  char *wsb = reinterpret_cast<char *>(ws);
  void *q = wsb;
  void *o = wsb + align_up(nq, 256);
  const int C = d->C;
  const int M = (int)nt;
  // 1. Q for every token (every band's own queries), fresh K/V into kv_next
  GemmArgs qkv{x, {wq, wk, wv}, C, M, 3 * C, C, q, C, C, kv_next, 2 * C, tl, tl, te};
  void *wo16 = wsb + 2 * align_up(nq, 256);
  const bool wo16_ready = attach_wo16(qkv, *d, wo, wo16);
  cudaError_t e = gemm(qkv, s);
  if (e != cudaSuccess) return DPP_ERR_CUDA;
  // 2. displaced attention core
  AttnArgs a{q,      kv_next, d->band_local ? nullptr : kv_prev, o, d->B, d->H * d->W,
             d->H * d->W, C,      d->heads, d->P, te, d->band_local ? 1 : 0};
  e = attn_core(a, s);
  if (e != cudaSuccess) return DPP_ERR_CUDA;
  // 3. output projection
  return from_cuda(out_proj(*d, o, wo, wo16, y, M, s, wo16_ready));
}

dpp_status dpp_cross_attn_kv(const dpp_attn_desc *d, const void *ctx, const void *wk,
                             const void *wv, void *kv_ctx, dpp_stream stream) {
  dpp_status st = check_attn(d, true);
  if (st != DPP_OK) return st;
  if (!ctx || !wk || !wv || !kv_ctx) return DPP_ERR_INVALID_ARG;
  const void *ptrs[] = {ctx, wk, wv, kv_ctx};
  for (const void *p : ptrs)
    if (!aligned16(p)) return DPP_ERR_ALIGN;
  const size_t es = elem_size(d->dtype);
  const size_t nkv = ctx_kv_bytes(*d);
  if (overlap(kv_ctx, nkv, ctx, (size_t)d->B * d->n_ctx * d->c_ctx * es) ||
      overlap(kv_ctx, nkv, wk, (size_t)d->C * d->c_ctx * es) ||
      overlap(kv_ctx, nkv, wv, (size_t)d->C * d->c_ctx * es))
    return DPP_ERR_ALIAS;
  const Elem te = inter_elem(d->dtype), tl = layer_elem(d->dtype);
  const int C = d->C;
  GemmArgs kvg{ctx, {wk, wv, nullptr}, C, d->B * d->n_ctx, 2 * C, d->c_ctx,
               kv_ctx, 2 * C, 2 * C, nullptr, 0, tl, tl, te};
  return from_cuda(gemm(kvg, (cudaStream_t)stream));
}

size_t dpp_cross_attn_cached_workspace_bytes(const dpp_attn_desc *d) {
  if (check_attn(d, true) != DPP_OK) return 0;
  const size_t n = attn_tokens(*d) * d->C * elem_bytes(inter_elem(d->dtype));
  return 2 * align_up(n, 256) + wo16_bytes(*d);  // Q, O, fp16 Wo
}

dpp_status dpp_cross_attn_cached(const dpp_attn_desc *d, const void *x, const void *kv_ctx,
                                 const void *wq, const void *wo, void *y, void *ws,
                                 size_t ws_bytes, dpp_stream stream) {
  dpp_status st = check_attn(d, true);
  if (st != DPP_OK) return st;
  if (!x || !kv_ctx || !wq || !wo || !y) return DPP_ERR_INVALID_ARG;
  const void *ptrs[] = {x, kv_ctx, wq, wo, y, ws};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return DPP_ERR_ALIGN;
  const size_t need = dpp_cross_attn_cached_workspace_bytes(d);
  if (!ws || ws_bytes < need) return DPP_ERR_WORKSPACE;
  const size_t es = elem_size(d->dtype);
  const Elem te = inter_elem(d->dtype), tl = layer_elem(d->dtype);
  const size_t nt = attn_tokens(*d);
  const size_t nx = nt * d->C * es;
  const size_t nq = nt * d->C * elem_bytes(te);
  const size_t nkv = ctx_kv_bytes(*d);
  if (overlap(ws, need, y, nx) || overlap(ws, need, x, nx) || overlap(ws, need, kv_ctx, nkv) ||
      overlap(y, nx, kv_ctx, nkv))
    return DPP_ERR_ALIAS;
  if (y != x && overlap(y, nx, x, nx)) return DPP_ERR_ALIAS;
  cudaStream_t s = (cudaStream_t)stream;
  char *wsb = reinterpret_cast<char *>(ws);
  void *q = wsb;
  void *o = wsb + align_up(nq, 256);
  const int C = d->C;
  GemmArgs qg{x, {wq, nullptr, nullptr}, C, (int)nt, C, C, q, C, C, nullptr, 0, tl, tl, te};
  void *wo16 = wsb + 2 * align_up(nq, 256);
  const bool wo16_ready = attach_wo16(qg, *d, wo, wo16);
  cudaError_t e = gemm(qg, s);
  if (e != cudaSuccess) return DPP_ERR_CUDA;
  AttnArgs a{q, kv_ctx, nullptr, o, d->B, d->H * d->W, d->n_ctx, C, d->heads, 1, te, 0};
  e = attn_core(a, s);
  if (e != cudaSuccess) return DPP_ERR_CUDA;
  return from_cuda(out_proj(*d, o, wo, wo16, y, (int)nt, s, wo16_ready));
}

dpp_status dpp_cross_attn(const dpp_attn_desc *d, const void *x, const void *ctx, const void *wq,
                          const void *wk, const void *wv, const void *wo, void *y, void *ws,
                          size_t ws_bytes, dpp_stream stream) {
  dpp_status st = check_attn(d, true);
  if (st != DPP_OK) return st;
  if (!x || !ctx || !wq || !wk || !wv || !wo || !y) return DPP_ERR_INVALID_ARG;
  const void *ptrs[] = {x, ctx, wq, wk, wv, wo, y, ws};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return DPP_ERR_ALIGN;
  const size_t need = dpp_cross_attn_workspace_bytes(d);
  if (!ws || ws_bytes < need) return DPP_ERR_WORKSPACE;
  const size_t es = elem_size(d->dtype);
  const size_t nt = attn_tokens(*d);
  const size_t nx = nt * d->C * es;
  if (overlap(ws, need, y, nx) || overlap(ws, need, x, nx) ||
      overlap(ws, need, ctx, (size_t)d->B * d->n_ctx * d->c_ctx * es))
    return DPP_ERR_ALIAS;
  if (y != x && overlap(y, nx, x, nx)) return DPP_ERR_ALIAS;
  // the context K/V in the workspace after the cached call's Q, O and Wo
  char *wsb = reinterpret_cast<char *>(ws);
  const size_t cached = dpp_cross_attn_cached_workspace_bytes(d);
  void *kv = wsb + cached;
  st = dpp_cross_attn_kv(d, ctx, wk, wv, kv, stream);
  if (st != DPP_OK) return st;
  return dpp_cross_attn_cached(d, x, kv, wq, wo, y, ws, cached, stream);
}

dpp_status dpp_wait_selftest(int kind, void *scratch, dpp_stream stream) {
  if (kind != 0 && kind != 1) return DPP_ERR_INVALID_ARG;
  if (kind == 0 && !scratch) return DPP_ERR_INVALID_ARG;
  if (scratch && !aligned16(scratch)) return DPP_ERR_ALIGN;
  cudaStream_t s = (cudaStream_t)stream;
  if (kind == 0)
    return from_cuda(counted(
        launch_wait_selftest_counter(reinterpret_cast<const unsigned *>(scratch), s), 1));
  return from_cuda(counted(launch_wait_selftest_mbarrier(s), 1));
}

size_t dpp_workspace_bytes(int op, const void *desc) {
  if (!desc) return 0;
  switch (op) {
    case DPP_OP_GROUPNORM:
      return dpp_groupnorm_workspace_bytes(static_cast<const dpp_gn_desc *>(desc));
    case DPP_OP_SELF_ATTN:
      return dpp_self_attn_workspace_bytes(static_cast<const dpp_attn_desc *>(desc));
    case DPP_OP_CROSS_ATTN:
      return dpp_cross_attn_workspace_bytes(static_cast<const dpp_attn_desc *>(desc));
    case DPP_OP_CFG_COMBINE:
      return dpp_cfg_workspace_bytes(*static_cast<const size_t *>(desc));
    default:
      return 0;
  }
}

// ---------------------------------------------------- per-token layers
dpp_status dpp_layernorm(const dpp_ln_desc *d, const void *x, const float *gamma,
                         const float *beta, void *y, dpp_stream stream) {
  if (!d || !x || !y || !dtype_ok(d->dtype)) return DPP_ERR_INVALID_ARG;
  if (d->T < 1 || d->C < 1 || !(d->eps >= 0.f)) return DPP_ERR_INVALID_ARG;
  if ((gamma == nullptr) != (beta == nullptr)) return DPP_ERR_INVALID_ARG;
  const int q = chan_quantum(d->dtype);
  if (d->C % q) return DPP_ERR_INVALID_ARG;
  if (d->C > 256 * q) return DPP_ERR_UNSUPPORTED;
  if ((long long)d->T * d->C > kMaxElems) return DPP_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(y) || (gamma && !aligned16(gamma)) ||
      (beta && !aligned16(beta)))
    return DPP_ERR_ALIGN;
  const size_t n = (size_t)d->T * d->C * elem_size(d->dtype);
  if (y != x && overlap(y, n, x, n)) return DPP_ERR_ALIAS;
  if (overlap(y, n, gamma, d->C * sizeof(float)) || overlap(y, n, beta, d->C * sizeof(float)))
    return DPP_ERR_ALIAS;
  return from_cuda(
      counted(launch_layernorm(*d, x, gamma, beta, y, (cudaStream_t)stream), 1));
}

dpp_status dpp_linear(const dpp_linear_desc *d, const void *x, const void *w, const float *bias,
                      void *y, dpp_stream stream) {
  if (!d || !x || !w || !y || !dtype_ok(d->dtype)) return DPP_ERR_INVALID_ARG;
  if (d->M < 1 || d->K < 1 || d->N < 1) return DPP_ERR_INVALID_ARG;
  if (d->epilogue != DPP_EPI_NONE && d->epilogue != DPP_EPI_GEGLU) return DPP_ERR_INVALID_ARG;
  if (d->dtype != DPP_BF16) return DPP_ERR_UNSUPPORTED;
  if (d->K % 8 || d->N % 64) return DPP_ERR_INVALID_ARG;
  const bool geglu = d->epilogue == DPP_EPI_GEGLU;
  const long long wrows = geglu ? 2ll * d->N : d->N;
  if ((long long)d->M * d->K > kMaxElems || (long long)d->M * d->N > kMaxElems ||
      wrows * d->K > kMaxElems)
    return DPP_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (bias && !aligned16(bias)))
    return DPP_ERR_ALIGN;
  const size_t nx = (size_t)d->M * d->K * 2, ny = (size_t)d->M * d->N * 2;
  const size_t nw = (size_t)wrows * d->K * 2;
  if (overlap(y, ny, x, nx) || overlap(y, ny, w, nw) ||
      overlap(y, ny, bias, (size_t)wrows * sizeof(float)))
    return DPP_ERR_ALIAS;
  const char *wb = reinterpret_cast<const char *>(w);
  GemmArgs g{x, {w, geglu ? wb + (size_t)d->N * d->K * 2 : nullptr, nullptr}, d->N, d->M, d->N,
             d->K, y, d->N, d->N, nullptr, 0, E_BF16, E_BF16, E_BF16};
  g.bias = bias;
  g.accumulate = d->accumulate ? 1 : 0;
  g.geglu = geglu ? 1 : 0;
  if (!gemm_tc_supported(g)) return DPP_ERR_UNSUPPORTED;
  return from_cuda(counted(launch_gemm_tc(g, device_status_ptr(), (cudaStream_t)stream), 1));
}

}  // extern "C"

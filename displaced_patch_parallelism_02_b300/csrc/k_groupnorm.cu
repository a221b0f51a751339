// Displaced GroupNorm (DistriGroupNorm, section 归一化层拆分 of the
// DistriFusion developer guide).
//
// Per band p, batch b, group g the statistics combine the band's fresh
// partial sums (sum x, sum x^2) with the stale partials of every other band
// from the previous step; the band's fresh partials are published to
// stats_next (the refresh of the GroupNorm state).  With no stale input
// (the synchronous first step) all bands' fresh partials are combined.
//
// Two passes over NHWC data, both HBM-bound and fully coalesced:
//   1. partials: the (band, batch) unit is cut into pixel chunks; a block
//      reads 16-byte vectors (thread t always holds vector t % (C/VE) of a
//      pixel, so its channels -- and the at most two groups they straddle --
//      are fixed) and reduces per channel, then per group, in a fixed order.
//   2. apply: each block rebuilds the unit's group statistics from the chunk
//      partials (fp64, fixed order), folds mean/rstd/gamma/beta into one
//      scale and shift per channel and normalises its chunk.  Pass 2
//      re-reads the chunk pass 1 just read; it comes from L2 when the
//      tensor fits there.
#include <mutex>

#include "dpp_internal.h"

namespace dpp {
namespace {

template <typename T>
struct Vec16;

template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void load(const float *p, float f[4]) {
    const float4 v = *reinterpret_cast<const float4 *>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
  __device__ static void store(float *p, const float f[4]) {
    *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
};

template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const __nv_bfloat16 *p, float f[8]) {
    const uint4 v = *reinterpret_cast<const uint4 *>(p);
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ static void store(__nv_bfloat16 *p, const float f[8]) {
    uint4 v;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    *reinterpret_cast<uint4 *>(p) = v;
  }
};

struct GnGeom {
  int B, H, W, C, G, P;
  int pix_per_chunk, chunks;
};

template <typename T>
__global__ void __launch_bounds__(1024)
gn_partials_kernel(const T *__restrict__ x, GnGeom g, float *__restrict__ partials) {
  constexpr int VE = Vec16<T>::N;
  extern __shared__ float sm[];
  const int VPP = g.C / VE;
  const int R = blockDim.x / VPP;
  float *s1 = sm, *s2 = sm + R * g.C, *c1 = sm + 2 * R * g.C, *c2 = c1 + g.C;
  const int unit = blockIdx.y, b = unit / g.P, p = unit % g.P, chunk = blockIdx.x;
  const int Hp = g.H / g.P;
  const int npix = Hp * g.W;
  const size_t base = ((size_t)b * g.H + (size_t)p * Hp) * g.W;  // first pixel of the band
  const int j0 = chunk * g.pix_per_chunk;
  const int j1 = min(j0 + g.pix_per_chunk, npix);
  const int v = threadIdx.x % VPP, r = threadIdx.x / VPP;
  if (r < R) {
    float a1[VE], a2[VE];
#pragma unroll
    for (int e = 0; e < VE; ++e) a1[e] = a2[e] = 0.f;
    for (int j = j0 + r; j < j1; j += R) {
      float f[VE];
      Vec16<T>::load(x + (base + j) * g.C + v * VE, f);
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        a1[e] += f[e];
        a2[e] = fmaf(f[e], f[e], a2[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      s1[r * g.C + v * VE + e] = a1[e];
      s2[r * g.C + v * VE + e] = a2[e];
    }
  }
  __syncthreads();
  for (int ch = threadIdx.x; ch < g.C; ch += blockDim.x) {
    float t1 = 0.f, t2 = 0.f;
    for (int rr = 0; rr < R; ++rr) {
      t1 += s1[rr * g.C + ch];
      t2 += s2[rr * g.C + ch];
    }
    c1[ch] = t1;
    c2[ch] = t2;
  }
  __syncthreads();
  const int cg = g.C / g.G;
  for (int gg = threadIdx.x; gg < g.G; gg += blockDim.x) {
    float t1 = 0.f, t2 = 0.f;
    for (int k = 0; k < cg; ++k) {
      t1 += c1[gg * cg + k];
      t2 += c2[gg * cg + k];
    }
    float *dst = partials + (((size_t)unit * g.chunks + chunk) * g.G + gg) * 2;
    dst[0] = t1;
    dst[1] = t2;
  }
}

template <typename T>
__global__ void __launch_bounds__(1024)
gn_apply_kernel(const T *x, T *y, GnGeom g, const float *__restrict__ partials,
                const float *__restrict__ stats_prev, float *__restrict__ stats_next,
                const float *__restrict__ gamma, const float *__restrict__ beta, float eps) {
  constexpr int VE = Vec16<T>::N;
  extern __shared__ float sm[];
  float *mean_s = sm, *rstd_s = sm + g.G;
  const int unit = blockIdx.y, b = unit / g.P, p = unit % g.P, chunk = blockIdx.x;
  const int Hp = g.H / g.P;
  const int npix = Hp * g.W;
  for (int gg = threadIdx.x; gg < g.G; gg += blockDim.x) {
    double f1 = 0.0, f2 = 0.0;
    for (int k = 0; k < g.chunks; ++k) {
      const float *src = partials + (((size_t)unit * g.chunks + k) * g.G + gg) * 2;
      f1 += src[0];
      f2 += src[1];
    }
    double t1 = f1, t2 = f2;
    for (int q = 0; q < g.P; ++q) {
      if (q == p) continue;
      if (stats_prev) {
        const float *src = stats_prev + (((size_t)q * g.B + b) * g.G + gg) * 2;
        t1 += src[0];
        t2 += src[1];
      } else {
        const int uq = b * g.P + q;
        for (int k = 0; k < g.chunks; ++k) {
          const float *src = partials + (((size_t)uq * g.chunks + k) * g.G + gg) * 2;
          t1 += src[0];
          t2 += src[1];
        }
      }
    }
    const double n = (double)g.H * g.W * (g.C / g.G);
    const double mean = t1 / n;
    const double var = fmax(t2 / n - mean * mean, 0.0);
    mean_s[gg] = (float)mean;
    rstd_s[gg] = (float)(1.0 / sqrt(var + (double)eps));
    if (chunk == 0) {
      float *dst = stats_next + (((size_t)p * g.B + b) * g.G + gg) * 2;
      dst[0] = (float)f1;
      dst[1] = (float)f2;
    }
  }
  __syncthreads();
  const int VPP = g.C / VE;
  const int R = blockDim.x / VPP;
  const int v = threadIdx.x % VPP, r = threadIdx.x / VPP;
  if (r >= R) return;
  const int cg = g.C / g.G;
  float sc[VE], sh[VE];
#pragma unroll
  for (int e = 0; e < VE; ++e) {
    const int ch = v * VE + e, gg = ch / cg;
    const float a = rstd_s[gg] * (gamma ? gamma[ch] : 1.f);
    sc[e] = a;
    sh[e] = (beta ? beta[ch] : 0.f) - mean_s[gg] * a;
  }
  const size_t base = ((size_t)b * g.H + (size_t)p * Hp) * g.W;
  const int j0 = chunk * g.pix_per_chunk;
  const int j1 = min(j0 + g.pix_per_chunk, npix);
  for (int j = j0 + r; j < j1; j += R) {
    float f[VE];
    const size_t off = (base + j) * g.C + v * VE;
    Vec16<T>::load(x + off, f);
#pragma unroll
    for (int e = 0; e < VE; ++e) f[e] = fmaf(f[e], sc[e], sh[e]);
    Vec16<T>::store(y + off, f);
  }
}

int gn_threads(const dpp_gn_desc &d) {
  const int VE = d.dtype == DPP_BF16 ? 8 : 4;
  const int VPP = d.C / VE;
  int R = 512 / VPP;
  if (R < 1) R = 1;
  return R * VPP;
}

}  // namespace

GnPlan gn_plan(const dpp_gn_desc &d) {
  GnPlan pl;
  pl.units = d.P * d.B;
  pl.pix_per_unit = (d.H / d.P) * d.W;
  int want = (592 + pl.units - 1) / pl.units;  // about one wave of blocks in total
  int cap = (pl.pix_per_unit + 63) / 64;     // at least 64 pixels per chunk
  int chunks = want < cap ? want : cap;
  if (chunks < 1) chunks = 1;
  pl.pix_per_chunk = (pl.pix_per_unit + chunks - 1) / chunks;
  pl.chunks = (pl.pix_per_unit + pl.pix_per_chunk - 1) / pl.pix_per_chunk;
  return pl;
}

size_t gn_workspace(const dpp_gn_desc &d) {
  const GnPlan pl = gn_plan(d);
  return align_up((size_t)pl.units * pl.chunks * d.G * 2 * sizeof(float), 256);
}

cudaError_t launch_groupnorm(const dpp_gn_desc &d, const void *x, const float *stats_prev,
                             float *stats_next, const float *gamma, const float *beta,
                             void *y, void *ws, cudaStream_t s) {
  const GnPlan pl = gn_plan(d);
  GnGeom g{d.B, d.H, d.W, d.C, d.G, d.P, pl.pix_per_chunk, pl.chunks};
  const int threads = gn_threads(d);
  const int VE = d.dtype == DPP_BF16 ? 8 : 4;
  const int R = threads / (d.C / VE);
  const size_t smem1 = (size_t)(2 * R * d.C + 2 * d.C) * sizeof(float);
  const size_t smem2 = (size_t)(2 * d.G) * sizeof(float);
  float *partials = reinterpret_cast<float *>(ws);
  dim3 grid(pl.chunks, pl.units);
  if (d.dtype == DPP_BF16) {
    auto k1 = gn_partials_kernel<__nv_bfloat16>;
    cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
    k1<<<grid, threads, smem1, s>>>((const __nv_bfloat16 *)x, g, partials);
    gn_apply_kernel<__nv_bfloat16><<<grid, threads, smem2, s>>>(
        (const __nv_bfloat16 *)x, (__nv_bfloat16 *)y, g, partials, stats_prev, stats_next,
        gamma, beta, d.eps);
  } else {
    auto k1 = gn_partials_kernel<float>;
    cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
    k1<<<grid, threads, smem1, s>>>((const float *)x, g, partials);
    gn_apply_kernel<float><<<grid, threads, smem2, s>>>((const float *)x, (float *)y, g,
                                                         partials, stats_prev, stats_next,
                                                         gamma, beta, d.eps);
  }
  return cudaGetLastError();
}

}  // namespace dpp

// ---------------------------------------------------------------------------
// Allocation-free GroupNorm.  Some callers cannot allocate device memory:
// plugins that run inside a host program which owns the whole device-memory
// budget (an inference server's pre-planned arena, a framework layer API
// that hands out no workspace), or code that must not call cudaMalloc on a
// hot path because cudaMalloc may synchronise the device.  For them the
// partial-sum scratch lives in this file-scope device array instead of a
// caller workspace.  Every GPU that loads the library holds the array until
// the process exits.  All calls share it: calls whose kernels overlap on the
// GPU (two streams, or two host threads) race on it.
namespace dpp {

static __device__ __align__(256) unsigned char g_gn_static_scratch[kGnStaticScratchBytes];

namespace {
std::mutex g_gn_static_mutex;
void *g_gn_static_ptr[64] = {};
}  // namespace

cudaError_t launch_groupnorm_static(const dpp_gn_desc &d, const void *x, const float *stats_prev,
                                    float *stats_next, const float *gamma, const float *beta,
                                    void *y, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void *scratch = nullptr;
  {
    // Set-up, once per device, with that device current: the host-side name
    // of the array is not a device address, so look the address up.
    std::lock_guard<std::mutex> lock(g_gn_static_mutex);
    if (!g_gn_static_ptr[dev]) {
      void *p = nullptr;
      e = cudaGetSymbolAddress(&p, g_gn_static_scratch);
      if (e != cudaSuccess) return e;
      g_gn_static_ptr[dev] = p;
    }
    scratch = g_gn_static_ptr[dev];
  }
  // The partial sums are fully written by the first pass before the second
  // reads them, so nothing in the array needs clearing between calls.
  return launch_groupnorm(d, x, stats_prev, stats_next, gamma, beta, y, scratch, s);
}

}  // namespace dpp

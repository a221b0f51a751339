// Classifier-free-guidance combine and the denoising-discrepancy sums.
//
// out = eps_u + s * (eps_c - eps_u); sums3 = (sum|c-u|, sum|u|, sum|c|).
// The guided estimate is the combine of the conditional and unconditional
// branches that the Hydiff summaries split across devices (gist.science,
// "基于条件的数据划分"); the sums feed the rel-MAE switching signal of
// "自适应并行切换" (Avetisyan, "Адаптивное переключение": the discrepancy is
// the conditional minus the unconditional estimate).
//
// HBM-bound single pass: 16-byte loads of u and c, one 16-byte store.
// Reduction: fp32 within a block (per thread, then a warp-shuffle tree, then
// the 8 warp sums), fp64 across blocks; block partials go to the workspace
// and the last block to finish (a wrapping atomicInc counter, which it
// leaves at zero) adds them in a fixed order.  The grid depends only on n,
// so the sums are bit-reproducible.  FP64 arithmetic runs at a small
// fraction of the FP32 rate on this part, so it is kept to the few
// additions per block that the cross-block combine needs; a block's fp32
// tree over at most a few thousand terms carries a relative error of a few
// times 2^-24.
#include "dpp_internal.h"

namespace dpp {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__global__ void __launch_bounds__(kThreads)
cfg_kernel(const float *__restrict__ u, const float *__restrict__ c, float s, size_t n,
           float *out, double *sums3, unsigned *counter, double *partials) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f;
  const size_t n4 = n / 4;
  const size_t stride = (size_t)gridDim.x * kThreads;
  const float4 *u4 = reinterpret_cast<const float4 *>(u);
  const float4 *c4 = reinterpret_cast<const float4 *>(c);
  float4 *o4 = reinterpret_cast<float4 *>(out);
  // four vectors of each map per thread per pass, all loads issued before
  // any arithmetic: one DRAM round trip per pass instead of four
  for (size_t i0 = (size_t)blockIdx.x * kThreads + threadIdx.x; i0 < n4; i0 += 4 * stride) {
    float4 uu[4], cc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const size_t i = i0 + k * stride;
      uu[k] = i < n4 ? __ldcs(u4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      cc[k] = i < n4 ? __ldcs(c4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const size_t i = i0 + k * stride;
      const float4 a = uu[k], c = cc[k];
      const float dx = c.x - a.x, dy = c.y - a.y, dz = c.z - a.z, dw = c.w - a.w;
      if (i < n4)
        __stcs(o4 + i, make_float4(fmaf(s, dx, a.x), fmaf(s, dy, a.y), fmaf(s, dz, a.z),
                                   fmaf(s, dw, a.w)));
      a0 += fabsf(dx) + fabsf(dy) + fabsf(dz) + fabsf(dw);
      a1 += fabsf(a.x) + fabsf(a.y) + fabsf(a.z) + fabsf(a.w);
      a2 += fabsf(c.x) + fabsf(c.y) + fabsf(c.z) + fabsf(c.w);
    }
  }
  if (blockIdx.x == 0 && threadIdx.x < n - 4 * n4) {  // scalar tail (< 4 elements)
    const size_t i = 4 * n4 + threadIdx.x;
    const float d = c[i] - u[i];
    out[i] = fmaf(s, d, u[i]);
    a0 += fabsf(d);
    a1 += fabsf(u[i]);
    a2 += fabsf(c[i]);
  }
  if (sums3 == nullptr) return;

  __shared__ float sm[kThreads / 32][3];
  __shared__ bool is_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a0 = warp_sum(a0);
  a1 = warp_sum(a1);
  a2 = warp_sum(a2);
  if (lane == 0) {
    sm[warp][0] = a0;
    sm[warp][1] = a1;
    sm[warp][2] = a2;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 0; k < 3; ++k) {
      double t = 0.0;
      for (int w = 0; w < kThreads / 32; ++w) t += (double)sm[w][k];
      partials[blockIdx.x * 3 + k] = t;
    }
    __threadfence();
    const unsigned prev = atomicInc(counter, gridDim.x - 1);  // wraps to 0 on the last block
    is_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  if (warp < 3) {  // warp k adds quantity k: lane l takes blocks l, l + 32, ...
    double t4[4] = {0.0, 0.0, 0.0, 0.0};  // independent sums: many L2 loads in flight
    unsigned b = lane;
    for (; b + 96 < gridDim.x; b += 128)
#pragma unroll
      for (int k = 0; k < 4; ++k) t4[k] += __ldcg(partials + (b + 32 * k) * 3 + warp);
    for (; b < gridDim.x; b += 32) t4[0] += __ldcg(partials + b * 3 + warp);
    double t = (t4[0] + t4[1]) + (t4[2] + t4[3]);
    t = warp_sum(t);
    if (lane == 0) sums3[warp] = t;
  }
}

}  // namespace

// Two blocks per SM: each thread keeps several 16-byte loads in flight and
// the final combine adds few partials.  A function of n only.
constexpr size_t kCfgMaxBlocks = 296;

size_t cfg_blocks(size_t n) {
  size_t b = (n / 4 + kThreads - 1) / kThreads;
  if (b < 1) b = 1;
  if (b > kCfgMaxBlocks) b = kCfgMaxBlocks;
  return b;
}

cudaError_t launch_cfg(const float *u, const float *c, float scale, size_t n, float *out,
                       double *sums3, void *ws, cudaStream_t s) {
  const unsigned blocks = (unsigned)cfg_blocks(n);
  unsigned *counter = sums3 ? reinterpret_cast<unsigned *>(ws) : nullptr;
  double *partials = sums3 ? reinterpret_cast<double *>((char *)ws + 16) : nullptr;
  cfg_kernel<<<blocks, kThreads, 0, s>>>(u, c, scale, n, out, sums3, counter, partials);
  return cudaGetLastError();
}

}  // namespace dpp

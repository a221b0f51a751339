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
// Reduction: fp32 per thread over a handful of elements, fp64 from the warp
// level up; block partials go to the workspace and the last block to finish
// (a wrapping atomicInc counter, which it leaves at zero) adds them in block
// order.  The grid depends only on n, so the sums are bit-reproducible.
#include "dpp_internal.h"

namespace dpp {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Sums three per-thread values over the block in a fixed order; result
// valid in thread 0.
__device__ __forceinline__ void block_sum3(double v[3], double (*sm)[3]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < 3; ++k) v[k] = warp_sum(v[k]);
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < 3; ++k) sm[warp][k] = v[k];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 0; k < 3; ++k) {
      double t = 0.0;
      for (int w = 0; w < kThreads / 32; ++w) t += sm[w][k];
      v[k] = t;
    }
  }
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
  for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < n4; i += stride) {
    const float4 uu = __ldcs(u4 + i), cc = __ldcs(c4 + i);
    const float dx = cc.x - uu.x, dy = cc.y - uu.y, dz = cc.z - uu.z, dw = cc.w - uu.w;
    __stcs(o4 + i, make_float4(fmaf(s, dx, uu.x), fmaf(s, dy, uu.y), fmaf(s, dz, uu.z),
                               fmaf(s, dw, uu.w)));
    a0 += fabsf(dx) + fabsf(dy) + fabsf(dz) + fabsf(dw);
    a1 += fabsf(uu.x) + fabsf(uu.y) + fabsf(uu.z) + fabsf(uu.w);
    a2 += fabsf(cc.x) + fabsf(cc.y) + fabsf(cc.z) + fabsf(cc.w);
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

  __shared__ double sm[kThreads / 32][3];
  __shared__ bool is_last;
  double v[3] = {a0, a1, a2};
  block_sum3(v, sm);
  if (threadIdx.x == 0) {
    for (int k = 0; k < 3; ++k) partials[blockIdx.x * 3 + k] = v[k];
    __threadfence();
    const unsigned prev = atomicInc(counter, gridDim.x - 1);  // wraps to 0 on the last block
    is_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  double t[3] = {0.0, 0.0, 0.0};
  for (unsigned b = threadIdx.x; b < gridDim.x; b += kThreads)
    for (int k = 0; k < 3; ++k) t[k] += __ldcg(partials + b * 3 + k);
  __syncthreads();  // sm reuse
  block_sum3(t, sm);
  if (threadIdx.x == 0)
    for (int k = 0; k < 3; ++k) sums3[k] = t[k];
}

}  // namespace

size_t cfg_blocks(size_t n) {
  size_t b = (n / 4 + kThreads - 1) / kThreads;
  if (b < 1) b = 1;
  if (b > (size_t)kReduceBlocks) b = kReduceBlocks;
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

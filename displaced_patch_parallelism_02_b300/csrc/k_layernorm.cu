// Token-wise LayerNorm of the U-Net's transformer blocks: each token's C
// channels are normalised by their own mean and biased variance.  A token is
// local to its band, so no stale state enters (the DistriFusion developer
// guide replaces only the convolutions, attention layers and GroupNorms).
//
// One warp per token: the token's 16-byte channel vectors are spread over the
// lanes (lane l holds vectors l, l + 32, ... -- at most V per lane) and stay
// in registers, so the mean and then the variance about it are two warp
// reductions over registers and x is read from HBM exactly once.  The grid is
// whole waves of the SM count; each warp walks tokens with a grid stride.
// Bound: HBM (read x, write y).
#include <cuda_bf16.h>

#include "dpp_internal.h"

namespace dpp {
namespace {

constexpr int kLnWarps = 8;  // warps per CTA

template <typename T>
struct LnVec;

template <>
struct LnVec<float> {
  static constexpr int N = 4;
  __device__ static void unpack(const uint4 &v, float f[4]) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  __device__ static uint4 pack(const float f[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

template <>
struct LnVec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void unpack(const uint4 &v, float f[8]) {  // bf16 -> fp32: 16-bit shift
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static uint4 pack(const float f[8]) {
    uint4 v;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return v;
  }
};

__device__ __forceinline__ float ln_warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <typename T, int V>
__global__ void __launch_bounds__(kLnWarps * 32)
layernorm_kernel(const T *x, T *y, const float *__restrict__ gamma,
                 const float *__restrict__ beta, int tokens, int C, float eps) {
  constexpr int VE = LnVec<T>::N;
  const int lane = threadIdx.x % 32;
  const int nvec = C / VE;
  // gamma and beta for the whole token, once per CTA, in shared memory (the
  // registers go to keeping more tokens' loads in flight)
  extern __shared__ float ln_aff[];  // [2][C]
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    ln_aff[c] = gamma ? gamma[c] : 1.f;
    ln_aff[C + c] = beta ? beta[c] : 0.f;
  }
  __syncthreads();
  const float inv_c = 1.f / (float)C;
  const int warps = gridDim.x * kLnWarps;
  for (int t = blockIdx.x * kLnWarps + threadIdx.x / 32; t < tokens; t += warps) {
    const T *xr = x + (size_t)t * C;
    uint4 raw[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int v = lane + 32 * i;
      raw[i] = v < nvec ? __ldcs(reinterpret_cast<const uint4 *>(xr) + v)
                        : make_uint4(0u, 0u, 0u, 0u);
    }
    float f[V][VE];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      LnVec<T>::unpack(raw[i], f[i]);
#pragma unroll
      for (int e = 0; e < VE; ++e) s += f[i][e];
    }
    const float mean = ln_warp_sum(s) * inv_c;
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      if (lane + 32 * i < nvec) {
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          const float d = f[i][e] - mean;
          q = fmaf(d, d, q);
        }
      }
    }
    const float rstd = rsqrtf(ln_warp_sum(q) * inv_c + eps);
    T *yr = y + (size_t)t * C;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int v = lane + 32 * i;
      if (v < nvec) {
        // 16-byte shared loads of the vector's gains and shifts (a lane's
        // VE floats are contiguous: at most a 2-way bank conflict)
        float ga[VE], be[VE];
#pragma unroll
        for (int q = 0; q < VE / 4; ++q) {
          const float4 g4 = reinterpret_cast<const float4 *>(ln_aff + v * VE)[q];
          const float4 b4 = reinterpret_cast<const float4 *>(ln_aff + C + v * VE)[q];
          ga[4 * q] = g4.x; ga[4 * q + 1] = g4.y; ga[4 * q + 2] = g4.z; ga[4 * q + 3] = g4.w;
          be[4 * q] = b4.x; be[4 * q + 1] = b4.y; be[4 * q + 2] = b4.z; be[4 * q + 3] = b4.w;
        }
        float o[VE];
#pragma unroll
        for (int e = 0; e < VE; ++e) o[e] = fmaf((f[i][e] - mean) * rstd, ga[e], be[e]);
        __stcs(reinterpret_cast<uint4 *>(yr) + v, LnVec<T>::pack(o));
      }
    }
  }
}

template <typename T, int V>
cudaError_t run_ln(const dpp_ln_desc &d, const void *x, const float *gamma, const float *beta,
                   void *y, cudaStream_t s) {
  auto k = layernorm_kernel<T, V>;
  int dev = 0, sms = 148, per_sm = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t smem = (size_t)2 * d.C * sizeof(float);
  cudaError_t e =
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kLnWarps * 32, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const long long need = (d.T + kLnWarps - 1) / kLnWarps;
  const long long full = (long long)sms * per_sm;
  const int grid = (int)(need < full ? need : full);
  k<<<grid, kLnWarps * 32, smem, s>>>((const T *)x, (T *)y, gamma, beta, d.T, d.C, d.eps);
  return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_ln(const dpp_ln_desc &d, const void *x, const float *gamma,
                        const float *beta, void *y, cudaStream_t s) {
  const int nvec = d.C / LnVec<T>::N;
  const int v = (nvec + 31) / 32;  // vectors per lane
  if (v <= 1) return run_ln<T, 1>(d, x, gamma, beta, y, s);
  if (v <= 2) return run_ln<T, 2>(d, x, gamma, beta, y, s);
  if (v <= 3) return run_ln<T, 3>(d, x, gamma, beta, y, s);
  if (v <= 4) return run_ln<T, 4>(d, x, gamma, beta, y, s);
  if (v <= 8) return run_ln<T, 8>(d, x, gamma, beta, y, s);
  return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_layernorm(const dpp_ln_desc &d, const void *x, const float *gamma,
                             const float *beta, void *y, cudaStream_t s) {
  if (d.dtype == DPP_BF16) return dispatch_ln<__nv_bfloat16>(d, x, gamma, beta, y, s);
  return dispatch_ln<float>(d, x, gamma, beta, y, s);
}

}  // namespace dpp

// SIMT (CUDA-core, fp32 arithmetic) kernels: the fp32 path of the library and
// the shape-general path for bf16.  No TF32: the fp32 tolerance of the
// displaced ops (1e-4 of the output RMS) is below TF32's 10-bit mantissa.
//
//   conv_simt   displaced 3x3 conv as an implicit GEMM, 64x64 output tile,
//               16-wide K chunks; the A loader picks the fresh or stale
//               tensor per input row (DistriConv2dPP: only the halo rows
//               next to the band are stale).
//   gemm_simt   D = A B^T for the attention projections, B split into up to
//               three weight blocks and D split into two destinations, so
//               one launch writes Q to the workspace and the fresh K/V of
//               every token straight into the next step's state.
//   attn_simt   flash-style attention for head_dim 64 (online softmax in the
//               exp2 domain); the K/V loader picks fresh rows for the query
//               band's own tokens and stale rows elsewhere
//               (DistriSelfAttentionPP).
#include "dpp_internal.h"

namespace dpp {
namespace {

template <typename T>
__device__ __forceinline__ void load4(const T *p, float f[4]);

template <>
__device__ __forceinline__ void load4<float>(const float *p, float f[4]) {
  const float4 v = *reinterpret_cast<const float4 *>(p);
  f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}

template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16 *p, float f[4]) {
  const uint2 v = *reinterpret_cast<const uint2 *>(p);
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
  const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

template <>
__device__ __forceinline__ void load4<__half>(const __half *p, float f[4]) {
  const uint2 v = *reinterpret_cast<const uint2 *>(p);
  const __half2 *h = reinterpret_cast<const __half2 *>(&v);
  const float2 a = __half22float2(h[0]), b = __half22float2(h[1]);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f(__half v) { return __half2float(v); }

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

// ----------------------------------------------------------------- conv
struct ConvGeom {
  int B, H, W, Ci, Co, P, fresh_halo, zero_halo, accumulate;
};

template <typename T>
__global__ void __launch_bounds__(NT)
conv_simt_kernel(const T *__restrict__ x, const T *__restrict__ stale, const T *__restrict__ w,
                 const float *__restrict__ bias, T *__restrict__ y, ConvGeom g) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int M = g.B * g.H * g.W;
  const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  const int lm = tid / 4, lq = tid % 4;
  const int m = m0 + lm;
  const bool m_ok = m < M;
  const int w_ = m_ok ? m % g.W : 0;
  const int h_ = m_ok ? (m / g.W) % g.H : 0;
  const int b_ = m_ok ? m / (g.W * g.H) : 0;
  const int Hp = g.H / g.P;
  const int lo = (h_ / Hp) * Hp, hi = lo + Hp;
  const int co_l = n0 + lm;
  float acc[4][4] = {};
  for (int tap = 0; tap < 9; ++tap) {
    const int dy = tap / 3, dx = tap % 3;
    const int r = h_ + dy - 1, c = w_ + dx - 1;
    const bool in_img = m_ok && r >= 0 && r < g.H && c >= 0 && c < g.W &&
                        !(g.zero_halo && (r < lo || r >= hi));
    const T *src = (g.fresh_halo || (r >= lo && r < hi)) ? x : stale;
    const T *arow = src + (((size_t)b_ * g.H + (in_img ? r : 0)) * g.W + (in_img ? c : 0)) * g.Ci;
    const T *wrow = w + ((size_t)(co_l < g.Co ? co_l : 0) * 9 + tap) * g.Ci;
    for (int ci0 = 0; ci0 < g.Ci; ci0 += BK) {
      const int ch = ci0 + lq * 4;
      float a4[4] = {0.f, 0.f, 0.f, 0.f}, b4[4] = {0.f, 0.f, 0.f, 0.f};
      if (in_img && ch < g.Ci) load4<T>(arow + ch, a4);
      if (co_l < g.Co && ch < g.Ci) load4<T>(wrow + ch, b4);
      __syncthreads();
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        As[lq * 4 + e][lm] = a4[e];
        Bs[lq * 4 + e][lm] = b4[e];
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < BK; ++k) {
        float a[4], bb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = As[k][ty + 16 * i];
#pragma unroll
        for (int j = 0; j < 4; ++j) bb[j] = Bs[k][tx + 16 * j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int mm = m0 + ty + 16 * i;
    if (mm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int co = n0 + tx + 16 * j;
      if (co < g.Co) {
        float v = acc[i][j] + (bias ? bias[co] : 0.f);
        if (g.accumulate) v += to_f(y[(size_t)mm * g.Co + co]);
        y[(size_t)mm * g.Co + co] = from_f<T>(v);
      }
    }
  }
}

// ----------------------------------------------------------------- gemm
template <typename TA, typename TB, typename TO>
__global__ void __launch_bounds__(NT) gemm_simt_kernel(const __grid_constant__ GemmArgs g) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const TA *A = reinterpret_cast<const TA *>(g.A);
  const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  const int lm = tid / 4, lq = tid % 4;
  const int am = m0 + lm, bn = n0 + lm;
  const TA *arow = A + (size_t)(am < g.M ? am : 0) * g.K;
  const TB *brow = reinterpret_cast<const TB *>(g.B[bn < g.N ? bn / g.b_rows : 0]) +
                   (size_t)(bn < g.N ? bn % g.b_rows : 0) * g.K;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < g.K; k0 += BK) {
    const int kk = k0 + lq * 4;
    float a4[4] = {0.f, 0.f, 0.f, 0.f}, b4[4] = {0.f, 0.f, 0.f, 0.f};
    if (am < g.M && kk < g.K) load4<TA>(arow + kk, a4);
    if (bn < g.N && kk < g.K) load4<TB>(brow + kk, b4);
    __syncthreads();
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      As[lq * 4 + e][lm] = a4[e];
      Bs[lq * 4 + e][lm] = b4[e];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      float a[4], bb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[k][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bb[j] = Bs[k][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
    }
  }
  TO *o0 = reinterpret_cast<TO *>(g.out0);
  TO *o1 = reinterpret_cast<TO *>(g.out1);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int mm = m0 + ty + 16 * i;
    if (mm >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int nn = n0 + tx + 16 * j;
      if (nn >= g.N) continue;
      if (nn < g.split) {
        float v = acc[i][j] + (g.bias ? g.bias[nn] : 0.f);
        if (g.accumulate) v += to_f(o0[(size_t)mm * g.ld0 + nn]);
        o0[(size_t)mm * g.ld0 + nn] = from_f<TO>(v);
      } else
        o1[(size_t)mm * g.ld1 + (nn - g.split)] = from_f<TO>(acc[i][j]);
    }
  }
}

// ----------------------------------------------------------------- attention
constexpr int AQ = 64, AK = 64, AD = 64;
constexpr int kAttnSmemFloats = AD * (AQ + 4) + AD * (AK + 1) + AK * (AD + 4) + AQ * (AK + 1);

template <typename T>
__global__ void __launch_bounds__(NT) attn_simt_kernel(AttnArgs a) {
  extern __shared__ float sm[];
  float(*Qs)[AQ + 4] = reinterpret_cast<float(*)[AQ + 4]>(sm);                   // [d][q]
  float(*Ks)[AK + 1] = reinterpret_cast<float(*)[AK + 1]>(sm + AD * (AQ + 4));  // [d][kv]
  float(*Vs)[AD + 4] =
      reinterpret_cast<float(*)[AD + 4]>(sm + AD * (AQ + 4) + AD * (AK + 1));  // [kv][d]
  float(*Ps)[AK + 1] = reinterpret_cast<float(*)[AK + 1]>(sm + AD * (AQ + 4) + AD * (AK + 1) +
                                                          AK * (AD + 4));     // [q][kv]
  const T *Q = reinterpret_cast<const T *>(a.q);
  const T *KVf = reinterpret_cast<const T *>(a.kv_fresh);
  const T *KVs = reinterpret_cast<const T *>(a.kv_stale);
  T *O = reinterpret_cast<T *>(a.o);
  const int head = blockIdx.y, b = blockIdx.z;
  const int Np = a.Nq / a.P;
  const int tpb = (Np + AQ - 1) / AQ;
  const int p = blockIdx.x / tpb, t = blockIdx.x % tpb;
  const int q0 = p * Np + t * AQ;
  const int qend = (p + 1) * Np;
  const int kv_lo = (a.Nkv == a.Nq) ? p * Np : 0;
  const int kv_hi = (a.Nkv == a.Nq) ? (p + 1) * Np : a.Nkv;
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  const int lr = tid / 4, lq = tid % 4;  // loader: row lr, 16-wide d chunk lq
  const float qscale = 0.125f * 1.4426950408889634f;  // 1/sqrt(64) * log2(e)

  {  // Q tile, pre-scaled into the exp2 domain, stored [d][q]
    const int q = q0 + lr;
    const bool ok = q < qend;
    const T *src = Q + ((size_t)b * a.Nq + (ok ? q : q0)) * a.C + head * AD + lq * 16;
#pragma unroll
    for (int e4 = 0; e4 < 4; ++e4) {
      float f[4] = {0.f, 0.f, 0.f, 0.f};
      if (ok) load4<T>(src + e4 * 4, f);
#pragma unroll
      for (int e = 0; e < 4; ++e) Qs[lq * 16 + e4 * 4 + e][lr] = f[e] * qscale;
    }
  }
  float m_i[4], l_i[4], acc[4][4] = {};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m_i[i] = -INFINITY;
    l_i[i] = 0.f;
  }
  // band-local (naive patches): only the band's own keys
  const int k_begin = a.band_local ? kv_lo : 0, k_end = a.band_local ? kv_hi : a.Nkv;
  for (int kv0 = k_begin; kv0 < k_end; kv0 += AK) {
    __syncthreads();  // previous tile fully consumed
    {
      const int kv = kv0 + lr;
      const bool ok = kv < k_end;
      const bool fresh = (KVs == nullptr) || (kv >= kv_lo && kv < kv_hi);
      const T *src = (fresh ? KVf : KVs) + ((size_t)b * a.Nkv + (ok ? kv : 0)) * 2 * a.C +
                     head * AD + lq * 16;
#pragma unroll
      for (int e4 = 0; e4 < 4; ++e4) {
        float fk[4] = {0.f, 0.f, 0.f, 0.f}, fv[4] = {0.f, 0.f, 0.f, 0.f};
        if (ok) {
          load4<T>(src + e4 * 4, fk);
          load4<T>(src + a.C + e4 * 4, fv);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          Ks[lq * 16 + e4 * 4 + e][lr] = fk[e];
          Vs[lr][lq * 16 + e4 * 4 + e] = fv[e];
        }
      }
    }
    __syncthreads();
    float s[4][4] = {};
#pragma unroll 8
    for (int d = 0; d < AD; ++d) {
      float qa[4], kb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) qa[i] = Qs[d][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) kb[j] = Ks[d][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[i][j] = fmaf(qa[i], kb[j], s[i][j]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (kv0 + tx + 16 * j >= k_end)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[i][j] = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float mx = fmaxf(fmaxf(s[i][0], s[i][1]), fmaxf(s[i][2], s[i][3]));
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m_i[i], mx);
      const float corr = exp2f(m_i[i] - m_new);
      float rs = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float pv = exp2f(s[i][j] - m_new);
        Ps[ty + 16 * i][tx + 16 * j] = pv;
        rs += pv;
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
      l_i[i] = l_i[i] * corr + rs;
      m_i[i] = m_new;
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] *= corr;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < AK; ++k) {
      float pa[4], vb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pa[i] = Ps[ty + 16 * i][k];
#pragma unroll
      for (int j = 0; j < 4; ++j) vb[j] = Vs[k][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(pa[i], vb[j], acc[i][j]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int q = q0 + ty + 16 * i;
    if (q >= qend) continue;
    const float inv = 1.f / l_i[i];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      O[((size_t)b * a.Nq + q) * a.C + head * AD + tx + 16 * j] = from_f<T>(acc[i][j] * inv);
  }
}

}  // namespace

cudaError_t launch_conv_simt(const dpp_conv_desc &d, const void *x, const void *stale,
                             const void *w, const float *bias, void *y, cudaStream_t s) {
  const int fresh_halo = (d.halo == DPP_HALO_FRESH || stale == nullptr || stale == x) ? 1 : 0;
  const int zero_halo = d.halo == DPP_HALO_ZERO ? 1 : 0;
  ConvGeom g{d.B, d.H, d.W, d.C_in, d.C_out, d.P, fresh_halo, zero_halo, d.accumulate ? 1 : 0};
  const void *st = fresh_halo ? x : stale;
  const long long M = (long long)d.B * d.H * d.W;
  dim3 grid((unsigned)((M + BM - 1) / BM), (unsigned)((d.C_out + BN - 1) / BN));
  if (d.dtype == DPP_BF16)
    conv_simt_kernel<__nv_bfloat16><<<grid, NT, 0, s>>>(
        (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)st, (const __nv_bfloat16 *)w, bias,
        (__nv_bfloat16 *)y, g);
  else
    conv_simt_kernel<float><<<grid, NT, 0, s>>>((const float *)x, (const float *)st,
                                                (const float *)w, bias, (float *)y, g);
  return cudaGetLastError();
}

cudaError_t launch_gemm_simt(const GemmArgs &g, cudaStream_t s) {
  if (g.geglu) return cudaErrorNotSupported;
  dim3 grid((unsigned)((g.M + BM - 1) / BM), (unsigned)((g.N + BN - 1) / BN));
  if (g.ta == E_F32 && g.tb == E_F32 && g.to == E_F32)
    gemm_simt_kernel<float, float, float><<<grid, NT, 0, s>>>(g);
  else if (g.ta == E_BF16 && g.tb == E_BF16 && g.to == E_F16)
    gemm_simt_kernel<__nv_bfloat16, __nv_bfloat16, __half><<<grid, NT, 0, s>>>(g);
  else if (g.ta == E_F16 && g.tb == E_BF16 && g.to == E_BF16)
    gemm_simt_kernel<__half, __nv_bfloat16, __nv_bfloat16><<<grid, NT, 0, s>>>(g);
  else if (g.ta == E_F16 && g.tb == E_F16 && g.to == E_BF16)
    gemm_simt_kernel<__half, __half, __nv_bfloat16><<<grid, NT, 0, s>>>(g);
  else
    return cudaErrorNotSupported;
  return cudaGetLastError();
}

cudaError_t launch_attn_simt(const AttnArgs &a, cudaStream_t s) {
  const int Np = a.Nq / a.P;
  const int tpb = (Np + AQ - 1) / AQ;
  dim3 grid((unsigned)(tpb * a.P), (unsigned)a.heads, (unsigned)a.B);
  const size_t smem = kAttnSmemFloats * sizeof(float);
  if (a.te == E_F16) {
    cudaFuncSetAttribute(attn_simt_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    attn_simt_kernel<__half><<<grid, NT, smem, s>>>(a);
  } else {
    cudaFuncSetAttribute(attn_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    attn_simt_kernel<float><<<grid, NT, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace dpp

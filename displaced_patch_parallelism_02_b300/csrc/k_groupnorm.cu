// Displaced GroupNorm (DistriGroupNorm, section 归一化层拆分 of the
// DistriFusion developer guide).
//
// Per band p, batch b, group g the statistics combine the band's fresh
// partial sums (sum x, sum x^2) with the stale partials of every other band
// from the previous step; the band's fresh partials are published to
// stats_next (the refresh of the GroupNorm state).  With no stale input
// (the synchronous first step) all bands' fresh partials are combined.
//
// One cooperative launch (every CTA resident at once).  The CTAs form
// kGnGroups groups; group k handles the (batch, band) units k, k + groups,
// ... in order, each of its CTAs owning the same pixel chunk of every unit:
//   A(u)  reads its chunk -- prefetched into shared memory by a bulk copy
//         issued as soon as the previous piece was read, with an L2
//         evict-last hint -- (thread t always holds vector t % (C/VE) of a
//         pixel, so its channels are fixed), reduces per channel and then
//         per group in a fixed order, adds the chunk's partials into the
//         unit's fp64 totals (atomics) and arrives on the unit's counter
//         (one release increment, nothing waited for).  The partials are
//         fp32 values of similar size, so their fp64 sum is exact and does
//         not depend on arrival order;
//   B(u)  after A of the group's next unit (so the group's barrier completes
//         while that unit streams), once the counter shows the whole group
//         (acquire loads; the group's first CTA then publishes the band's
//         stats_next entry): rebuilds the band's statistics
//         (fresh totals plus stale partials, fp64), folds mean/rstd/gamma/
//         beta into one scale and shift per channel and normalises the chunk
//         -- read again one unit after A(u), mostly from L2 (evict-first hints
//         on the re-read and on y).
// y crosses HBM once and x a little more than once (the re-reads that miss
// L2).  While one group waits at its barrier the others stream, and the bulk
// copy of the group's next unit is already in flight.  The synchronous step sums every unit first and then normalises
// (its statistics span all bands of an image), so there x is read twice.
//
// Every wait on a counter is bounded (DPP_ERR_TIMEOUT in the device
// status word, then the CTA stops).  The counters live in the workspace and
// are cleared by a small kernel launched just before.
#include <mutex>

#include "dpp_internal.h"

namespace dpp {
namespace {

constexpr uint64_t kGnWaitLimitNs = 1000000000ull;
constexpr int kGnLag = 1;  // a group's units between a chunk's two reads

__device__ __forceinline__ uint64_t gn_globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t gn_smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// L2 eviction-priority policies for single instructions (the data a pass
// reads twice is kept, what it has finished with goes first).
__device__ __forceinline__ uint64_t gn_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t gn_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Global -> shared bulk copy (16-byte aligned, size a multiple of 16) that
// completes `bytes` transactions on the mbarrier; its lines are kept in L2
// (evict_last) for the second read.
__device__ __forceinline__ void gn_bulk_load(void *dst, const void *src, uint32_t bytes,
                                             uint64_t *bar, uint64_t policy) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(gn_smem_u32(bar)),
               "r"(bytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(gn_smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(gn_smem_u32(bar)), "l"(policy)
      : "memory");
}

// 16-byte global load / store with an L2 eviction policy.
__device__ __forceinline__ uint4 gn_ld_hint(const void *p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}
__device__ __forceinline__ void gn_st_hint(void *p, const uint4 &v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy)
               : "memory");
}

// Bounded wait for the given phase parity of a shared-memory mbarrier.
__device__ __forceinline__ bool gn_bar_wait(uint64_t *bar, uint32_t parity, int *status) {
  const uint64_t t0 = gn_globaltimer();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(gn_smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if (gn_globaltimer() - t0 > kGnWaitLimitNs) {
      if (status) atomicExch(status, (int)DPP_ERR_TIMEOUT);
      return false;
    }
  }
}

// The activation that may follow the affine (DPP_ACT_SILU: x * sigmoid(x),
// the GroupNorm -> SiLU of a ResNet block).  The exponent is clamped at 80 so
// that 1 + e stays far below 2^126, the range of the fast divide; below
// x = -80 both the clamped and the exact value are under 1e-33 in size.
__device__ __forceinline__ float gn_act(float x, int act) {
  return act == DPP_ACT_SILU ? __fdividef(x, 1.f + __expf(fminf(-x, 80.f))) : x;
}

template <typename T>
struct Vec16;

template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void cvt(const uint4 &v, float f[4]) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  __device__ static void load(const float *p, float f[4]) {
    const float4 v = *reinterpret_cast<const float4 *>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
  __device__ static void store(float *p, const float f[4]) {
    *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
  __device__ static uint4 pack(const float f[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void cvt(const uint4 &v, float f[8]) {  // bf16 -> fp32 is a 16-bit shift
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
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
    *reinterpret_cast<uint4 *>(p) = pack(f);
  }
  __device__ static uint4 pack(const float f[8]) {
    uint4 v;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return v;
  }
};

struct GnGeom {
  int B, H, W, C, G, P;
  int units;  // B * P; unit u = b * P + p
  int npix;   // pixels of one unit
  int ppc;    // pixels per CTA chunk
  int groups; // CTA groups; group k handles units k, k + groups, ...
  int sms;    // SM count when the grid is whole waves of it, else 0
  int R;      // pixel rows in flight per CTA (threads = R * C / VE)
  int sync;   // 1: no stale statistics
  int band_local;  // 1: each band's statistics over its own rows only
  int act;    // DPP_ACT_* applied after the affine
  int ppp;    // pixels per prefetched piece (the shared-memory buffer)
};

struct GnWs {
  unsigned *arrive;         // per unit: CTAs of its group that have added their partials
  double *tot;              // [units][G][2] fresh totals
};


// Bounded wait by thread 0 until every unit in [v0, v1] counts `target`
// arrivals (acquire loads, so the units' totals are visible afterwards); the
// result is shared through `flag` (1 = proceed).
__device__ __forceinline__ bool gn_wait_units(const unsigned *arrive, int v0, int v1,
                                              unsigned target, int *flag, int *status) {
  if (threadIdx.x == 0) {
    int ok = 1;
    for (int v = v0; v <= v1 && ok; ++v) {
      const uint64_t t0 = gn_globaltimer();
      while (true) {
        unsigned n;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(n) : "l"(arrive + v) : "memory");
        if (n >= target) break;
        if (gn_globaltimer() - t0 > kGnWaitLimitNs) {
          ok = 0;
          if (status) atomicExch(status, (int)DPP_ERR_TIMEOUT);
          break;
        }
      }
    }
    *flag = ok;
  }
  __syncthreads();
  return *flag != 0;
}

template <typename T>
__global__ void __launch_bounds__(1024)
gn_fused_kernel(const T *x, T *y, GnGeom g, const float *__restrict__ stats_prev,
                float *__restrict__ stats_next, const float *__restrict__ gamma,
                const float *__restrict__ beta, float eps, GnWs ws, int *status) {
  constexpr int VE = Vec16<T>::N;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ int s_flag;
  __shared__ __align__(8) uint64_t s_bar;  // completion of the prefetched piece
  const int VPP = g.C / VE, R = g.R;
  T *buf = reinterpret_cast<T *>(smem_raw);  // one piece: ppp pixels x C
  float *sm = reinterpret_cast<float *>(smem_raw + (size_t)g.ppp * g.C * sizeof(T));
  float *s1 = sm, *s2 = sm + R * g.C;  // [R][C] per-row channel sums (also the reduction scratch)
  float *c1 = sm + 2 * R * g.C, *c2 = c1 + g.C;
  float *mean_s = c2 + g.C, *rstd_s = mean_s + g.G;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int v = tid % VPP, r = tid / VPP;
  const bool active = r < R;
  const int Hp = g.H / g.P;
  const int cg = g.C / g.G;
  // The group's CTAs split every unit.  CTAs c and c + sms usually share an
  // SM; when the grid is whole waves of the SM count, each wave's groups are
  // rotated by one so that an SM hosts CTAs of different groups (one group
  // waiting at its barrier then leaves the SM to the other).
  const int c = blockIdx.x;
  int grp, rank;
  if (g.sms > 0 && g.sms % g.groups == 0) {
    const int wave = c / g.sms, idx = c % g.sms;
    grp = (idx + wave) % g.groups;
    rank = wave * (g.sms / g.groups) + idx / g.groups;
  } else {
    grp = c % g.groups;
    rank = c / g.groups;
  }
  const int gsize = gridDim.x / g.groups;
  const int j0 = rank * g.ppc;
  const int j1 = min(j0 + g.ppc, g.npix);

  auto unit_base = [&](int u) -> size_t {  // first pixel of unit u
    const int b = u / g.P, p = u % g.P;
    return ((size_t)b * g.H + (size_t)p * Hp) * g.W;
  };
  const uint64_t keep = gn_policy_evict_last(), drop = gn_policy_evict_first();
  // thread 0 starts the bulk copy of piece pc of this CTA's chunk of unit u
  auto prefetch = [&](int u, int pc) {
    const int pj0 = j0 + pc * g.ppp, pj1 = min(pj0 + g.ppp, j1);
    gn_bulk_load(buf, x + (unit_base(u) + pj0) * g.C, (uint32_t)((pj1 - pj0) * g.C * sizeof(T)),
                 &s_bar, keep);
  };
  const int pieces = j1 > j0 ? (j1 - j0 + g.ppp - 1) / g.ppp : 0;  // per unit
  uint32_t bar_phase = 0;
  bool pending = pieces > 0 && grp < g.units;  // a copy issued and not yet waited for
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(gn_smem_u32(&s_bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (pending) prefetch(grp, 0);
  }
  __syncthreads();

  // ---- A(u): chunk partials, arrival, and (last CTA) the unit totals
  auto pass_a = [&](int u) -> bool {
    float a1[VE], a2[VE];
#pragma unroll
    for (int e = 0; e < VE; ++e) a1[e] = a2[e] = 0.f;
    for (int pc = 0; pc < pieces; ++pc) {
      const bool landed = gn_bar_wait(&s_bar, bar_phase, status);
      if (!__syncthreads_and(landed)) return false;  // `pending` stays set: drained at exit
      bar_phase ^= 1u;
      pending = false;
      const int pj0 = j0 + pc * g.ppp, pj1 = min(pj0 + g.ppp, j1);
      if (active)
        for (int j = pj0 + r; j < pj1; j += R) {
          float f[VE];
          Vec16<T>::cvt(*reinterpret_cast<const uint4 *>(buf + (size_t)(j - pj0) * g.C + v * VE),
                        f);
#pragma unroll
          for (int e = 0; e < VE; ++e) {
            a1[e] += f[e];
            a2[e] = fmaf(f[e], f[e], a2[e]);
          }
        }
      __syncthreads();  // the buffer is free: start the next piece's copy
      const bool more = pc + 1 < pieces || u + g.groups < g.units;  // the group's next unit
      if (more && tid == 0) {
        if (pc + 1 < pieces)
          prefetch(u, pc + 1);
        else
          prefetch(u + g.groups, 0);
      }
      pending = more;
    }
    if (active) {  // 16-byte stores: a quarter of the bank conflicts of scalar ones
#pragma unroll
      for (int e = 0; e < VE; e += 4) {
        *reinterpret_cast<float4 *>(s1 + r * g.C + v * VE + e) =
            make_float4(a1[e], a1[e + 1], a1[e + 2], a1[e + 3]);
        *reinterpret_cast<float4 *>(s2 + r * g.C + v * VE + e) =
            make_float4(a2[e], a2[e + 1], a2[e + 2], a2[e + 3]);
      }
    }
    __syncthreads();
    for (int ch = tid; ch < g.C; ch += nthr) {
      float t1 = 0.f, t2 = 0.f;
      for (int rr = 0; rr < R; ++rr) {
        t1 += s1[rr * g.C + ch];
        t2 += s2[rr * g.C + ch];
      }
      c1[ch] = t1;
      c2[ch] = t2;
    }
    __syncthreads();
    double *tot = ws.tot + (size_t)u * g.G * 2;
    for (int gg = tid; gg < g.G; gg += nthr) {
      float t1 = 0.f, t2 = 0.f;
      for (int k = 0; k < cg; ++k) {
        t1 += c1[gg * cg + k];
        t2 += c2[gg * cg + k];
      }
      atomicAdd(tot + gg * 2, (double)t1);
      atomicAdd(tot + gg * 2 + 1, (double)t2);
    }
    // arrive: the barrier orders every thread's additions before thread 0's
    // release increment (fire and forget: nothing here waits for L2)
    __syncthreads();
    if (tid == 0)
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ws.arrive + u) : "memory");
    return true;
  };

  // ---- B(u): band statistics, then normalise the chunk (second read: L2)
  auto pass_b = [&](int u) -> bool {
    const int b = u / g.P, p = u % g.P;
    const bool whole = g.sync && !g.band_local;  // statistics of every band of the image
    const int first = whole ? b * g.P : u, last = whole ? b * g.P + g.P - 1 : u;
    if (!gn_wait_units(ws.arrive, first, last, (unsigned)gsize, &s_flag, status)) return false;
    if (rank == 0)  // the band's fresh partials: the refresh of the GroupNorm state
      for (int i = tid; i < 2 * g.G; i += nthr)
        stats_next[((size_t)p * g.B + b) * 2 * g.G + i] =
            (float)__ldcg(ws.tot + (size_t)u * 2 * g.G + i);
    for (int gg = tid; gg < g.G; gg += nthr) {
      double t1 = 0.0, t2 = 0.0;
      if (g.band_local) {
        const double *tu = ws.tot + ((size_t)u * g.G + gg) * 2;
        t1 = __ldcg(tu);
        t2 = __ldcg(tu + 1);
      } else if (g.sync) {
        for (int q = 0; q < g.P; ++q) {
          const double *tq = ws.tot + ((size_t)(b * g.P + q) * g.G + gg) * 2;
          t1 += __ldcg(tq);
          t2 += __ldcg(tq + 1);
        }
      } else {
        const double *tu = ws.tot + ((size_t)u * g.G + gg) * 2;
        t1 = __ldcg(tu);
        t2 = __ldcg(tu + 1);
        for (int q = 0; q < g.P; ++q) {
          if (q == p) continue;
          const float *sq = stats_prev + (((size_t)q * g.B + b) * g.G + gg) * 2;
          t1 += sq[0];
          t2 += sq[1];
        }
      }
      const double n = (double)(g.band_local ? Hp : g.H) * g.W * cg;
      const double mean = t1 / n;
      const double var = fmax(t2 / n - mean * mean, 0.0);
      mean_s[gg] = (float)mean;
      rstd_s[gg] = (float)(1.0 / sqrt(var + (double)eps));
    }
    __syncthreads();
    if (active) {
      float sc[VE], sh[VE];
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        const int ch = v * VE + e, gg = ch / cg;
        const float a = rstd_s[gg] * (gamma ? gamma[ch] : 1.f);
        sc[e] = a;
        sh[e] = (beta ? beta[ch] : 0.f) - mean_s[gg] * a;
      }
      const size_t base = unit_base(u);
      for (int j = j0 + r; j < j1; j += 4 * R) {  // four rows per iteration
        uint4 raw[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          raw[k] = j + k * R < j1 ? gn_ld_hint(x + (base + j + k * R) * g.C + v * VE, drop)
                                  : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (j + k * R < j1) {
            float f[VE];
            Vec16<T>::cvt(raw[k], f);
#pragma unroll
            for (int e = 0; e < VE; ++e) f[e] = gn_act(fmaf(f[e], sc[e], sh[e]), g.act);
            gn_st_hint(y + (base + j + k * R) * g.C + v * VE, Vec16<T>::pack(f), drop);
          }
        }
      }
    }
    __syncthreads();  // mean_s / rstd_s are rewritten by the next B
    return true;
  };

  bool ok = true;
  if (!g.sync || g.band_local) {
    // the group's k-th unit is normalised after its (k + kGnLag)-th is summed:
    // the chunk was read moments ago and is still in L2, and the lag lets the
    // group's barrier complete while the next unit streams
    const int n = grp < g.units ? (g.units - grp + g.groups - 1) / g.groups : 0;
    for (int k = 0; ok && k < n; ++k) {
      ok = pass_a(grp + k * g.groups);
      if (ok && k >= kGnLag) ok = pass_b(grp + (k - kGnLag) * g.groups);
    }
    for (int k = n - kGnLag < 0 ? 0 : n - kGnLag; ok && k < n; ++k) ok = pass_b(grp + k * g.groups);
  } else {
    // the synchronous step needs every band of an image first
    for (int u = grp; ok && u < g.units; u += g.groups) ok = pass_a(u);
    for (int u = grp; ok && u < g.units; u += g.groups) ok = pass_b(u);
  }
  // A CTA that gave up may still have a bulk copy in flight into its shared
  // memory: wait for it (bounded) before the CTA exits.
  if (pending) gn_bar_wait(&s_bar, bar_phase, nullptr);
}

__global__ void gn_reset_kernel(unsigned *counters, int n_cnt, double *tot, int n_tot) {
  for (int i = threadIdx.x; i < n_cnt; i += blockDim.x) counters[i] = 0u;
  for (int i = threadIdx.x; i < n_tot; i += blockDim.x) tot[i] = 0.0;
}

int gn_vec(const dpp_gn_desc &d) { return d.dtype == DPP_BF16 ? 8 : 4; }

int gn_rows(const dpp_gn_desc &d) {
  const int VPP = d.C / gn_vec(d);
  return VPP <= 512 ? 512 / VPP : 1;
}

size_t gn_pixel_bytes(const dpp_gn_desc &d) { return (size_t)d.C * (d.dtype == DPP_BF16 ? 2 : 4); }

// The prefetch buffer holds up to 64 KB of whole pixels.
constexpr size_t kGnBufBytes = 64 * 1024;
constexpr int kGnGroups = 4;
int gn_buf_pixels(const dpp_gn_desc &d) {
  const size_t n = kGnBufBytes / gn_pixel_bytes(d);
  return n < 1 ? 1 : (int)n;
}

size_t gn_smem(const dpp_gn_desc &d) {
  return (size_t)gn_buf_pixels(d) * gn_pixel_bytes(d) +
         (size_t)(2 * gn_rows(d) * d.C + 2 * d.C + 2 * d.G) * sizeof(float);
}

// workspace carve-up: counters, then unit totals (256-byte aligned)
size_t gn_layout(const dpp_gn_desc &d, void *base, GnWs *w) {
  const size_t U = (size_t)d.B * d.P;
  const size_t n_cnt = align_up(U * sizeof(unsigned), 256);
  const size_t n_tot = align_up(U * d.G * 2 * sizeof(double), 256);
  if (w) {
    char *c = reinterpret_cast<char *>(base);
    w->arrive = reinterpret_cast<unsigned *>(c);
    w->tot = reinterpret_cast<double *>(c + n_cnt);
  }
  return n_cnt + n_tot;
}

template <typename T>
cudaError_t run_gn(const dpp_gn_desc &d, const void *x, const float *stats_prev,
                   float *stats_next, const float *gamma, const float *beta, void *y, void *ws,
                   int *status, cudaStream_t s) {
  GnWs w;
  gn_layout(d, ws, &w);

  const int VPP = d.C / gn_vec(d), R = gn_rows(d);
  const int threads = R * VPP;
  const size_t smem = gn_smem(d);
  auto k = gn_fused_kernel<T>;
  cudaError_t e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  {
    // the attribute and the occupancy query cost host time on every call:
    // keep them per (device, block shape, shared memory)
    struct Entry {
      int dev, threads;
      size_t smem;
      int sms, per_sm;
    };
    static std::mutex mu;
    static Entry cache[16];
    static int n_cache = 0;
    static size_t attr_max[64] = {};  // the kernel's dynamic shared-memory limit, per device
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (smem > attr_max[dev]) {  // the limit only ever grows, so it covers every shape seen
      if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
          cudaSuccess)
        return e;
      attr_max[dev] = smem;
    }
    int hit = -1;
    for (int i = 0; i < n_cache; ++i)
      if (cache[i].dev == dev && cache[i].threads == threads && cache[i].smem == smem) hit = i;
    if (hit >= 0) {
      sms = cache[hit].sms;
      per_sm = cache[hit].per_sm;
    } else {
      if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
      if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem)) !=
          cudaSuccess)
        return e;
      if (n_cache < 16) cache[n_cache++] = Entry{dev, threads, smem, sms, per_sm};
    }
  }
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  GnGeom g;
  g.B = d.B; g.H = d.H; g.W = d.W; g.C = d.C; g.G = d.G; g.P = d.P;
  g.units = d.B * d.P;
  g.npix = (d.H / d.P) * d.W;
  g.R = R;
  g.sync = stats_prev == nullptr ? 1 : 0;
  g.band_local = d.band_local ? 1 : 0;
  g.act = d.act;
  long long grid = (long long)per_sm * sms;
  if (grid > kGnMaxGrid) grid = kGnMaxGrid;
  // CTA groups work on different units at the same time, so one group's
  // barrier overlaps the others' streaming; each group takes whole units
  g.groups = g.units < kGnGroups ? g.units : kGnGroups;
  long long gsize = grid / g.groups;
  const long long by_pixels = (g.npix + R - 1) / R;  // at least R pixels per CTA
  if (gsize > by_pixels) gsize = by_pixels;
  if (gsize < 1) gsize = 1;
  grid = gsize * g.groups;
  g.sms = grid % sms == 0 ? sms : 0;
  g.ppc = (int)((g.npix + gsize - 1) / gsize);
  g.ppp = g.ppc < gn_buf_pixels(d) ? g.ppc : gn_buf_pixels(d);
  const int n_cnt = g.units;
  gn_reset_kernel<<<1, 256, 0, s>>>(w.arrive, n_cnt, w.tot, g.units * 2 * d.G);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const T *xp = reinterpret_cast<const T *>(x);
  T *yp = reinterpret_cast<T *>(y);
  float eps = d.eps;
  void *args[] = {(void *)&xp, (void *)&yp, (void *)&g, (void *)&stats_prev,
                  (void *)&stats_next, (void *)&gamma, (void *)&beta, (void *)&eps,
                  (void *)&w, (void *)&status};
  return cudaLaunchCooperativeKernel((const void *)k, dim3((unsigned)grid), dim3(threads), args,
                                     smem, s);
}

// Self-test of the bounded wait above: one thread waits for a unit counter
// that nothing advances; after the wait limit it records DPP_ERR_TIMEOUT in
// the status word and the kernel returns.
__global__ void gn_wait_selftest_kernel(const unsigned *counter, int *status) {
  __shared__ int flag;
  gn_wait_units(counter, 0, 0, 1u, &flag, status);
}

}  // namespace

cudaError_t launch_wait_selftest_counter(const unsigned *counter, cudaStream_t s) {
  gn_wait_selftest_kernel<<<1, 32, 0, s>>>(counter, device_status_ptr());
  return cudaGetLastError();
}

size_t gn_workspace(const dpp_gn_desc &d) { return gn_layout(d, nullptr, nullptr); }

cudaError_t launch_groupnorm(const dpp_gn_desc &d, const void *x, const float *stats_prev,
                             float *stats_next, const float *gamma, const float *beta,
                             void *y, void *ws, cudaStream_t s) {
  int *status = device_status_ptr();
  if (d.dtype == DPP_BF16)
    return run_gn<__nv_bfloat16>(d, x, stats_prev, stats_next, gamma, beta, y, ws, status, s);
  return run_gn<float>(d, x, stats_prev, stats_next, gamma, beta, y, ws, status, s);
}

}  // namespace dpp

// ---------------------------------------------------------------------------
// GroupNorm when the producing conv has already summed each band
// (dpp_conv3x3_gn): one streaming pass.  A CTA takes one chunk of one
// (batch, band) unit, rebuilds the band's statistics (its fresh sums plus
// the other bands' stale partials, fp64), folds mean/rstd/gamma/beta into a
// scale and shift per channel in shared memory and normalises its chunk with
// 16-byte loads and stores, four in flight per thread (each thread always
// holds the same channel vector, so its scale and shift stay in registers).
// The first chunk of each unit publishes the band's fresh sums to
// stats_next.
namespace dpp {
namespace {

// Band p's statistics of image b and group g: its fresh sums gn_sums[p] plus
// the other bands' stale partials stats_prev[q] (every band's fresh sums in
// the synchronous step, stats_prev == NULL; the band's own alone when
// band_local), in fp64; mean and 1/sqrt(var + eps) rounded to fp32.
__device__ __forceinline__ void gn_band_stats(const double *__restrict__ gn_sums,
                                              const float *__restrict__ stats_prev, int B, int H,
                                              int W, int cg, int G, int P, int band_local, int p,
                                              int b, int g, float eps, float &mean_f,
                                              float &rstd_f) {
  const double *fr = gn_sums + (((size_t)p * B + b) * G + g) * 2;
  double t1 = fr[0], t2 = fr[1];
  for (int q = 0; q < P && !band_local; ++q) {
    if (q == p) continue;
    if (stats_prev) {
      const float *sq = stats_prev + (((size_t)q * B + b) * G + g) * 2;
      t1 += sq[0];
      t2 += sq[1];
    } else {
      const double *fq = gn_sums + (((size_t)q * B + b) * G + g) * 2;
      t1 += fq[0];
      t2 += fq[1];
    }
  }
  const double n = (double)(band_local ? H / P : H) * W * cg;
  const double mean = t1 / n;
  const double var = fmax(t2 / n - mean * mean, 0.0);
  mean_f = (float)mean;
  rstd_f = (float)(1.0 / sqrt(var + (double)eps));
}

template <typename T>
__global__ void __launch_bounds__(512)
gn_apply_kernel(const T *x, T *y, int B, int H, int W, int C, int G, int P, int ppc, int band_local,
                int act, const double *__restrict__ gn_sums, const float *__restrict__ stats_prev,
                float *__restrict__ stats_next, const float *__restrict__ gamma,
                const float *__restrict__ beta, float eps) {
  constexpr int VE = Vec16<T>::N;
  __shared__ float mean_s[1024], rstd_s[1024];  // per group (G <= C/VE*VE <= 8192 checked on host)
  const int unit = blockIdx.y, b = unit / P, p = unit % P;
  const int cg = C / G, Hp = H / P;
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    gn_band_stats(gn_sums, stats_prev, B, H, W, cg, G, P, band_local, p, b, g, eps, mean_s[g],
                  rstd_s[g]);
    if (blockIdx.x == 0) {
      const double *fr = gn_sums + (((size_t)p * B + b) * G + g) * 2;
      float *sn = stats_next + (((size_t)p * B + b) * G + g) * 2;
      sn[0] = (float)fr[0];
      sn[1] = (float)fr[1];
    }
  }
  __syncthreads();
  // thread t always holds channel vector t % (C/VE): its scale and shift stay
  // in registers; R pixel rows per pass, four passes' loads in flight
  const int VPP = C / VE, R = blockDim.x / VPP;
  const int v = threadIdx.x % VPP, r = threadIdx.x / VPP;
  if (r >= R) return;
  float sc[VE], sh[VE];
#pragma unroll
  for (int e = 0; e < VE; ++e) {
    const int ch = v * VE + e, g = ch / cg;
    const float a = rstd_s[g] * (gamma ? gamma[ch] : 1.f);
    sc[e] = a;
    sh[e] = (beta ? beta[ch] : 0.f) - mean_s[g] * a;
  }
  const int npix = Hp * W;
  const int j0 = blockIdx.x * ppc, j1 = min(j0 + ppc, npix);
  const size_t base = ((size_t)b * H + (size_t)p * Hp) * W;
  const uint64_t drop = gn_policy_evict_first();
  for (int j = j0 + r; j < j1; j += 4 * R) {
    uint4 raw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      raw[k] = j + k * R < j1 ? gn_ld_hint(x + (base + j + k * R) * C + v * VE, drop)
                              : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (j + k * R < j1) {
        float f[VE];
        Vec16<T>::cvt(raw[k], f);
#pragma unroll
        for (int e = 0; e < VE; ++e) f[e] = gn_act(fmaf(f[e], sc[e], sh[e]), act);
        gn_st_hint(y + (base + j + k * R) * C + v * VE, Vec16<T>::pack(f), drop);
      }
    }
  }
}

// The band sums of x alone (what dpp_conv3x3_gn's epilogue produces for its
// output), for a GroupNorm whose input no conv summed: one read of x.  A CTA
// takes one chunk of one (batch, band) unit; thread t always holds channel
// vector t % (C/VE) and adds its pixels' values and squares in fp32.  The
// CTA then folds them in a fixed order -- per channel over its pixel rows,
// per group over its channels -- and adds each group's fp32 sums into the
// fp64 totals (zeroed by the launcher).  fp32 values of similar size add
// exactly in fp64, so the totals do not depend on the order the CTAs' atomics
// land in: the sums are bit-reproducible.
template <typename T>
__global__ void __launch_bounds__(512)
gn_sums_kernel(const T *x, int B, int H, int W, int C, int G, int P, int ppc,
               double *__restrict__ gn_sums) {
  constexpr int VE = Vec16<T>::N;
  __shared__ float part[2][512 * VE];  // [R][C] per-thread channel sums (R * C = blockDim * VE)
  const int unit = blockIdx.y, b = unit / P, p = unit % P;
  const int cg = C / G, Hp = H / P;
  const int VPP = C / VE, R = blockDim.x / VPP;
  const int v = threadIdx.x % VPP, r = threadIdx.x / VPP;
  if (r < R) {
    float s1[VE], s2[VE];
#pragma unroll
    for (int e = 0; e < VE; ++e) s1[e] = s2[e] = 0.f;
    const int npix = Hp * W;
    const int j0 = blockIdx.x * ppc, j1 = min(j0 + ppc, npix);
    const size_t base = ((size_t)b * H + (size_t)p * Hp) * W;
    for (int j = j0 + r; j < j1; j += 4 * R) {
      uint4 raw[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        raw[k] = j + k * R < j1
                     ? *reinterpret_cast<const uint4 *>(x + (base + j + k * R) * C + v * VE)
                     : make_uint4(0u, 0u, 0u, 0u);  // zeros add nothing
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float f[VE];
        Vec16<T>::cvt(raw[k], f);
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          s1[e] += f[e];
          s2[e] = fmaf(f[e], f[e], s2[e]);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      part[0][r * C + v * VE + e] = s1[e];
      part[1][r * C + v * VE + e] = s2[e];
    }
  }
  __syncthreads();
  for (int ch = threadIdx.x; ch < C; ch += blockDim.x) {  // column ch: this thread's alone
    float t1 = 0.f, t2 = 0.f;
    for (int k = 0; k < R; ++k) {
      t1 += part[0][k * C + ch];
      t2 += part[1][k * C + ch];
    }
    part[0][ch] = t1;
    part[1][ch] = t2;
  }
  __syncthreads();
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    float t1 = 0.f, t2 = 0.f;
    for (int ch = g * cg; ch < (g + 1) * cg; ++ch) {
      t1 += part[0][ch];
      t2 += part[1][ch];
    }
    double *t = gn_sums + (((size_t)p * B + b) * G + g) * 2;
    atomicAdd(t, (double)t1);
    atomicAdd(t + 1, (double)t2);
  }
}

// The statistics half of a displaced GroupNorm as a per-channel affine of
// each band: affine[p][b][c] = (a, s) with a = rstd * gamma[c] and
// s = beta[c] - mean * a (the scale and shift gn_apply_kernel applies, in
// the same operations), and band p's fresh sums published to stats_next[p].
// One CTA per (batch, band) unit.
__global__ void __launch_bounds__(256)
gn_affine_kernel(int B, int H, int W, int C, int G, int P, int band_local,
                 const double *__restrict__ gn_sums, const float *__restrict__ stats_prev,
                 float *__restrict__ stats_next, const float *__restrict__ gamma,
                 const float *__restrict__ beta, float eps, float *__restrict__ affine) {
  __shared__ float mean_s[1024], rstd_s[1024];
  const int unit = blockIdx.x, b = unit / P, p = unit % P;
  const int cg = C / G;
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    gn_band_stats(gn_sums, stats_prev, B, H, W, cg, G, P, band_local, p, b, g, eps, mean_s[g],
                  rstd_s[g]);
    if (stats_next) {
      const double *fr = gn_sums + (((size_t)p * B + b) * G + g) * 2;
      float *sn = stats_next + (((size_t)p * B + b) * G + g) * 2;
      sn[0] = (float)fr[0];
      sn[1] = (float)fr[1];
    }
  }
  __syncthreads();
  float2 *out = reinterpret_cast<float2 *>(affine) + ((size_t)p * B + b) * C;
  for (int ch = threadIdx.x; ch < C; ch += blockDim.x) {
    const int g = ch / cg;
    const float a = rstd_s[g] * (gamma ? gamma[ch] : 1.f);
    out[ch] = make_float2(a, (beta ? beta[ch] : 0.f) - mean_s[g] * a);
  }
}

}  // namespace

cudaError_t launch_groupnorm_apply(const dpp_gn_desc &d, const void *x, const float *stats_prev,
                                   const double *gn_sums, float *stats_next, const float *gamma,
                                   const float *beta, void *y, cudaStream_t s) {
  if (d.G > 1024) return cudaErrorNotSupported;
  const int VPP = d.C / gn_vec(d), R = gn_rows(d);
  const int threads = R * VPP;
  const int units = d.B * d.P;
  const int npix = (d.H / d.P) * d.W;
  int chunks = (4 * 148 + units - 1) / units;  // about four CTAs per SM in all
  const int max_chunks = (npix + 4 * R - 1) / (4 * R);  // at least four passes per CTA
  if (chunks > max_chunks) chunks = max_chunks;
  if (chunks < 1) chunks = 1;
  const int ppc = (npix + chunks - 1) / chunks;
  dim3 grid((unsigned)chunks, (unsigned)units);
  if (d.dtype == DPP_BF16)
    gn_apply_kernel<__nv_bfloat16><<<grid, threads, 0, s>>>(
        (const __nv_bfloat16 *)x, (__nv_bfloat16 *)y, d.B, d.H, d.W, d.C, d.G, d.P, ppc,
        d.band_local ? 1 : 0, d.act, gn_sums, stats_prev, stats_next, gamma, beta, d.eps);
  else
    gn_apply_kernel<float><<<grid, threads, 0, s>>>(
        (const float *)x, (float *)y, d.B, d.H, d.W, d.C, d.G, d.P, ppc, d.band_local ? 1 : 0,
        d.act, gn_sums, stats_prev,
        stats_next, gamma, beta, d.eps);
  return cudaGetLastError();
}


cudaError_t launch_groupnorm_sums(const dpp_gn_desc &d, const void *x, double *gn_sums,
                                  cudaStream_t s) {
  // the kernel's per-thread sums fill [R][C] <= 512 x VE floats of shared memory
  if (d.G > 1024 || d.C / gn_vec(d) > 512) return cudaErrorNotSupported;
  const size_t n = (size_t)d.P * d.B * d.G * 2;
  cudaError_t e = launch_zero_f64(gn_sums, n, s);
  if (e != cudaSuccess) return e;
  const int VPP = d.C / gn_vec(d), R = gn_rows(d);
  const int threads = R * VPP;
  const int units = d.B * d.P;
  const int npix = (d.H / d.P) * d.W;
  int chunks = (4 * 148 + units - 1) / units;
  const int max_chunks = (npix + 4 * R - 1) / (4 * R);
  if (chunks > max_chunks) chunks = max_chunks;
  if (chunks < 1) chunks = 1;
  const int ppc = (npix + chunks - 1) / chunks;
  dim3 grid((unsigned)chunks, (unsigned)units);
  if (d.dtype == DPP_BF16)
    gn_sums_kernel<__nv_bfloat16><<<grid, threads, 0, s>>>(
        (const __nv_bfloat16 *)x, d.B, d.H, d.W, d.C, d.G, d.P, ppc, gn_sums);
  else
    gn_sums_kernel<float><<<grid, threads, 0, s>>>((const float *)x, d.B, d.H, d.W, d.C, d.G,
                                                   d.P, ppc, gn_sums);
  return cudaGetLastError();
}

cudaError_t launch_groupnorm_affine(const dpp_gn_desc &d, const double *gn_sums,
                                    const float *stats_prev, float *stats_next,
                                    const float *gamma, const float *beta, float *affine,
                                    cudaStream_t s) {
  if (d.G > 1024) return cudaErrorNotSupported;
  gn_affine_kernel<<<(unsigned)(d.B * d.P), 256, 0, s>>>(
      d.B, d.H, d.W, d.C, d.G, d.P, d.band_local ? 1 : 0, gn_sums, stats_prev, stats_next, gamma,
      beta, d.eps, affine);
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
  // Every call clears the unit counters at the start of the array before
  // its main kernel runs, and writes each partial sum before reading it, so
  // the previous call's contents never leak into this one.
  return launch_groupnorm(d, x, stats_prev, stats_next, gamma, beta, y, scratch, s);
}

}  // namespace dpp

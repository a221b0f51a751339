// Displaced 3x3 conv (DistriConv2dPP, section 卷积层拆分 of the DistriFusion
// developer guide) as an implicit GEMM on tcgen05.
//
//   Y[b,h,w,:] = bias + sum_{dy,dx} W_tap[:, :] . Z_p[b, h+dy-1, w+dx-1, :]
//
// GEMM view: M = output pixels, N = C_out, K = 9 taps x C_in.  An M tile is
// 128 consecutive pixels of ONE image row (b, h, w0..w0+127), so for each tap
// the A tile is a single TMA box of the input row h+dy-1 shifted by dx-1
// pixels.  That row is either in the band that owns h (fresh input) or in a
// neighbouring band (stale input, the halo); the producer picks the tensor
// map per tap.  Rows -1 and H and columns -1 and W fall outside the tensor
// and TMA fills them with zeros: the image padding costs nothing.
//
// Persistent, warp-specialised, one CTA per SM (the GEMM kernel's layout):
//   warps 0, 6  TMA producers, each owning alternate stages (converged
//               warps; an elected lane issues each copy): A box {64 ch,
//               128 px} from the fresh or stale map, B box {64 ch, 1 tap,
//               BN out-ch} of the weights [C_out][3][3][C_in], 128-byte
//               swizzle, STAGES-deep ring;
//   warp 1      TMEM owner and tcgen05.mma issuer (converged warp, one
//               elected lane per instruction)
//               (M 128, N BN, K 16), two accumulators 256 columns apart;
//   warps 2..5  epilogue: tcgen05.ld, + bias (+ the residual already in y
//               when accumulating), bf16, 16-byte stores; with
//               STATS also the per-group sums of the stored values (for a
//               GroupNorm of this output), reduced over the warp's 32 pixels
//               and added into fp64 totals per (band, image, group).
//
// conv_norm_tc_kernel (further down) is the same conv reading its input
// through a GroupNorm affine and SiLU applied as the input is loaded
// (dpp_conv3x3_norm), with its K loop organised around input-row strips.
#include "tc_common.cuh"

namespace dpp {
namespace {

using namespace tc;

struct ConvTcParams {
  int B, H, W, Cin, Cout, P;
  int nseg;      // 128-pixel segments per image row
  int cblocks;   // 64-channel blocks of C_in
  int m_tiles, n_tiles;
  int use_stale; // 0: every input row comes from the fresh map
  int zero_halo; // 1: rows outside the band read as zero (naive patches)
  int accumulate; // 1: y += result (the residual already in y is read first)
  const float *bias;
  __nv_bfloat16 *y;
  int *status;
  double *gn_sums;  // [P][B][G][2] (sum y, sum y^2) per band, image and group; may be null
  int G;            // groups (channels C_out / G each)
  // normalised input (conv_norm_tc_kernel): the conv reads act(x * a + s)
  const float *affine;       // [P][B][C_in] (a, s) of this step, per band of the row read
  const float *affine_prev;  // the previous step's, for halo rows read from the stale input
  int act;                   // DPP_ACT_*
};

// warps 0 and 6 produce (alternate stages), warp 1 issues MMAs, warps 2..5
// convert: one thread issuing every copy could not keep up with 320 MMA
// cycles per stage, and a second issuing warp nearly doubles the copy rate
constexpr int kProducers = 2;
constexpr int kThreads = 192 + 32 * (kProducers - 1);
constexpr int BM = 128, BK = 64;

// Butterfly reduce-scatter over the warp: lane l ends with the sum over all
// 32 lanes of a[l] (31 shuffles; a[] is clobbered).
__device__ __forceinline__ float warp_reduce_scatter32(float (&a)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 16; k >= 1; k >>= 1) {
    const bool up = (lane & k) != 0;
#pragma unroll
    for (int i = 0; i < k; ++i) {
      const float send = up ? a[i] : a[i + k];
      const float keep = up ? a[i + k] : a[i];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, k);
    }
  }
  return a[0];
}

// Epilogue warps (q = warp % 4 owns TMEM lanes / tile pixels 32q..32q+31):
// per finished tile, tcgen05.ld of the accumulator, + bias (+ the residual
// already in y when accumulating), bf16, 16-byte stores; with STATS also the
// per-group sums of the stored values, reduced over the warp's 32 pixels and
// added into fp64 totals per (band, image, group).
template <int BN, bool STATS>
__device__ __forceinline__ void conv_epilogue(const ConvTcParams &p, uint32_t tmem,
                                              uint64_t *tfull, uint64_t *tempty,
                                              volatile int *abort_flag, float *chs, int q,
                                              int lane) {
  const int tiles = p.m_tiles * p.n_tiles;
  const int Hp = p.H / p.P;
  const int px = q * 32 + lane;
  int it = 0;
  for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
    const int acc = it & 1;
    const uint32_t acc_phase = (it >> 1) & 1;
    if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status)) break;
    tc_fence_after();
    const int mt = t / p.n_tiles, n0 = (t % p.n_tiles) * BN;
    const int seg = mt % p.nseg, rowid = mt / p.nseg;  // rowid = b * H + h
    const int w = seg * BM + px;
    __nv_bfloat16 *yrow = p.y + ((size_t)rowid * p.W + w) * p.Cout;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + acc * 256 + c * 32, r);
      tmem_wait_ld();
      const int n = n0 + c * 32;
      float st1[32], st2[32];  // STATS: this pixel's stored values and their squares
      if (w < p.W && n < p.Cout) {
        uint4 res[4];  // accumulate: the residual already in y, all four loads in flight
#pragma unroll
        for (int v = 0; v < 4; ++v)
          res[v] = p.accumulate && n + 8 * v < p.Cout
                       ? *reinterpret_cast<const uint4 *>(yrow + n + 8 * v)
                       : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int nv = n + 8 * v;
          if (nv < p.Cout) {
            float bv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) bv[e] = p.bias ? __ldg(p.bias + nv + e) : 0.f;
            {  // bf16 -> fp32 is a 16-bit shift; zero when not accumulating
              const uint32_t rw[4] = {res[v].x, res[v].y, res[v].z, res[v].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                bv[2 * e] += __uint_as_float(rw[e] << 16);
                bv[2 * e + 1] += __uint_as_float(rw[e] & 0xffff0000u);
              }
            }
            uint4 o;
            uint32_t *ow = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              ow[e] = pack_bf162(__uint_as_float(r[8 * v + 2 * e]) + bv[2 * e],
                                 __uint_as_float(r[8 * v + 2 * e + 1]) + bv[2 * e + 1]);
            *reinterpret_cast<uint4 *>(yrow + nv) = o;
            if (STATS) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float lo = __uint_as_float(ow[e] << 16);
                const float hi = __uint_as_float(ow[e] & 0xffff0000u);
                st1[8 * v + 2 * e] = lo;
                st1[8 * v + 2 * e + 1] = hi;
              }
            }
          } else if (STATS) {
#pragma unroll
            for (int e = 0; e < 8; ++e) st1[8 * v + e] = 0.f;
          }
        }
      } else if (STATS) {
#pragma unroll
        for (int e = 0; e < 32; ++e) st1[e] = 0.f;
      }
      if (STATS) {
#pragma unroll
        for (int e = 0; e < 32; ++e) st2[e] = st1[e] * st1[e];
        const float t1 = warp_reduce_scatter32(st1);  // channel n + lane, this warp's pixels
        const float t2 = warp_reduce_scatter32(st2);
        float *dst = chs + ((q * BN) + c * 32 + lane) * 2;
        dst[0] = t1;
        dst[1] = t2;
      }
    }
    if (STATS) {
      // this warp's channel sums -> group sums -> fp64 totals.  fp32 sums of
      // similar size add exactly in fp64, so the totals do not depend on
      // the order the atomics land in.
      __syncwarp();
      const int cg = p.Cout / p.G;
      const int n1 = min(n0 + BN, p.Cout);
      const int g0 = n0 / cg, g1 = (n1 - 1) / cg;
      const int h = rowid % p.H, b = rowid / p.H, band = h / Hp;
      for (int g = g0 + lane; g <= g1; g += 32) {
        const int c0 = max(g * cg, n0) - n0, c1 = min((g + 1) * cg, n1) - n0;
        float s1 = 0.f, s2 = 0.f;
        for (int ch = c0; ch < c1; ++ch) {
          s1 += chs[(q * BN + ch) * 2];
          s2 += chs[(q * BN + ch) * 2 + 1];
        }
        double *gs = p.gn_sums + (((size_t)band * p.B + b) * p.G + g) * 2;
        atomicAdd(gs, (double)s1);
        atomicAdd(gs + 1, (double)s2);
      }
      __syncwarp();  // the slice is rewritten by the next tile
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&tempty[acc]);
  }
}

// STATS: the epilogue also adds, per band, image and GroupNorm group, the
// sum and the sum of squares of the values it stores (as rounded to bf16),
// into p.gn_sums -- the fresh partials a displaced GroupNorm of this output
// needs, so that GroupNorm is left with a single streaming pass.
template <int BN, int STAGES, bool STATS>
__global__ void __launch_bounds__(kThreads, 1)
conv_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmS,
               const __grid_constant__ CUtensorMap tmW, const ConvTcParams p) {
  constexpr uint32_t A_BYTES = BM * BK * 2;
  constexpr uint32_t B_BYTES = BN * BK * 2;
  constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr uint32_t IDESC = idesc_f16(BM, BN, true);
  static_assert(B_BYTES % 1024 == 0, "stage tiles must stay 1024-byte aligned");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  // STATS: each epilogue warp's channel sums over its 32 pixels: [4][BN][2]
  float *chs = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES + 512);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmS);
    prefetch_tmap(&tmW);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int KB = 9 * p.cblocks;
  const int tiles = p.m_tiles * p.n_tiles;
  const int Hp = p.H / p.P;

  if (warp == 0 || warp >= 6) {
    const int pid = warp == 0 ? 0 : warp - 5;  // this producer's stages: stage % kProducers
    {  // ------------------------- TMA producer (converged warp, elected lane)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;
      for (int t = blockIdx.x; t < tiles && !*abort_flag; t += gridDim.x) {
        const int mt = t / p.n_tiles, n0 = (t % p.n_tiles) * BN;
        const int seg = mt % p.nseg, rowid = mt / p.nseg;
        const int h = rowid % p.H, b = rowid / p.H;
        const int lo = (h / Hp) * Hp, hi = lo + Hp;
        const int w0 = seg * BM;
        for (int kb = 0; kb < KB; ++kb) {
          const int tap = kb / p.cblocks, cb = kb - tap * p.cblocks;
          const int hh = h + tap / 3 - 1;
          const bool halo_row = hh < lo || hh >= hi;
          // rows outside [0, H) are zero-filled whichever map is used; a
          // zero halo asks for row -1, which TMA fills with zeros as well
          const int hc = (p.zero_halo && halo_row) ? -1 : hh;
          const int ww = w0 + tap % 3 - 1;
          const CUtensorMap *src = (p.use_stale && halo_row) ? &tmS : &tmX;
          if (stage % kProducers != pid) {  // another producer warp's stage
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (!mbar_wait_w(&empty[stage], phase ^ 1u, abort_flag, p.status)) break;
          uint8_t *sa = smem + stage * STAGE_BYTES;
          mbar_arrive_expect_tx_w(&full[stage], STAGE_BYTES);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          tma_load_4d_w(sa, src, &full[stage], cb * BK, ww, hc, b);
          tma_load_3d_w(sa + A_BYTES, &tmW, &full[stage], cb * BK, tap, n0);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_flag)
        for (int s = 0; s < STAGES; ++s)
          if ((armed >> s) & 1u) mbar_drain(&full[s], (armed_parity >> s) & 1u);
    }
  } else if (warp == 1) {
    {  // ---------------------------- MMA issuer (converged warp, elected lane)
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait_w(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * 256;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_w(&full[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint64_t ad = desc_sw128_kmajor(sa);
          const uint64_t bd = desc_sw128_kmajor(sa + A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_f16_ss_w(d, ad + 2 * k, bd + 2 * k, IDESC, (kb | k) != 0);
          mma_commit_w(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_w(&tfull[acc]);
      }
      if (*abort_flag) {
        mma_commit_w(drain);
        mbar_drain(drain, 0);
      }
    }
  } else {  // ------------------------------------------------ epilogue
    conv_epilogue<BN, STATS>(p, tmem, tfull, tempty, abort_flag, chs, warp & 3, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}


// ---------------------------------------------------------------------------
// GroupNorm (+ SiLU) applied to the conv's input as it is loaded: the
// ResNet block's GroupNorm -> SiLU -> conv with the normalised tensor never
// stored.  The producer-side half of the fusion is the conv epilogue's
// GroupNorm sums (STATS); dpp_groupnorm_affine turns those sums into one
// scale and shift per (band, image, channel), and this kernel reads
//   Z'[b,hh,ww,c] = act(Z[b,hh,ww,c] * a[q,b,c] + s[q,b,c])
// with q the band of row hh, (a, s) of this step for the rows the band
// computes fresh and of the previous step for the halo rows it reads from
// the stale input -- exactly the values the unfused GroupNorm of the
// previous step wrote into the tensor the displaced conv reads as stale.
// Zero padding (rows -1 and H, columns -1 and W, and the zero halo of
// naive patches) stays zero: it pads the normalised tensor.
//
// A k-step is one input row (dy) and one 64-channel block: the producer
// loads the row's 130-pixel strip w0-1 .. w0+128 once (TMA, 128-byte
// swizzle), eight transform warps normalise it in place in shared memory,
// and the three horizontal taps are the strip read from row 0, 1 and 2:
// the MMA's A descriptor starts dx * 128 bytes into the strip (the swizzle
// follows the absolute shared-memory address, so a row-offset start reads
// the rows the copy wrote).  Each input value is loaded and normalised once
// per input row of a tile instead of once per tap.  The weights of the
// three taps of a row arrive in one box {64 ch, BN, 3 taps} of a map that
// walks [C_out][3][3][C_in] with the tap as its slowest coordinate.
//
//   warp 0      strip producer (A ring, SA slots)
//   warp 6      weight producer (B ring, SB slots of 3 taps)
//   warp 1      TMEM owner and MMA issuer: per k-step 3 taps x 4 K-steps
//   warps 2..5  epilogue (as conv_tc_kernel)
//   warps 7..14 transform: thread t normalises 16-byte chunk t % 8 of
//               pixels t / 8 + 32 i of the strip (conflict-free: 4 whole
//               128-byte rows per warp access); two warps per scheduler
//               hide each other's load and special-function latency
// The activation is SiLU(v) = h + h tanh(h), h = v / 2 (PTX tanh.approx.f32:
// one special-function op per value, |error| about |h| 2^-11), so the
// transform's special-function work stays inside the tensor time of a
// k-step.
constexpr int kNormThreads = 480;
constexpr uint32_t kStripRows = BM + 2;
constexpr uint32_t kStripBytes = kStripRows * 128;                  // transaction bytes
constexpr uint32_t kStripSlot = (kStripBytes + 1023u) & ~1023u;     // 1024-aligned slots

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float norm_act(float x, float a, float s, int act) {
  const float v = fmaf(x, a, s);
  if (act != DPP_ACT_SILU) return v;
  const float h = 0.5f * v;
  return fmaf(h, tanh_approx(h), h);
}

template <int BN, int SA, int SB, bool STATS>
__global__ void __launch_bounds__(kNormThreads, 1)
conv_norm_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmS,
                    const __grid_constant__ CUtensorMap tmW3, const ConvTcParams p) {
  constexpr uint32_t B_TAP = BN * BK * 2;
  constexpr uint32_t B_SLOT = 3 * B_TAP;
  constexpr uint32_t IDESC = idesc_f16(BM, BN, true);
  static_assert(B_TAP % 1024 == 0, "tap tiles must stay 1024-byte aligned");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t *sA = smem;
  uint8_t *sB = smem + SA * kStripSlot;
  uint64_t *a_full = reinterpret_cast<uint64_t *>(sB + SB * B_SLOT);
  uint64_t *a_ready = a_full + SA;
  uint64_t *a_empty = a_ready + SA;
  uint64_t *b_full = a_empty + SA;
  uint64_t *b_empty = b_full + SB;
  uint64_t *tfull = b_empty + SB;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  float *chs = reinterpret_cast<float *>(sB + SB * B_SLOT + 512);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_ready[s], 8);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmS);
    prefetch_tmap(&tmW3);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int KS = 3 * p.cblocks;  // k-steps per tile: input rows x channel blocks
  const int tiles = p.m_tiles * p.n_tiles;
  const int Hp = p.H / p.P;

  if (warp == 0) {  // --------------------------------- strip producer
    int slot = 0;
    uint32_t phase = 0, armed = 0, armed_parity = 0;
    for (int t = blockIdx.x; t < tiles && !*abort_flag; t += gridDim.x) {
      const int mt = t / p.n_tiles;
      const int seg = mt % p.nseg, rowid = mt / p.nseg;
      const int h = rowid % p.H, b = rowid / p.H;
      const int lo = (h / Hp) * Hp, hi = lo + Hp;
      const int w0 = seg * BM;
      bool ok = true;
      for (int dy = 0; dy < 3 && ok; ++dy) {
        const int hh = h + dy - 1;
        const bool halo_row = hh < lo || hh >= hi;
        const int hc = (p.zero_halo && halo_row) ? -1 : hh;
        const CUtensorMap *src = (p.use_stale && halo_row) ? &tmS : &tmX;
        for (int cb = 0; cb < p.cblocks; ++cb) {
          if (!mbar_wait_w(&a_empty[slot], phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx_w(&a_full[slot], kStripBytes);
          armed |= 1u << slot;
          armed_parity = (armed_parity & ~(1u << slot)) | (phase << slot);
          tma_load_4d_w(sA + slot * kStripSlot, src, &a_full[slot], cb * BK, w0 - 1, hc, b);
          if (++slot == SA) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) break;
    }
    if (*abort_flag)
      for (int s = 0; s < SA; ++s)
        if ((armed >> s) & 1u) mbar_drain(&a_full[s], (armed_parity >> s) & 1u);
  } else if (warp == 6) {  // ------------------------- weight producer
    int slot = 0;
    uint32_t phase = 0, armed = 0, armed_parity = 0;
    for (int t = blockIdx.x; t < tiles && !*abort_flag; t += gridDim.x) {
      const int n0 = (t % p.n_tiles) * BN;
      bool ok = true;
      for (int ks = 0; ks < KS; ++ks) {
        const int dy = ks / p.cblocks, cb = ks - dy * p.cblocks;
        if (!mbar_wait_w(&b_empty[slot], phase ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx_w(&b_full[slot], B_SLOT);
        armed |= 1u << slot;
        armed_parity = (armed_parity & ~(1u << slot)) | (phase << slot);
        tma_load_3d_w(sB + slot * B_SLOT, &tmW3, &b_full[slot], cb * BK, n0, 3 * dy);
        if (++slot == SB) {
          slot = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
    if (*abort_flag)
      for (int s = 0; s < SB; ++s)
        if ((armed >> s) & 1u) mbar_drain(&b_full[s], (armed_parity >> s) & 1u);
  } else if (warp == 1) {  // --------------------------------- MMA issuer
    int sa = 0, sb = 0;
    uint32_t pa = 0, pb = 0;
    int it = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!mbar_wait_w(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t d = tmem + acc * 256;
      bool ok = true;
      for (int ks = 0; ks < KS; ++ks) {
        if (!mbar_wait_w(&a_ready[sa], pa, abort_flag, p.status) ||
            !mbar_wait_w(&b_full[sb], pb, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + sa * kStripSlot);
        const uint32_t b0 = smem_u32(sB + sb * B_SLOT);
#pragma unroll
        for (int dx = 0; dx < 3; ++dx) {
          const uint64_t ad = desc_sw128_kmajor(a0 + dx * 128);
          const uint64_t bd = desc_sw128_kmajor(b0 + dx * B_TAP);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_f16_ss_w(d, ad + 2 * k, bd + 2 * k, IDESC, (ks | dx | k) != 0);
        }
        mma_commit_w(&a_empty[sa]);
        mma_commit_w(&b_empty[sb]);
        if (++sa == SA) {
          sa = 0;
          pa ^= 1u;
        }
        if (++sb == SB) {
          sb = 0;
          pb ^= 1u;
        }
      }
      if (!ok) break;
      mma_commit_w(&tfull[acc]);
    }
    if (*abort_flag) {
      mma_commit_w(drain);
      mbar_drain(drain, 0);
    }
  } else if (warp >= 7) {  // ---------------------------------- transform
    const int tid = threadIdx.x - 7 * 32;  // 0 .. 255
    const int j = tid & 7, p0 = tid >> 3;
    int slot = 0;
    uint32_t phase = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
      const int mt = t / p.n_tiles;
      const int seg = mt % p.nseg, rowid = mt / p.nseg;
      const int h = rowid % p.H, b = rowid / p.H;
      const int lo = (h / Hp) * Hp, hi = lo + Hp;
      const int w0 = seg * BM;
      bool ok = true;
      for (int dy = 0; dy < 3 && ok; ++dy) {
        const int hh = h + dy - 1;
        const bool halo_row = hh < lo || hh >= hi;
        // rows outside the image and the zero halo were filled with zeros
        // by the copy, which is what the padded normalised tensor holds
        const bool live = hh >= 0 && hh < p.H && !(p.zero_halo && halo_row);
        const float *tab = (p.use_stale && halo_row) ? p.affine_prev : p.affine;
        const float *tb = live ? tab + ((size_t)(hh / Hp) * p.B + b) * p.Cin * 2 : nullptr;
        for (int cb = 0; cb < p.cblocks; ++cb) {
          if (!mbar_wait_w(&a_full[slot], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const int c0 = cb * BK + 8 * j;
          if (live && c0 < p.Cin) {
            float sc[8], sh[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float4 v = __ldg(reinterpret_cast<const float4 *>(tb + (size_t)c0 * 2) + e);
              sc[2 * e] = v.x;
              sh[2 * e] = v.y;
              sc[2 * e + 1] = v.z;
              sh[2 * e + 1] = v.w;
            }
            uint8_t *strip = sA + slot * kStripSlot;
#pragma unroll
            for (int i = 0; i < 5; ++i) {
              const int px = p0 + 32 * i;
              const int ww = w0 - 1 + px;
              if (px < (int)kStripRows && ww >= 0 && ww < p.W) {
                uint4 *ptr = reinterpret_cast<uint4 *>(strip + px * 128 + ((j ^ (px & 7)) << 4));
                uint4 v = *ptr;
                uint32_t *vw = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  vw[e] = pack_bf162(
                      norm_act(__uint_as_float(vw[e] << 16), sc[2 * e], sh[2 * e], p.act),
                      norm_act(__uint_as_float(vw[e] & 0xffff0000u), sc[2 * e + 1],
                               sh[2 * e + 1], p.act));
                *ptr = v;
              }
            }
            fence_proxy_async_smem();  // the MMA reads the strip through the async proxy
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_ready[slot]);
          if (++slot == SA) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) break;
    }
  } else {  // ------------------------------------------------ epilogue
    conv_epilogue<BN, STATS>(p, tmem, tfull, tempty, abort_flag, chs, warp & 3, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

constexpr size_t kSmemBudget = 227 * 1024;

template <int BN, bool STATS>
constexpr int stages_for() {
  return (int)((kSmemBudget - 2048 - (STATS ? 4 * BN * 2 * sizeof(float) : 0)) /
               (size_t)(BM * BK * 2 + BN * BK * 2)) > 8
             ? 8
             : (int)((kSmemBudget - 2048 - (STATS ? 4 * BN * 2 * sizeof(float) : 0)) /
                     (size_t)(BM * BK * 2 + BN * BK * 2));
}

template <int BN, bool STATS>
cudaError_t run(const dpp_conv_desc &d, const CUtensorMap &mx, const CUtensorMap &ms,
                const void *w, const float *bias, void *y, int use_stale, int zero_halo,
                double *gn_sums, int G, int *status, cudaStream_t s) {
  constexpr int STAGES = stages_for<BN, STATS>();
  CUtensorMap mw;
  {
    const uint64_t dims[3] = {(uint64_t)d.C_in, 9, (uint64_t)d.C_out};
    const uint64_t str[2] = {(uint64_t)d.C_in * 2, (uint64_t)d.C_in * 9 * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)BN};
    if (!encode_tiled(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, w, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  ConvTcParams p;
  p.B = d.B; p.H = d.H; p.W = d.W; p.Cin = d.C_in; p.Cout = d.C_out; p.P = d.P;
  p.nseg = (d.W + BM - 1) / BM;
  p.cblocks = (d.C_in + BK - 1) / BK;
  p.m_tiles = d.B * d.H * p.nseg;
  p.n_tiles = (d.C_out + BN - 1) / BN;
  p.use_stale = use_stale;
  p.zero_halo = zero_halo;
  p.accumulate = d.accumulate ? 1 : 0;
  p.bias = bias;
  p.y = reinterpret_cast<__nv_bfloat16 *>(y);
  p.status = status;
  p.gn_sums = gn_sums;
  p.G = G;
  constexpr size_t smem = (size_t)STAGES * (BM * BK * 2 + BN * BK * 2) + 1024 + 512 +
                          (STATS ? (size_t)4 * BN * 2 * sizeof(float) : 0);
  static_assert(smem <= kSmemBudget, "shared memory budget");
  auto k = conv_tc_kernel<BN, STAGES, STATS>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long tiles = (long long)p.m_tiles * p.n_tiles;
  const int grid = tiles < sms ? (int)tiles : sms;
  k<<<grid, kThreads, smem, s>>>(mx, ms, mw, p);
  return cudaGetLastError();
}

// N tile for C_out: the candidate with the least padded work (tiles x BN),
// the larger one on ties.
int pick_bn(int cout) {
  const int cands[4] = {64, 128, 160, 256};
  int best = 0;
  long long best_work = -1;
  for (int bn : cands) {
    const long long work = (long long)((cout + bn - 1) / bn) * bn;
    if (best_work < 0 || work <= best_work) {
      best = bn;
      best_work = work;
    }
  }
  return best;
}


// Ring depths of the normalising conv: weight slots (3 taps each) by N
// tile, strip slots from what shared memory has left (at most 6).
template <int BN>
constexpr int norm_sb() {
  return BN <= 64 ? 4 : (BN <= 128 ? 3 : 2);
}
template <int BN, bool STATS>
constexpr size_t norm_extra() {
  return 1024 + 512 + (STATS ? (size_t)4 * BN * 2 * sizeof(float) : 0);
}
template <int BN, bool STATS>
constexpr int norm_sa() {
  return (int)((kSmemBudget - (size_t)norm_sb<BN>() * 3 * BN * BK * 2 - norm_extra<BN, STATS>()) /
               kStripSlot) > 6
             ? 6
             : (int)((kSmemBudget - (size_t)norm_sb<BN>() * 3 * BN * BK * 2 -
                      norm_extra<BN, STATS>()) /
                     kStripSlot);
}

template <int BN, bool STATS>
cudaError_t run_norm(const dpp_conv_desc &d, const CUtensorMap &mx, const CUtensorMap &ms,
                     const void *w, ConvTcParams p, cudaStream_t s) {
  constexpr int SB = norm_sb<BN>(), SA = norm_sa<BN, STATS>();
  static_assert(SA >= 3, "strip ring too shallow");
  CUtensorMap mw;
  {  // [C_out][3][3][C_in] walked as {C_in, C_out, tap}: one box = 3 taps of a row
    const uint64_t dims[3] = {(uint64_t)d.C_in, (uint64_t)d.C_out, 9};
    const uint64_t str[2] = {(uint64_t)d.C_in * 9 * 2, (uint64_t)d.C_in * 2};
    const uint32_t box[3] = {64, (uint32_t)BN, 3};
    if (!encode_tiled(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, w, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  p.nseg = (d.W + BM - 1) / BM;
  p.m_tiles = d.B * d.H * p.nseg;
  p.n_tiles = (d.C_out + BN - 1) / BN;
  constexpr size_t smem = (size_t)SA * kStripSlot + (size_t)SB * 3 * BN * BK * 2 +
                          norm_extra<BN, STATS>();
  static_assert(smem <= kSmemBudget, "shared memory budget");
  auto k = conv_norm_tc_kernel<BN, SA, SB, STATS>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long tiles = (long long)p.m_tiles * p.n_tiles;
  const int grid = tiles < sms ? (int)tiles : sms;
  k<<<grid, kNormThreads, smem, s>>>(mx, ms, mw, p);
  return cudaGetLastError();
}

// N tile of the normalising conv: the least padded work among 64, 128 and
// 160 columns, the larger on ties (each input strip is normalised once per
// N tile, so fewer, wider tiles also mean fewer transforms).
int pick_bn_norm(int cout) {
  const int cands[3] = {64, 128, 160};
  int best = 0;
  long long best_work = -1;
  for (int bn : cands) {
    const long long work = (long long)((cout + bn - 1) / bn) * bn;
    if (best_work < 0 || work <= best_work) {
      best = bn;
      best_work = work;
    }
  }
  return best;
}

}  // namespace

__global__ void zero_f64_kernel(double *p, size_t n) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    p[i] = 0.0;
}

cudaError_t launch_zero_f64(double *p, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  zero_f64_kernel<<<(unsigned)((n + 255) / 256 < 148 ? (n + 255) / 256 : 148), 256, 0, s>>>(p, n);
  return cudaGetLastError();
}

cudaError_t launch_conv_norm_tc(const dpp_conv_desc &d, const void *x, const void *stale,
                                const float *affine, const float *affine_prev, int act,
                                const void *w, const float *bias, void *y, int *status,
                                cudaStream_t s, double *gn_sums, int G) {
  if (!conv_tc_supported(d)) return cudaErrorNotSupported;
  const int use_stale = (stale && stale != x && d.halo == DPP_HALO_STALE) ? 1 : 0;
  CUtensorMap mx, ms;
  const uint64_t dims[4] = {(uint64_t)d.C_in, (uint64_t)d.W, (uint64_t)d.H, (uint64_t)d.B};
  const uint64_t str[3] = {(uint64_t)d.C_in * 2, (uint64_t)d.W * d.C_in * 2,
                           (uint64_t)d.H * d.W * d.C_in * 2};
  const uint32_t box[4] = {64, kStripRows, 1, 1};  // one row's strip: 128 pixels and both neighbours
  if (!encode_tiled(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, x, dims, str, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_tiled(&ms, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, use_stale ? stale : x, dims, str,
                    box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (gn_sums) {
    const cudaError_t e = launch_zero_f64(gn_sums, (size_t)d.P * d.B * G * 2, s);
    if (e != cudaSuccess) return e;
  }
  ConvTcParams p{};
  p.B = d.B; p.H = d.H; p.W = d.W; p.Cin = d.C_in; p.Cout = d.C_out; p.P = d.P;
  p.cblocks = (d.C_in + BK - 1) / BK;
  p.use_stale = use_stale;
  p.zero_halo = d.halo == DPP_HALO_ZERO ? 1 : 0;
  p.accumulate = d.accumulate ? 1 : 0;
  p.bias = bias;
  p.y = reinterpret_cast<__nv_bfloat16 *>(y);
  p.status = status;
  p.gn_sums = gn_sums;
  p.G = G;
  p.affine = affine;
  p.affine_prev = use_stale ? affine_prev : affine;
  p.act = act;
  const bool st = gn_sums != nullptr;
  switch (pick_bn_norm(d.C_out)) {
    case 64:
      return st ? run_norm<64, true>(d, mx, ms, w, p, s) : run_norm<64, false>(d, mx, ms, w, p, s);
    case 128:
      return st ? run_norm<128, true>(d, mx, ms, w, p, s)
                : run_norm<128, false>(d, mx, ms, w, p, s);
    default:
      return st ? run_norm<160, true>(d, mx, ms, w, p, s)
                : run_norm<160, false>(d, mx, ms, w, p, s);
  }
}

bool conv_tc_supported(const dpp_conv_desc &d) {
  return d.dtype == DPP_BF16 && d.C_in % 8 == 0 && d.C_out % 8 == 0 && d.H % d.P == 0 &&
         (long long)d.B * d.H * ((d.W + BM - 1) / BM) < (1ll << 31);
}

cudaError_t launch_conv_tc(const dpp_conv_desc &d, const void *x, const void *stale,
                           const void *w, const float *bias, void *y, int *status,
                           cudaStream_t s, double *gn_sums, int G) {
  if (!conv_tc_supported(d)) return cudaErrorNotSupported;
  const int use_stale = (stale && stale != x && d.halo == DPP_HALO_STALE) ? 1 : 0;
  const int zero_halo = d.halo == DPP_HALO_ZERO ? 1 : 0;
  CUtensorMap mx, ms;
  const uint64_t dims[4] = {(uint64_t)d.C_in, (uint64_t)d.W, (uint64_t)d.H, (uint64_t)d.B};
  const uint64_t str[3] = {(uint64_t)d.C_in * 2, (uint64_t)d.W * d.C_in * 2,
                           (uint64_t)d.H * d.W * d.C_in * 2};
  const uint32_t box[4] = {64, 128, 1, 1};
  if (!encode_tiled(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, x, dims, str, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_tiled(&ms, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, use_stale ? stale : x, dims, str,
                    box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (gn_sums) {  // the epilogue accumulates into it: start from zero
    const cudaError_t e = launch_zero_f64(gn_sums, (size_t)d.P * d.B * G * 2, s);
    if (e != cudaSuccess) return e;
  }
  const bool st = gn_sums != nullptr;
  switch (pick_bn(d.C_out)) {
    case 64:
      return st ? run<64, true>(d, mx, ms, w, bias, y, use_stale, zero_halo, gn_sums, G, status, s)
                : run<64, false>(d, mx, ms, w, bias, y, use_stale, zero_halo, nullptr, 0, status, s);
    case 128:
      return st ? run<128, true>(d, mx, ms, w, bias, y, use_stale, zero_halo, gn_sums, G, status, s)
                : run<128, false>(d, mx, ms, w, bias, y, use_stale, zero_halo, nullptr, 0, status, s);
    case 160:
      return st ? run<160, true>(d, mx, ms, w, bias, y, use_stale, zero_halo, gn_sums, G, status, s)
                : run<160, false>(d, mx, ms, w, bias, y, use_stale, zero_halo, nullptr, 0, status, s);
    default:
      return st ? run<256, true>(d, mx, ms, w, bias, y, use_stale, zero_halo, gn_sums, G, status, s)
                : run<256, false>(d, mx, ms, w, bias, y, use_stale, zero_halo, nullptr, 0, status, s);
  }
}

}  // namespace dpp

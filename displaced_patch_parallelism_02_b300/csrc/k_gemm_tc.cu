// Tensor-core GEMM for the attention projections: D = A * B^T on tcgen05.
//
// A [M, K] and the weight blocks B_i [b_rows, K] are K-major 16-bit tensors
// (both fp16 or both bf16).  The output columns are split between two
// destinations: the QKV projection writes Q to the workspace and the fresh
// K/V of every token straight into the next step's attention state (the
// refresh of DistriSelfAttentionPP's state costs no extra pass).
//
// Persistent, warp-specialised, one CTA per SM:
//   warp 0      TMA producer (converged warp, an elected lane issues each
//               copy): per stage the A tile 128 x 64 and the B tile BN x 64
//               as ONE box each (column tiles never straddle two weight
//               blocks, so a tile's B rows are one box of one block),
//               128-byte swizzle, STAGES-deep mbarrier ring.  Few large
//               copies matter: a thread that issues bulk tensor copies pays
//               a fixed cost per copy, and four 64-row boxes per stage fed
//               the tensor pipe at under half its rate;
//   warp 1      TMEM allocation and the tcgen05.mma issuer (converged warp,
//               one elected lane per instruction), M = 128, N = the tile's
//               width, K = 16 per instruction, fp32 accumulators
//               double-buffered in TMEM (2 x BN columns);
//   warps 2..9  epilogue, two warps per TMEM lane quadrant, each converting
//               half of the tile's columns: tcgen05.ld 32 columns at a time
//               (the next chunk's load in flight while one is converted),
//               + bias (broadcast 16-byte loads), + the residual already in
//               out0 (loaded a chunk ahead), convert, stage in shared memory
//               (64-byte swizzle: conflict-free), one bulk tensor store per
//               32 x 32 chunk; or the gated-GELU epilogue (value * GELU(gate)).
// Tiles are ordered n-fastest so CTAs running together share A rows in L2.
#include "tc_common.cuh"

namespace dpp {

namespace tc {

bool encode_tiled(CUtensorMap *map, CUtensorMapDataType type, int rank, const void *base,
                  const uint64_t *dims, const uint64_t *strides, const uint32_t *box,
                  CUtensorMapSwizzle swizzle) {
  using Fn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                          const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                          const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                          CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static Fn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
      return false;
    fn = reinterpret_cast<Fn>(p);
  }
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(map, type, (cuuint32_t)rank, const_cast<void *>(base),
            reinterpret_cast<const cuuint64_t *>(dims),
            reinterpret_cast<const cuuint64_t *>(strides),
            reinterpret_cast<const cuuint32_t *>(box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

namespace {

using namespace tc;

struct GemmTcParams {
  int M, N, K, b_rows;
  void *out0;
  int ld0, split;
  void *out1;
  int ld1;
  int out_f16;  // 1: fp16 output, 0: bf16 output
  int m_tiles, n_tiles;
  int tpb;      // column tiles per weight block (plain GEMM)
  int *status;
  const float *bias;  // per out0 column ([2 N] with geglu: value then gate), or null
  int accumulate;     // out0 += result
  int geglu;          // tile = BN/2 value rows of B0 + BN/2 gate rows of B1
  int pf_boxes;       // residual L2 prefetch boxes per tile (0: no residual)
  int pf_cols;        // columns per prefetch box
  const void *cast_src;  // bf16 -> fp16 side copy (cast_n elements), or null
  void *cast_dst;
  size_t cast_n;
};

// erf(x) by Abramowitz & Stegun, Handbook of Mathematical Functions, 7.1.25:
// erf(x) = 1 - (a1 t + a2 t^2 + a3 t^3) exp(-x^2) + e(x), t = 1 / (1 + p x),
// |e(x)| <= 2.5e-5 for x >= 0 (odd extension for x < 0) -- four orders below
// half a bf16 ulp of the gated-GELU output it feeds.
__device__ __forceinline__ float erf_as7125(float x) {
  const float ax = fabsf(x);
  const float t = __fdividef(1.f, fmaf(0.47047f, ax, 1.f));
  const float poly = t * fmaf(t, fmaf(t, 0.7478556f, -0.0958798f), 0.3480242f);
  return copysignf(1.f - poly * __expf(-ax * ax), x);
}

constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int BM = 128, BK = 64;
constexpr uint32_t kStageOut = 2048;  // one 32 x 32 chunk of 16-bit outputs

// Columns of column tile j: output columns [n0, n0 + w) from weight block
// `mat`, rows [brow, brow + w) of it.  A plain GEMM tiles each weight block
// on its own (tiles of BN, the last one narrower); gated GELU tiles the N
// output columns by BN/2 (value and gate rows of the same columns).
template <int BN>
__device__ __forceinline__ bool tile_cols(const GemmTcParams &p, int j, int &n0, int &w, int &mat,
                                          int &brow) {
  if (p.geglu) {
    n0 = j * (BN / 2);
    w = min(BN / 2, p.N - n0);
    mat = 0;
    brow = n0;
  } else {
    const int blk = j / p.tpb, off = (j % p.tpb) * BN;
    n0 = blk * p.b_rows + off;
    w = min(min(BN, p.b_rows - off), p.N - n0);
    mat = blk;
    brow = off;
  }
  return w > 0;
}

template <int BN, int STAGES, bool IN_BF16>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
               const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
               const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmO1,
               const __grid_constant__ CUtensorMap tmR, const GemmTcParams p) {
  constexpr uint32_t A_BYTES = BM * BK * 2;
  constexpr uint32_t B_BYTES = BN * BK * 2;
  constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr uint32_t TMEM_COLS = (2 * BN <= 256) ? 256 : 512;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  // per epilogue warp two output staging buffers, then the barriers
  uint8_t *stage_out = smem + STAGES * STAGE_BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(stage_out + kEpiWarps * 2 * kStageOut);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;  // MMA completion on the abort path
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiWarps);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB0);
    prefetch_tmap(&tmB1);
    prefetch_tmap(&tmB2);
    if (p.pf_boxes) prefetch_tmap(&tmR);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int KB = (p.K + BK - 1) / BK;
  const int tiles = p.m_tiles * p.n_tiles;

  if (warp == 0) {
    {  // ------------------------- TMA producer (converged warp, elected lane)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;  // per-stage bits, for the abort drain
      for (int t = blockIdx.x; t < tiles && !*abort_flag; t += gridDim.x) {
        int n0, w, mat, brow;
        if (!tile_cols<BN>(p, t % p.n_tiles, n0, w, mat, brow)) continue;
        const int m0 = (t / p.n_tiles) * BM;
        const CUtensorMap *mb = mat == 0 ? &tmB0 : (mat == 1 ? &tmB1 : &tmB2);
        // The residual the epilogue adds is pulled into L2 now, a whole tile
        // of MMAs before it is read: per-thread loads issued only a chunk
        // ahead cannot keep enough bytes in flight to cover DRAM latency.
        if (p.pf_boxes && n0 < p.split)
          for (int b = 0; b < p.pf_boxes && b * p.pf_cols < w; ++b)
            tma_prefetch_l2_2d_w(&tmR, n0 + b * p.pf_cols, m0);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_w(&empty[stage], phase ^ 1u, abort_flag, p.status)) break;
          uint8_t *sa = smem + stage * STAGE_BYTES;
          // full boxes are always credited (rows outside a block read as zero)
          mbar_arrive_expect_tx_w(&full[stage], STAGE_BYTES);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          tma_load_2d_w(sa, &tmA, &full[stage], kb * BK, m0);
          if (p.geglu) {  // value rows, then the gate rows of the same columns
            tma_load_2d_w(sa + A_BYTES, &tmB0, &full[stage], kb * BK, brow);
            tma_load_2d_w(sa + A_BYTES + (BN / 2) * 128, &tmB1, &full[stage], kb * BK, brow);
          } else {
            tma_load_2d_w(sa + A_BYTES, mb, &full[stage], kb * BK, brow);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_flag)  // let copies already in flight land before the CTA exits
        for (int s = 0; s < STAGES; ++s)
          if ((armed >> s) & 1u) mbar_drain(&full[s], (armed_parity >> s) & 1u);
    }
  } else if (warp == 1) {
    {  // ---------------------------- MMA issuer (converged warp, elected lane)
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        int n0, w, mat, brow;
        if (!tile_cols<BN>(p, t % p.n_tiles, n0, w, mat, brow)) continue;
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        ++it;
        if (!mbar_wait_w(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        // a narrow last tile multiplies only its own columns
        const uint32_t idesc = idesc_f16(BM, p.geglu ? BN : ((w + 15) & ~15), IN_BF16);
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
            mma_f16_ss_w(d, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0);
          mma_commit_w(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_w(&tfull[acc]);
      }
      if (*abort_flag) {  // no MMA may still be writing TMEM when it is freed
        mma_commit_w(drain);
        mbar_drain(drain, 0);
      }
    }
  } else {  // ------------------------------------------------ epilogue
    const int q = warp & 3;         // TMEM lane quadrant this warp may access
    const int half = (warp - 2) / 4;  // which half of the tile's columns it converts
    const int row = q * 32 + lane;
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
    // this warp's two output staging buffers (32 rows x 64 bytes each,
    // 16-byte units swizzled by the row as the 64-byte tensor-map swizzle does)
    uint8_t *stage_o = stage_out + (warp - 2) * 2 * kStageOut;
    int n_stored = 0;  // chunks this warp has handed to the bulk-store engine
    if (p.cast_n) {
      // The side copy (the output projection's weight, bf16 -> fp16, for a
      // later launch) while the first accumulator is still being computed:
      // 16-byte vectors, grid-strided over every epilogue thread.
      const size_t nv = p.cast_n / 8;
      const size_t nthr = (size_t)gridDim.x * kEpiWarps * 32;
      const uint4 *src = reinterpret_cast<const uint4 *>(p.cast_src);
      uint4 *dst = reinterpret_cast<uint4 *>(p.cast_dst);
      for (size_t v = (size_t)blockIdx.x * kEpiWarps * 32 + (threadIdx.x - 64); v < nv;
           v += nthr) {
        const uint4 in = __ldg(src + v);
        const uint32_t iw[4] = {in.x, in.y, in.z, in.w};
        uint4 o;
        uint32_t *ow = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          ow[e] = pack_half2(__uint_as_float(iw[e] << 16), __uint_as_float(iw[e] & 0xffff0000u));
        dst[v] = o;
      }
    }
    int it = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
      int n0, w, mat, brow;
      if (!tile_cols<BN>(p, t % p.n_tiles, n0, w, mat, brow)) continue;
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      ++it;
      const int m0 = (t / p.n_tiles) * BM;
      const int m = m0 + row;
      // every lane leaves together (a lane that timed out has set the abort flag)
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status)))
        break;
      tc_fence_after();
      if (p.geglu) {
        // value columns [0, BN/2) and gate columns [BN/2, BN) of the
        // accumulator: out[n0 + j] = (value_j + b_j) * GELU(gate_j + b_{N + j}),
        // staged and stored like the plain epilogue's chunks
        constexpr int CH = BN / 128;  // value chunks per warp
#pragma unroll 1
        for (int cc = 0; cc < CH; ++cc) {
          const int c = half * CH + cc;
          if (c * 32 >= w) break;  // warp-uniform
          uint32_t rv[32], rg[32];
          const uint32_t ta = tq + acc * BN + c * 32;
          tmem_ld32(ta, rv);
          tmem_ld32(ta + BN / 2, rg);
          const int n = n0 + c * 32;
          const bool ld = p.accumulate && m < p.M;
          uint4 res[4];  // loads in flight while the accumulator is read
#pragma unroll
          for (int v = 0; v < 4; ++v)
            res[v] = ld ? reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(
                              p.out0) + (size_t)m * p.ld0 + n)[v]
                        : make_uint4(0u, 0u, 0u, 0u);
          tmem_wait_ld();
          uint8_t *buf = stage_o + (n_stored & 1) * kStageOut;
          if (n_stored >= 2) {  // the store that read this buffer two chunks ago
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
          }
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            // this 8-column group's value and gate biases (broadcast loads)
            float4 b4[4] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f),
                            make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
            if (p.bias) {
              const float4 *bv = reinterpret_cast<const float4 *>(p.bias + n + 8 * v);
              const float4 *bg = reinterpret_cast<const float4 *>(p.bias + p.N + n + 8 * v);
              b4[0] = __ldg(bv);
              b4[1] = __ldg(bv + 1);
              b4[2] = __ldg(bg);
              b4[3] = __ldg(bg + 1);
            }
            const float *bvf = reinterpret_cast<const float *>(&b4[0]);
            const float *bgf = reinterpret_cast<const float *>(&b4[2]);
            const uint32_t rw[4] = {res[v].x, res[v].y, res[v].z, res[v].w};
            uint4 o;
            uint32_t *ow = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float f[2];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int k = v * 8 + 2 * e + h;
                const float a = __uint_as_float(rv[k]) + bvf[2 * e + h];
                const float g = __uint_as_float(rg[k]) + bgf[2 * e + h];
                f[h] = a * (0.5f * g * (1.f + erf_as7125(g * 0.70710678118654752f)));
              }
              f[0] += __uint_as_float(rw[e] << 16);
              f[1] += __uint_as_float(rw[e] & 0xffff0000u);
              ow[e] = pack_bf162(f[0], f[1]);
            }
            *reinterpret_cast<uint4 *>(buf + lane * 64 + ((v ^ ((lane >> 1) & 3)) * 16)) = o;
          }
          fence_proxy_async_smem();  // the generic-proxy writes, before the bulk copy reads them
          __syncwarp();
          if (lane == 0) tma_store_2d(&tmO0, buf, n, m0 + q * 32);  // rows past M clipped
          ++n_stored;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        continue;
      }
      float amax = 0.f;  // largest |value| this thread stores (fp16 range check)
      constexpr int CH = BN / 64;  // 32-column chunks per warp
      const int c_begin = half * CH;
      const int c_end = min(c_begin + CH, (w + 31) / 32);
      // Each 32 x 32 chunk is converted into a staging buffer and written by
      // one bulk tensor store: whole cache lines, asynchronous, rows past M
      // clipped by the tensor map.  The residual is loaded a chunk ahead,
      // and the next chunk's accumulator columns are read while this one is
      // converted; the bias is a broadcast load that hits L1.
      auto residual = [&](int c, uint4 (&rr)[4]) {
        const int n = n0 + c * 32;
        const bool ld = p.accumulate && n < p.split && m < p.M;
#pragma unroll
        for (int v = 0; v < 4; ++v)
          rr[v] = ld ? reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(p.out0) +
                                                       (size_t)m * p.ld0 + n)[v]
                     : make_uint4(0u, 0u, 0u, 0u);
      };
      if (c_begin < c_end) {
        uint4 res_next[4];
        residual(c_begin, res_next);
        uint32_t rr2[2][32];
        tmem_ld32(tq + acc * BN + c_begin * 32, rr2[0]);
#pragma unroll
        for (int cc = 0; cc < CH; ++cc) {
          const int c = c_begin + cc;
          if (c >= c_end) break;  // warp-uniform
          uint32_t(&r)[32] = rr2[cc & 1];
          const int n = n0 + c * 32;
          const bool first = n < p.split;
          const bool acc_in = first && p.accumulate;
          uint4 res[4];
#pragma unroll
          for (int v = 0; v < 4; ++v) res[v] = res_next[v];
          if (c + 1 < c_end) residual(c + 1, res_next);
          tmem_wait_ld();
          if (cc + 1 < CH && c + 1 < c_end) tmem_ld32(tq + acc * BN + (c + 1) * 32, rr2[(cc + 1) & 1]);
          float4 bias4[8];  // the chunk's bias, zero outside out0's columns
#pragma unroll
          for (int v = 0; v < 8; ++v)
            bias4[v] = p.bias && first ? __ldg(reinterpret_cast<const float4 *>(p.bias + n) + v)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
          const float *bf = reinterpret_cast<const float *>(bias4);
          uint8_t *buf = stage_o + (n_stored & 1) * kStageOut;
          if (n_stored >= 2) {  // the store that read this buffer two chunks ago
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
          }
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 o;
            uint32_t *ow = reinterpret_cast<uint32_t *>(&o);
            const uint32_t rw[4] = {res[v].x, res[v].y, res[v].z, res[v].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int k = v * 8 + 2 * e;
              float a = __uint_as_float(r[k]) + bf[k];
              float b = __uint_as_float(r[k + 1]) + bf[k + 1];
              if (acc_in) {  // out0 is bf16 or fp16, as the output
                if (p.out_f16) {
                  const float2 old = __half22float2(*reinterpret_cast<const __half2 *>(&rw[e]));
                  a += old.x;
                  b += old.y;
                } else {
                  a += __uint_as_float(rw[e] << 16);
                  b += __uint_as_float(rw[e] & 0xffff0000u);
                }
              }
              if (p.out_f16) amax = fmaxf(amax, fmaxf(fabsf(a), fabsf(b)));
              ow[e] = p.out_f16 ? pack_half2(a, b) : pack_bf162(a, b);
            }
            *reinterpret_cast<uint4 *>(buf + lane * 64 + ((v ^ ((lane >> 1) & 3)) * 16)) = o;
          }
          fence_proxy_async_smem();  // the generic-proxy writes, before the bulk copy reads them
          __syncwarp();
          if (lane == 0)  // lane 0 issues, and later waits for, this warp's stores
            tma_store_2d(first ? &tmO0 : &tmO1, buf, first ? n : n - p.split, m0 + q * 32);
          ++n_stored;
        }
      }
      // An fp16 output (the attention state of a bf16 layer) cannot hold a
      // value above 65504: such a call is reported, not silently saturated.
      if (p.out_f16 && __any_sync(0xffffffffu, amax > 65504.f) && lane == 0 && p.status)
        atomicCAS(p.status, 0, (int)DPP_ERR_RANGE);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
    if (lane == 0) bulk_wait_all();  // every bulk store has landed before the CTA exits
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int BN, int STAGES, bool IN_BF16>
cudaError_t run(const GemmArgs &g, int *status, cudaStream_t s) {
  const CUtensorMapDataType ty = tma_type(g.ta);
  CUtensorMap ma, mb[3];
  {
    const uint64_t dims[2] = {(uint64_t)g.K, (uint64_t)g.M};
    const uint64_t str[1] = {(uint64_t)g.K * 2};
    const uint32_t box[2] = {64, 128};
    if (!encode_tiled(&ma, ty, 2, g.A, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  // one box per weight block and stage: BN rows (gated GELU: BN/2 value rows
  // and BN/2 gate rows)
  for (int i = 0; i < 3; ++i) {
    const void *b = g.B[i] ? g.B[i] : g.B[0];
    const uint64_t dims[2] = {(uint64_t)g.K, (uint64_t)g.b_rows};
    const uint64_t str[1] = {(uint64_t)g.K * 2};
    const uint32_t box[2] = {64, (uint32_t)(g.geglu ? BN / 2 : BN)};
    if (!encode_tiled(&mb[i], ty, 2, b, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  // output tensor maps (16-bit, 32 x 32 boxes, 64-byte swizzle): out0 holds
  // columns [0, split) (all N without a second destination), out1 [split, N)
  CUtensorMap mo[2];
  {
    const CUtensorMapDataType to = tma_type(g.to);
    const int w0 = g.out1 ? g.split : g.N;
    const uint64_t d0[2] = {(uint64_t)w0, (uint64_t)g.M};
    const uint64_t s0[1] = {(uint64_t)g.ld0 * 2};
    const uint32_t box[2] = {32, 32};
    if (!encode_tiled(&mo[0], to, 2, g.out0, d0, s0, box, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
    mo[1] = mo[0];
    if (g.out1 && g.N > g.split) {
      const uint64_t d1[2] = {(uint64_t)(g.N - g.split), (uint64_t)g.M};
      const uint64_t s1[1] = {(uint64_t)g.ld1 * 2};
      if (!encode_tiled(&mo[1], to, 2, g.out1, d1, s1, box, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    }
  }
  // residual prefetch map over out0: one box of the tile's columns x 128
  // rows (64-column boxes if the wide box cannot be encoded)
  CUtensorMap mr = mo[0];
  int pf_boxes = 0, pf_cols = 0;
  if (g.accumulate) {
    const CUtensorMapDataType to = tma_type(g.to);
    const int w0 = g.out1 ? g.split : g.N;
    const uint64_t d0[2] = {(uint64_t)w0, (uint64_t)g.M};
    const uint64_t s0[1] = {(uint64_t)g.ld0 * 2};
    const uint32_t cols = g.geglu ? BN / 2 : BN;
    const uint32_t box[2] = {cols, 128};
    if (encode_tiled(&mr, to, 2, g.out0, d0, s0, box, CU_TENSOR_MAP_SWIZZLE_NONE)) {
      pf_boxes = 1;
      pf_cols = (int)cols;
    } else {
      const uint32_t box64[2] = {64, 128};
      if (!encode_tiled(&mr, to, 2, g.out0, d0, s0, box64, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
      pf_boxes = (int)cols / 64;
      pf_cols = 64;
    }
  }
  const int tpb = (g.b_rows + BN - 1) / BN;
  const int n_tiles = g.geglu ? (g.N + BN / 2 - 1) / (BN / 2)
                              : ((g.N + g.b_rows - 1) / g.b_rows) * tpb;
  GemmTcParams p{g.M, g.N, g.K, g.b_rows, g.out0, g.ld0, g.split, g.out1, g.ld1,
                 g.to == E_F16 ? 1 : 0, (g.M + BM - 1) / BM, n_tiles, tpb, status,
                 g.bias, g.accumulate ? 1 : 0, g.geglu ? 1 : 0, pf_boxes, pf_cols,
                 g.cast_src, g.cast_dst, g.cast_n};
  // stages, 1024-byte alignment slack, the epilogue warps' staging buffers, barriers
  constexpr size_t smem = (size_t)STAGES * (BM * BK * 2 + BN * BK * 2) + 1024 +
                          (size_t)kEpiWarps * 2 * kStageOut + 256;
  static_assert(smem <= 227 * 1024, "shared memory budget");
  auto k = gemm_tc_kernel<BN, STAGES, IN_BF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int tiles = p.m_tiles * p.n_tiles;
  const int grid = tiles < sms ? tiles : sms;
  k<<<grid, kThreads, smem, s>>>(ma, mb[0], mb[1], mb[2], mo[0], mo[1], mr, p);
  return cudaGetLastError();
}

__global__ void cast_bf16_f16_kernel(const __nv_bfloat16 *__restrict__ in, __half *__restrict__ out,
                                     size_t n) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    out[i] = __float2half_rn(__bfloat162float(in[i]));
}

}  // namespace

namespace {

// Self-test of the bounded mbarrier wait every tensor-core kernel uses: one
// thread waits for the first phase of a barrier nobody arrives on; after the
// wait limit mbar_wait records DPP_ERR_TIMEOUT and returns false.
__global__ void mbar_wait_selftest_kernel(int *status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0u, &abort_flag, status);
}

}  // namespace

cudaError_t launch_wait_selftest_mbarrier(cudaStream_t s) {
  mbar_wait_selftest_kernel<<<1, 32, 0, s>>>(device_status_ptr());
  return cudaGetLastError();
}

cudaError_t launch_cast_bf16_f16(const void *in, void *out, size_t n, cudaStream_t s) {
  size_t blocks = (n + 255) / 256;
  if (blocks > 1184) blocks = 1184;
  if (blocks < 1) blocks = 1;
  cast_bf16_f16_kernel<<<(unsigned)blocks, 256, 0, s>>>((const __nv_bfloat16 *)in,
                                                        (__half *)out, n);
  return cudaGetLastError();
}

bool gemm_tc_supported(const GemmArgs &g) {
  if (g.cast_n && (g.cast_n % 8 || !g.cast_src || !g.cast_dst ||
                   (reinterpret_cast<uintptr_t>(g.cast_src) & 15u) ||
                   (reinterpret_cast<uintptr_t>(g.cast_dst) & 15u)))
    return false;
  const bool in16 = (g.ta == E_BF16 || g.ta == E_F16) && g.ta == g.tb;
  const bool out16 = g.to == E_BF16 || g.to == E_F16;
  if (g.bias && (reinterpret_cast<uintptr_t>(g.bias) & 15u)) return false;  // float4 loads
  if (g.geglu)  // value / gate blocks of N rows; bf16 output; tiles of 64 or 128 columns
    return in16 && g.to == E_BF16 && g.K % 8 == 0 && g.N % 64 == 0 && g.b_rows == g.N &&
           g.split == g.N && g.out1 == nullptr && g.ld0 % 8 == 0 && g.M > 0 && g.B[1];
  return in16 && out16 && g.K % 8 == 0 && g.b_rows % 64 == 0 && g.N % 32 == 0 &&
         g.split % 32 == 0 && g.ld0 % 8 == 0 && (g.out1 == nullptr || g.ld1 % 8 == 0) &&
         (g.N + g.b_rows - 1) / g.b_rows <= 3 && g.M > 0;
}

cudaError_t launch_gemm_tc(const GemmArgs &g, int *status, cudaStream_t s) {
  if (!gemm_tc_supported(g)) return cudaErrorNotSupported;
  const bool bf = g.ta == E_BF16;
  if (g.geglu) {  // a tile holds BN/2 value and BN/2 gate columns
    if (g.N % 128 == 0)
      return bf ? run<256, 4, true>(g, status, s) : run<256, 4, false>(g, status, s);
    return bf ? run<128, 6, true>(g, status, s) : run<128, 6, false>(g, status, s);
  }
  // 256-column tiles: each 48 KB stage feeds 512 cycles of MMA (a 128-column
  // tile's 32 KB feed 256), and a ragged last tile runs a narrower MMA
  return bf ? run<256, 4, true>(g, status, s) : run<256, 4, false>(g, status, s);
}

}  // namespace dpp

// Displaced attention core on tcgen05 (DistriSelfAttentionPP, section
// 注意力机制拆分 of the DistriFusion developer guide): a band's queries attend
// over the fresh K/V of their own band and the stale K/V of every other band.
// Also serves cross-attention (one fresh segment, the text context).
//
// O = softmax(Q K^T / 8) V per (batch, head, band), head_dim 64, fp16 Q/K/V/P,
// fp32 accumulators and softmax.  One CTA handles two 128-query tiles of one
// band so that one tile's softmax overlaps the other tile's MMAs:
//   warp 0        TMA producer (converged warp, elected lane): both Q tiles once, then
//                 per tile of 128 keys ONE box of the K/V state viewed as
//                 {channel, token, K or V}, landing as the K tile followed by
//                 the V tile, into a 5-deep ring (128-byte swizzle): one copy
//                 and one barrier pair per key tile.  The key range is
//                 walked segment by segment -- own band from the fresh state,
//                 the keys before and after it from the stale state -- so each
//                 tile has one source; a segment's ragged last tile is aligned
//                 to end at the segment end (masking its leading columns), so
//                 no tile reads outside its segment when the segment holds at
//                 least 128 keys.
//   warps 1, 2    one MMA-issuing warp per query tile t (warp 1 also owns
//                 the TMEM allocation); the warp stays converged and one
//                 elected lane issues each MMA:
//                   S_t = Q_t K^T   (M 128, N 128, K 64), both from shared memory,
//                   O_t += P_t V    (M 128, N 64, K 128), P_t read from tensor
//                                   memory, V from shared memory (MN-major);
//                 separate issuers keep one tile's wait for its softmax from
//                 stalling the other tile's MMAs.
//   warps 3..18   softmax, eight warps per query tile, two threads per query
//                 row: a warp reads 16 TMEM lanes (rows) with the 16x32bx2
//                 access shape, its lanes 0..15 taking keys 0..63 of a row
//                 and lanes 16..31 keys 64..127, so every scheduler runs four
//                 softmax warps.  The two halves of a row agree on its max
//                 with one shuffle; each keeps its own partial row sum.  Row
//                 max (3-input max, four independent chains), p = 2^(s*scale
//                 - m) with the scale folded into paired fp32 FMAs and the
//                 exponentials taken as fp16 pairs on the special-function
//                 unit (P's fp16 pairs come out directly), running sum in
//                 paired fp16 adds folded into fp32 per tile, P written back
//                 to tensor memory; the reference max m only moves when a row
//                 max exceeds it by 4 (in log2 units), so the O accumulator in
//                 TMEM is rarely rescaled; final O / l stored as fp16.
//
// Tensor memory per query tile t (256 columns at t * 256): S in columns
// [0, 128), O in [128, 192), P in [192, 256) (fp16 pairs).  Keeping P out of
// shared memory leaves the shared-memory bandwidth to the MMA operand reads
// (Q, K, V), and lets a tile's exponentials run while the previous PV MMA
// still reads the previous P.
#include "tc_common.cuh"

namespace dpp {
namespace {

using namespace tc;

constexpr int kThreads = 608;  // 19 warps: producer, two MMA issuers, 16 softmax
constexpr int KVS = 5;  // K/V ring depth (a stage holds a key tile's K and V)
constexpr uint32_t TILE_BYTES = 128 * 128;  // 128 rows x 64 fp16
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_KV = OFF_Q + 2 * TILE_BYTES;
constexpr uint32_t OFF_BAR = OFF_KV + KVS * 2 * TILE_BYTES;
constexpr uint32_t OFF_TAB = OFF_BAR + 512;
constexpr int kTabTiles = 1024;  // key tiles described in shared memory (more: computed)
constexpr uint32_t SMEM_BYTES = OFF_TAB + kTabTiles * 16 + 1024;
constexpr float kRescaleThreshold = 4.f;

struct AttnTcParams {
  int B, Nq, Nkv, C, P;
  int has_stale;
  int band_local;  // keys of the query's own band only (naive patches)
  int tpb;  // CTAs per band (two query tiles each)
  void *o;
  int *status;
  float scale_log2;
};

struct __align__(16) KvTile {
  int kv0, vlo, vhi, fresh;
};

struct Segs {
  int lo[3], hi[3], fresh[3], ntiles[3], total;
};

__device__ __forceinline__ Segs make_segs(const AttnTcParams &p, int band) {
  Segs s;
  if (p.band_local && p.Nkv == p.Nq) {  // the band's own (fresh) keys only
    const int Np = p.Nq / p.P;
    s.lo[0] = band * Np; s.hi[0] = (band + 1) * Np; s.fresh[0] = 1;
    s.lo[1] = s.hi[1] = s.lo[2] = s.hi[2] = 0;
    s.fresh[1] = s.fresh[2] = 0;
  } else if (p.has_stale && p.Nkv == p.Nq) {
    const int Np = p.Nq / p.P;
    s.lo[0] = band * Np;  s.hi[0] = (band + 1) * Np; s.fresh[0] = 1;
    s.lo[1] = 0;          s.hi[1] = band * Np;       s.fresh[1] = 0;
    s.lo[2] = (band + 1) * Np; s.hi[2] = p.Nkv;      s.fresh[2] = 0;
  } else {
    s.lo[0] = 0; s.hi[0] = p.Nkv; s.fresh[0] = 1;
    s.lo[1] = s.hi[1] = s.lo[2] = s.hi[2] = 0;
    s.fresh[1] = s.fresh[2] = 0;
  }
  s.total = 0;
  for (int i = 0; i < 3; ++i) {
    const int L = s.hi[i] - s.lo[i];
    s.ntiles[i] = L > 0 ? (L + 127) / 128 : 0;
    s.total += s.ntiles[i];
  }
  return s;
}

__device__ __forceinline__ KvTile tile_of(const Segs &s, int j) {
  // segment i holding tile j, selected without indexing the arrays by a
  // runtime value (which would put them in local memory)
  const bool in0 = j < s.ntiles[0];
  const bool in1 = !in0 && j < s.ntiles[0] + s.ntiles[1];
  const int lo = in0 ? s.lo[0] : (in1 ? s.lo[1] : s.lo[2]);
  const int hi = in0 ? s.hi[0] : (in1 ? s.hi[1] : s.hi[2]);
  const int nt = in0 ? s.ntiles[0] : (in1 ? s.ntiles[1] : s.ntiles[2]);
  const int jj = in0 ? j : (in1 ? j - s.ntiles[0] : j - s.ntiles[0] - s.ntiles[1]);
  const int L = hi - lo;
  KvTile t;
  t.fresh = in0 ? s.fresh[0] : (in1 ? s.fresh[1] : s.fresh[2]);
  if (L < 128) {
    t.kv0 = lo; t.vlo = 0; t.vhi = L;
  } else if (jj == nt - 1 && (L & 127)) {
    t.kv0 = hi - 128; t.vlo = lo + 128 * jj - t.kv0; t.vhi = 128;
  } else {
    t.kv0 = lo + 128 * jj; t.vlo = 0; t.vhi = 128;
  }
  return t;
}

// 2^x for an fp16 pair on the special-function unit
__device__ __forceinline__ uint32_t ex2_f16x2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// ---- 3-input max (sm_100 family)
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// ---- grouped MMA issue: one asm block, one elected lane, the whole group.
// S = Q K^T over K = 64 (four K16 steps; descriptors advance 32 bytes per
// step inside the 128-byte swizzled rows), then the two commits.
__device__ __forceinline__ void issue_s(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc,
                                        uint64_t *done, uint64_t *slot_free) {
  asm volatile(
      "{\n\t.reg .pred e, pf, pt;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
      "setp.ne.b32 pf, 0, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
      "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"
      "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, pt;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, pt;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, pt;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%4];\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t}" ::"r"(d),
      "l"(ad), "l"(bd), "r"(idesc), "r"(smem_u32(done)), "r"(smem_u32(slot_free))
      : "memory");
}

// O (+)= P V over K = 128 keys: eight K16 steps, P from tensor memory (8
// columns of fp16 pairs per step), V from shared memory MN-major (16 rows of
// 128 bytes = 2048 bytes, i.e. 128 descriptor units, per step); `first`
// starts the accumulator instead of adding to it.  Then the two commits.
__device__ __forceinline__ void issue_pv(uint32_t d, uint32_t a, uint64_t bd, uint32_t idesc,
                                         uint32_t first, uint64_t *done, uint64_t *slot_free) {
  asm volatile(
      "{\n\t.reg .pred e, p0, pt;\n\t.reg .b64 b1, b2, b3, b4, b5, b6, b7;\n\t"
      ".reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t"
      "setp.eq.b32 p0, %4, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
      "add.s32 a1, %1, 8;\n\tadd.s32 a2, %1, 16;\n\tadd.s32 a3, %1, 24;\n\t"
      "add.s32 a4, %1, 32;\n\tadd.s32 a5, %1, 40;\n\tadd.s32 a6, %1, 48;\n\t"
      "add.s32 a7, %1, 56;\n\t"
      "add.s64 b1, %2, 128;\n\tadd.s64 b2, %2, 256;\n\tadd.s64 b3, %2, 384;\n\t"
      "add.s64 b4, %2, 512;\n\tadd.s64 b5, %2, 640;\n\tadd.s64 b6, %2, 768;\n\t"
      "add.s64 b7, %2, 896;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, pt;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, pt;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, pt;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b4, %3, pt;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b5, %3, pt;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b6, %3, pt;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], b7, %3, pt;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t}" ::"r"(d),
      "r"(a), "l"(bd), "r"(idesc), "r"(first), "r"(smem_u32(done)), "r"(smem_u32(slot_free))
      : "memory");
}

// One elected lane of a converged warp arrives on `bar`.
__device__ __forceinline__ void mbar_arrive_w(uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

// Warp-uniform bounded wait: every lane waits, then the warp agrees.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          int *status) {
  const bool ok = mbar_wait(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmF,
               const __grid_constant__ CUtensorMap tmS, const AttnTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  uint64_t *q_full = bars;
  uint64_t *kv_full = bars + 1, *kv_empty = kv_full + KVS;
  uint64_t *s_full = kv_empty + KVS, *s_empty = s_full + 2;
  uint64_t *p_full = s_empty + 2, *p_empty = p_full + 2;
  uint64_t *o_final = p_empty + 2, *drain = o_final + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int band = blockIdx.x / p.tpb, part = blockIdx.x % p.tpb;
  const int head = blockIdx.y, b = blockIdx.z;
  const int Np = p.Nq / p.P;
  const int q0 = band * Np + part * 256;
  const int qend = (band + 1) * Np;
  const Segs segs = make_segs(p, band);
  const int T = segs.total;
  // the band's last CTA may hold a single query tile (the band's tail)
  const int ntile = q0 + 128 < qend ? 2 : 1;
  // the key tiles of this band, walked once here instead of in every warp
  const KvTile *tab = reinterpret_cast<const KvTile *>(smem + OFF_TAB);
  for (int j = threadIdx.x; j < T && j < kTabTiles; j += blockDim.x)
    reinterpret_cast<KvTile *>(smem + OFF_TAB)[j] = tile_of(segs, j);
  auto kv_tile = [&](int j) -> KvTile { return j < kTabTiles ? tab[j] : tile_of(segs, j); };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    // a K or V slot is free once every query tile's MMAs have read it
    // (S and PV MMAs of every query tile)
    for (int i = 0; i < KVS; ++i) { mbar_init(&kv_full[i], 1); mbar_init(&kv_empty[i], 2 * ntile); }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&s_empty[t], 8);  // one arrival per softmax warp of the tile
      mbar_init(&p_full[t], 8);
      mbar_init(&p_empty[t], 1);
      mbar_init(&o_final[t], 1);
      mbar_init(&drain[t], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmF);
    prefetch_tmap(&tmS);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {  // ------------------------------------------------ producer
    // The whole warp runs the loop (warp-uniform operands); one elected lane
    // issues each copy.
    uint32_t kv_armed = 0, kv_par = 0;
    mbar_arrive_expect_tx_w(q_full, ntile * TILE_BYTES);
    tma_load_2d_w(smem + OFF_Q, &tmQ, q_full, head * 64, b * p.Nq + q0);
    if (ntile == 2)
      tma_load_2d_w(smem + OFF_Q + TILE_BYTES, &tmQ, q_full, head * 64, b * p.Nq + q0 + 128);
    for (int j = 0; j < T; ++j) {
      const KvTile kt = kv_tile(j);
      const CUtensorMap *m = kt.fresh ? &tmF : &tmS;
      const int row = b * p.Nkv + kt.kv0;
      const int ks = j % KVS;
      const uint32_t kph = (j / KVS) & 1;
      if (!mbar_wait_w(&kv_empty[ks], kph ^ 1u, abort_flag, p.status)) break;
      mbar_arrive_expect_tx_w(&kv_full[ks], 2 * TILE_BYTES);
      kv_armed |= 1u << ks;
      kv_par = (kv_par & ~(1u << ks)) | (kph << ks);
      // one box: the tile's K rows, then its V rows
      tma_load_3d_w(smem + OFF_KV + ks * 2 * TILE_BYTES, m, &kv_full[ks], head * 64, row, 0);
    }
    if (*abort_flag) {  // copies in flight must land before the CTA exits
      mbar_drain(q_full, 0);
      for (int i = 0; i < KVS; ++i)
        if ((kv_armed >> i) & 1u) mbar_drain(&kv_full[i], (kv_par >> i) & 1u);
    }
  } else if ((warp == 1 || warp == 2) && warp - 1 < ntile) {  // --- MMA issuer of tile t
    // Each query tile has its own issuing warp, so one tile's wait for its
    // softmax never holds back the other tile's MMAs.  Per key tile j:
    // S(j) = Q K(j)^T as soon as the softmax has read S(j-1), then
    // O += P(j-1) V(j-1) once it has written P(j-1).  The warp stays
    // converged; one elected lane issues each MMA and commit.
    const int t = warp - 1;
    constexpr uint32_t IDESC_S = idesc_f16(128, 128, false);
    constexpr uint32_t IDESC_O = idesc_f16(128, 64, false, true);
    const uint32_t sQ = smem_u32(smem + OFF_Q) + t * TILE_BYTES;
    const uint32_t sK = smem_u32(smem + OFF_KV), sV = sK + TILE_BYTES;
    const uint32_t dS = tmem + t * 256, dO = dS + 128, aP = dS + 192;
    auto pv = [&](int j) -> bool {  // O += P(j) V(j)
      // (the stage's K/V landed before S(j) was issued and stays until this
      // PV has read it)
      if (!mbar_wait_w(&p_full[t], j & 1, abort_flag, p.status)) return false;
      tc_fence_after();
      issue_pv(dO, aP, desc_sw128_mnmajor(sV + (j % KVS) * 2 * TILE_BYTES, 1024), IDESC_O,
               j == 0 ? 1u : 0u, &p_empty[t], &kv_empty[j % KVS]);
      return true;
    };
    bool ok = mbar_wait_w(q_full, 0, abort_flag, p.status);
    const uint64_t ad = desc_sw128_kmajor(sQ);
    for (int j = 0; ok && j < T; ++j) {
      ok = mbar_wait_w(&kv_full[j % KVS], (j / KVS) & 1, abort_flag, p.status) &&
           mbar_wait_w(&s_empty[t], (j & 1) ^ 1u, abort_flag, p.status);
      if (!ok) break;
      tc_fence_after();
      issue_s(dS, ad, desc_sw128_kmajor(sK + (j % KVS) * 2 * TILE_BYTES), IDESC_S, &s_full[t],
              &kv_empty[j % KVS]);
      if (j > 0) ok = pv(j - 1);
    }
    if (ok && T > 0) ok = pv(T - 1);
    if (ok) {
      mma_commit_w(&o_final[t]);
    } else {  // nothing may still be writing TMEM when it is freed
      mma_commit_w(&drain[t]);
      mbar_drain(&drain[t], 0);
    }
  } else if (warp >= 3 && (warp - 3) >> 3 < ntile) {  // -------------------- softmax
    const int sw = warp - 3;                // 0..15
    const int t = sw >> 3;                  // query tile
    const int quad = warp & 3;              // TMEM lanes this warp may access: 32*quad..
    const int h16 = (sw >> 2) & 1;          // which 16 of them
    const int half = lane >> 4;             // keys [64*half, 64*half + 64) of each tile
    const int row = quad * 32 + h16 * 16 + (lane & 15);
    const uint32_t lane_base = (uint32_t)(quad * 32 + h16 * 16) << 16;
    const uint32_t tS = tmem + lane_base + t * 256, tO = tS + 128, tP = tS + 192;
    float m_ref = -INFINITY, l = 0.f;  // l: this thread's half of the row sum
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const KvTile kt = kv_tile(j);
      if (!warp_wait(&s_full[t], j & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld16x2_32<64>(tS, *reinterpret_cast<uint32_t (*)[32]>(&sr[0]));
      tmem_ld16x2_32<64>(tS + 32, *reinterpret_cast<uint32_t (*)[32]>(&sr[32]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive_w(&s_empty[t]);
      if (kt.vlo != 0 || kt.vhi != 128) {  // ragged tile (uniform branch): mask
        const int k0 = half * 64;
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (k0 + i < kt.vlo || k0 + i >= kt.vhi) sr[i] = 0xff800000u;  // -inf
      }
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < 64; i += 8)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          m4[k] = max3f(m4[k], __uint_as_float(sr[i + 2 * k]), __uint_as_float(sr[i + 2 * k + 1]));
      float mh = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      mh = fmaxf(mh, __shfl_xor_sync(0xffffffffu, mh, 16));  // the row's other half
      const float mx = mh * p.scale_log2;
      float corr = 1.f;
      if (mx > m_ref + kRescaleThreshold) {  // both halves of the row decide alike
        corr = ex2_approx(m_ref - mx);  // 0 on the first tile
        m_ref = mx;
      }
      l *= corr;
      // p = 2^(s * scale - m_ref): the scaled argument of each pair of scores
      // (paired fp32 FMA) is rounded to an fp16 pair and exponentiated on the
      // special-function unit as a pair (ex2.approx.f16x2), which yields P's
      // fp16 pairs directly: two exponentials per instruction.  With m_ref at
      // most kRescaleThreshold below the running max, every argument is <= 4,
      // where fp16 resolves it to 2^-9 (p within 0.07 %).  The half-row sum
      // is taken over the fp16 pairs (four chains of paired fp16 adds, each
      // pair's sum at most 64 x 16) and added to l in fp32.
      const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
      const float2 nm2 = make_float2(-m_ref, -m_ref);
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 x = __ffma2_rn(
            make_float2(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])), sc2, nm2);
        pk[i] = ex2_f16x2(pack_half2(x.x, x.y));
      }
      __half2 acc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] = *reinterpret_cast<const __half2 *>(&pk[k]);
#pragma unroll
      for (int i = 4; i < 32; ++i)
        acc[i & 3] = __hadd2(acc[i & 3], *reinterpret_cast<const __half2 *>(&pk[i]));
      {
        const float2 a0 = __half22float2(acc[0]), a1 = __half22float2(acc[1]);
        const float2 a2 = __half22float2(acc[2]), a3 = __half22float2(acc[3]);
        l += ((a0.x + a0.y) + (a1.x + a1.y)) + ((a2.x + a2.y) + (a3.x + a3.y));
      }
      // PV(j-1) must be done reading P and writing O before both are rewritten
      if (!warp_wait(&p_empty[t], (j - 1) & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      tmem_st16x2_32<32>(tP, pk);  // lanes 0..15: P columns 0..31, lanes 16..31: 32..63
      if (j > 0 && __any_sync(0xffffffffu, corr != 1.f)) {  // rescale O (rare)
        uint32_t r[32];
        tmem_ld16x2_32<32>(tO, r);  // each half of the row rescales 32 of its 64 columns
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * corr);
        tmem_st16x2_32<32>(tO, r);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_w(&p_full[t]);
    }
    if (ok && warp_wait(&o_final[t], 0, abort_flag, p.status)) {
      tc_fence_after();
      const int q = q0 + t * 128 + row;
      const float inv = 1.f / (l + __shfl_xor_sync(0xffffffffu, l, 16));
      uint32_t r[32];
      tmem_ld16x2_32<32>(tO, r);  // lanes 0..15: O columns 0..31, lanes 16..31: 32..63
      tmem_wait_ld();
      if (q < qend) {
        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__half *>(p.o) +
                                               ((size_t)b * p.Nq + q) * p.C + head * 64 +
                                               32 * half);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 o;
          uint32_t *ow = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            ow[e] = pack_half2(__uint_as_float(r[8 * v + 2 * e]) * inv,
                               __uint_as_float(r[8 * v + 2 * e + 1]) * inv);
          dst[v] = o;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool attn_tc_supported(const AttnArgs &a) {
  return a.te == E_F16 && a.C % 64 == 0 && a.heads * 64 == a.C && a.Nq % a.P == 0 &&
         (a.P == 1 || a.Nkv == a.Nq) && a.Nkv > 0 && a.Nq > 0;
}

cudaError_t launch_attn_tc(const AttnArgs &a, int *status, cudaStream_t s) {
  if (!attn_tc_supported(a)) return cudaErrorNotSupported;
  CUtensorMap mq, mf, ms;
  {
    const uint64_t dims[2] = {(uint64_t)a.C, (uint64_t)a.B * a.Nq};
    const uint64_t str[1] = {(uint64_t)a.C * 2};
    const uint32_t box[2] = {64, 128};
    if (!encode_tiled(&mq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.q, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  // K/V state [B * Nkv][K | V] viewed as {channel, token, K or V}: one box
  // of 64 channels x 128 tokens x both planes lands as the K tile followed
  // by the V tile
  const uint64_t dims[3] = {(uint64_t)a.C, (uint64_t)a.B * a.Nkv, 2};
  const uint64_t str[2] = {(uint64_t)a.C * 4, (uint64_t)a.C * 2};
  const uint32_t box[3] = {64, 128, 2};
  if (!encode_tiled(&mf, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, a.kv_fresh, dims, str, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_tiled(&ms, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                    a.kv_stale ? a.kv_stale : a.kv_fresh, dims, str, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int Np = a.Nq / a.P;
  AttnTcParams p{a.B,       a.Nq, a.Nkv,  a.C, a.P, a.kv_stale != nullptr ? 1 : 0, a.band_local,
                 (Np + 255) / 256, a.o, status, 0.125f * 1.4426950408889634f};
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(a.P * p.tpb), (unsigned)a.heads, (unsigned)a.B);
  attn_tc_kernel<<<grid, kThreads, SMEM_BYTES, s>>>(mq, mf, ms, p);
  return cudaGetLastError();
}

}  // namespace dpp

// Attention core over a short key sequence on tcgen05: cross-attention over
// the text context (DistriCrossAttentionPP of the DistriFusion developer
// guide, section 注意力机制拆分: every device holds the whole context, so a
// band's queries attend over the same keys), or any attention whose keys fit
// one tile (at most 128) and that has no stale bands.
//
// O = softmax(Q K^T / 8) V per (batch, head), head_dim 64, fp16 Q/K/V/P,
// fp32 scores and accumulators.  With every key in one tile the softmax is a
// single exact pass (row max, exponentials, row sum) and needs no running
// rescale.  The work is the stream of 128-query tiles, so the kernel is
// persistent: one CTA per SM walks a contiguous range of (batch, head,
// query tile) items, keeps the head's K and V in shared memory while the
// range stays on that head, and streams the query tiles through a ring:
//   warp 0      TMA producer (converged warp, elected lane): the K and V of
//               a (batch, head) as one box of {64 channels, keys rounded up
//               to 16, K and V planes} into one of two slots; each Q tile
//               {64 channels, 128 queries} into a 4-deep ring;
//   warp 1      TMEM owner and MMA issuer: S_i = Q_i K^T (M 128, N keys
//               rounded to 16, K 64) into TMEM buffer i mod NB once that
//               buffer's previous tile is out, and once the softmax has
//               written P_i, O_i = P_i V (M 128, N 64, K keys; P from TMEM,
//               V MN-major from shared memory), each group of instructions
//               issued by one elected lane;
//   warps 2..   NB groups of four warps (NB = 3 when the keys round up to at
//               most 96, else 2), one per TMEM buffer, taking the tiles in
//               turn; one thread per query row: S row from TMEM (read twice:
//               once for the row max, then 32 keys at a time for P), keys
//               past the end masked, p = 2^(s * scale - max) as fp16 pairs on
//               the special-function unit, row sum, P written over the S
//               columns already read; then the tile's O / l as fp16 through
//               shared memory and one bulk tensor store per warp.  The
//               issuer runs S up to NB - 1 tiles ahead of PV, so every group
//               has a tile while the others wait on MMAs or memory.
// TMEM per buffer a (at a * kBuf): S, then P over it, in [0, kSP); O in
// [kSP, kSP + 64).
#include "tc_common.cuh"

namespace dpp {
namespace {

using namespace tc;

constexpr int QS = 4;           // Q ring depth
constexpr uint32_t QTILE = 128 * 128;   // 128 queries x 64 fp16
constexpr uint32_t KVSLOT = 2 * 128 * 128;  // K and V of up to 128 keys
constexpr uint32_t kStageBytes = 32 * 128;  // one warp's 32 output rows x 64 fp16
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_KV = OFF_Q + QS * QTILE;
constexpr uint32_t OFF_STAGE = OFF_KV + 2 * KVSLOT;  // one staging buffer per softmax warp

// NB TMEM buffers, each served by its own group of four softmax warps.  A
// buffer holds S (keys rounded up to 16) with P written over it, then O:
// 96 + 64 columns when the keys round to at most 96 (three buffers fit the
// 512 columns), 128 + 64 otherwise (two).
template <int NB>
struct XCfg {
  static constexpr int kThreads = 64 + 128 * NB;
  static constexpr uint32_t kSP = NB == 3 ? 96 : 128;  // S / P columns
  static constexpr uint32_t kBuf = kSP + 64;           // + O
  static constexpr uint32_t kOffBar = OFF_STAGE + 4 * NB * kStageBytes;
  static constexpr uint32_t kSmem = kOffBar + 256 + 1024;
};

struct XattnParams {
  int B, Nq, Nkv, C, heads;
  int tpq;    // 128-query tiles per (batch, head)
  int items;  // B * heads * tpq
  int nkv16;  // keys rounded up to a multiple of 16 (the MMA's N and K)
  void *o;
  int *status;
  float scale_log2;
};

// One elected lane of a converged warp arrives on `bar`.
__device__ __forceinline__ void arrive_w(uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ float max3f(float a, float b, float c) {  // 3-input max
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ uint32_t ex2_h2(uint32_t x) {  // 2^x for an fp16 pair
  uint32_t y;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// S = Q K^T over head_dim 64 (four K16 steps, descriptors advancing 32 bytes
// inside the 128-byte swizzled rows) and its two commits, as one group
// issued by one elected lane: a separate elect per instruction costs the
// issuing warp far more than the instructions themselves.
__device__ __forceinline__ void issue_s4(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc,
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

// O = P V over n16 K16 steps (1..8; 16 keys each: 8 columns of fp16 pairs of
// P in TMEM, 16 rows = 2048 bytes = 128 descriptor units of MN-major V),
// then the commit, as one group with one elected lane.
__device__ __forceinline__ void issue_pv_n(uint32_t d, uint32_t a, uint64_t bd, uint32_t idesc,
                                           int n16, uint64_t *done) {
  asm volatile(
      "{\n\t.reg .pred e, pf, pt, q1, q2, q3, q4, q5, q6, q7;\n\t"
      ".reg .b64 b1, b2, b3, b4, b5, b6, b7;\n\t.reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t"
      "setp.ne.b32 pf, 0, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
      "add.s32 a1, %1, 8;\n\tadd.s32 a2, %1, 16;\n\tadd.s32 a3, %1, 24;\n\t"
      "add.s32 a4, %1, 32;\n\tadd.s32 a5, %1, 40;\n\tadd.s32 a6, %1, 48;\n\t"
      "add.s32 a7, %1, 56;\n\t"
      "add.s64 b1, %2, 128;\n\tadd.s64 b2, %2, 256;\n\tadd.s64 b3, %2, 384;\n\t"
      "add.s64 b4, %2, 512;\n\tadd.s64 b5, %2, 640;\n\tadd.s64 b6, %2, 768;\n\t"
      "add.s64 b7, %2, 896;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.gt.and.s32 q1, %4, 1, e;\n\tsetp.gt.and.s32 q2, %4, 2, e;\n\t"
      "setp.gt.and.s32 q3, %4, 3, e;\n\tsetp.gt.and.s32 q4, %4, 4, e;\n\t"
      "setp.gt.and.s32 q5, %4, 5, e;\n\tsetp.gt.and.s32 q6, %4, 6, e;\n\t"
      "setp.gt.and.s32 q7, %4, 7, e;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pf;\n\t"
      "@q1 tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, pt;\n\t"
      "@q2 tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, pt;\n\t"
      "@q3 tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, pt;\n\t"
      "@q4 tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b4, %3, pt;\n\t"
      "@q5 tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b5, %3, pt;\n\t"
      "@q6 tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b6, %3, pt;\n\t"
      "@q7 tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], b7, %3, pt;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t}" ::"r"(d),
      "r"(a), "l"(bd), "r"(idesc), "r"(n16), "r"(smem_u32(done))
      : "memory");
}

// Shared -> global tiled bulk store (3-D) by the calling thread, committed
// as a bulk async-group of that thread; elements outside the tensor map's
// extent are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int c0,
                                             int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];\n\t"
      "cp.async.bulk.commit_group;" ::"l"(map),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}


template <int NB>
__global__ void __launch_bounds__(XCfg<NB>::kThreads, 1)
xattn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                const __grid_constant__ CUtensorMap tmO, const XattnParams p) {
  using Cfg = XCfg<NB>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
  uint64_t *q_full = bars, *q_empty = q_full + QS;
  uint64_t *kv_full = q_empty + QS, *kv_empty = kv_full + 2;
  uint64_t *s_full = kv_empty + 2, *p_full = s_full + NB;
  uint64_t *o_full = p_full + NB, *o_free = o_full + NB;
  uint64_t *drain = o_free + NB;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int begin = (int)((long long)p.items * blockIdx.x / gridDim.x);
  const int end = (int)((long long)p.items * (blockIdx.x + 1) / gridDim.x);
  const uint32_t kv_plane = (uint32_t)p.nkv16 * 128;  // bytes of the K plane of a slot

  if (threadIdx.x == 0) {
    for (int i = 0; i < QS; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);  // one arrival per softmax warp of the group
      mbar_init(&o_full[i], 1);
      mbar_init(&o_free[i], 4);
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
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmKV);
    prefetch_tmap(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {  // ------------------------------------------------ producer
    int qs = 0;
    uint32_t qph = 0;
    int pairs = 0, cur = -1;
    uint32_t armed = 0, par = 0;  // bits 0..3: Q slots, 4..5: K/V slots (abort drain)
    for (int item = begin; item < end && !*abort_flag; ++item) {
      const int pair = item / p.tpq, qt = item % p.tpq;
      const int b = pair / p.heads, head = pair % p.heads;
      if (pair != cur) {  // the (batch, head)'s K and V, once for its run of items
        const int slot = pairs & 1;
        const uint32_t ph = (pairs >> 1) & 1;
        if (!mbar_wait_w(&kv_empty[slot], ph ^ 1u, abort_flag, p.status)) break;
        mbar_arrive_expect_tx_w(&kv_full[slot], 2 * kv_plane);
        armed |= 1u << (4 + slot);
        par = (par & ~(1u << (4 + slot))) | (ph << (4 + slot));
        tma_load_3d_w(smem + OFF_KV + slot * KVSLOT, &tmKV, &kv_full[slot], head * 64,
                      b * p.Nkv, 0);
        cur = pair;
        ++pairs;
      }
      if (!mbar_wait_w(&q_empty[qs], qph ^ 1u, abort_flag, p.status)) break;
      mbar_arrive_expect_tx_w(&q_full[qs], QTILE);
      armed |= 1u << qs;
      par = (par & ~(1u << qs)) | (qph << qs);
      tma_load_2d_w(smem + OFF_Q + qs * QTILE, &tmQ, &q_full[qs], head * 64,
                    b * p.Nq + qt * 128);
      if (++qs == QS) {
        qs = 0;
        qph ^= 1u;
      }
    }
    if (*abort_flag) {  // copies in flight land before the CTA exits
      for (int i = 0; i < QS; ++i)
        if ((armed >> i) & 1u) mbar_drain(&q_full[i], (par >> i) & 1u);
      for (int i = 0; i < 2; ++i)
        if ((armed >> (4 + i)) & 1u) mbar_drain(&kv_full[i], (par >> (4 + i)) & 1u);
    }
  } else if (warp == 1) {  // ---------------------------------------- MMA issuer
    constexpr int L = NB - 1;  // S runs this many tiles ahead of PV
    const uint32_t idesc_s = idesc_f16(128, p.nkv16, false);
    constexpr uint32_t IDESC_O = idesc_f16(128, 64, false, true);
    const int ksteps = p.nkv16 / 16;
    int qs = 0;
    uint32_t qph = 0;
    int pairs = 0, cur = -1, slot = 0;
    uint32_t hist = 0;  // 2 bits per recent item: its K/V slot, last of its run
    bool ok = true;
    // O_j = P_j V of item j (P over S in buffer j % NB); frees the K/V slot
    // after the last item of a (batch, head)
    auto pv = [&](int j, uint32_t info) -> bool {
      const int a = j % NB;
      if (!mbar_wait_w(&p_full[a], (j / NB) & 1, abort_flag, p.status)) return false;
      tc_fence_after();
      const int kslot = info & 1;
      const uint32_t sV = smem_u32(smem + OFF_KV + kslot * KVSLOT) + kv_plane;
      const uint32_t tb = tmem + a * Cfg::kBuf;
      issue_pv_n(tb + Cfg::kSP, tb, desc_sw128_mnmajor(sV, 1024), IDESC_O, ksteps, &o_full[a]);
      if (info & 2u) mma_commit_w(&kv_empty[kslot]);
      return true;
    };
    int li = 0;
    for (int item = begin; ok && item < end; ++item, ++li) {
      const int pair = item / p.tpq;
      if (pair != cur) {
        slot = pairs & 1;
        if (!mbar_wait_w(&kv_full[slot], (pairs >> 1) & 1, abort_flag, p.status)) break;
        cur = pair;
        ++pairs;
      }
      const int a = li % NB;
      if (!mbar_wait_w(&q_full[qs], qph, abort_flag, p.status)) break;
      // the buffer's previous tile (li - NB) is out: its O read, and so its
      // PV, which read the P written over S, complete
      if (!mbar_wait_w(&o_free[a], ((li / NB) & 1) ^ 1u, abort_flag, p.status)) break;
      tc_fence_after();
      const uint64_t ad = desc_sw128_kmajor(smem_u32(smem + OFF_Q + qs * QTILE));
      const uint64_t bd = desc_sw128_kmajor(smem_u32(smem + OFF_KV + slot * KVSLOT));
      issue_s4(tmem + a * Cfg::kBuf, ad, bd, idesc_s, &s_full[a], &q_empty[qs]);
      if (++qs == QS) {
        qs = 0;
        qph ^= 1u;
      }
      const uint32_t last = item + 1 == end || (item + 1) / p.tpq != pair;
      hist = (hist << 2) | (uint32_t)slot | (last << 1);
      if (li >= L) ok = pv(li - L, (hist >> (2 * L)) & 3u);
    }
    // the last L tiles' PV
    for (int t = L; ok && t >= 1 && !*abort_flag; --t)
      if (li - t >= 0) ok = pv(li - t, (hist >> (2 * (t - 1))) & 3u);
    if (*abort_flag || !ok) {  // nothing may still be writing TMEM when it is freed
      mma_commit_w(drain);
      mbar_drain(drain, 0);
    }
  } else {  // ------------------------------------------------ softmax, epilogue
    const int g = (warp - 2) >> 2;  // group = TMEM buffer
    const int quad = warp & 3;      // TMEM lanes this warp may access
    const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16) + g * Cfg::kBuf;
    const uint32_t tS = tq, tO = tq + Cfg::kSP;  // P is written over S
    const int nch = (p.nkv16 + 31) / 32;  // 32-column chunks of S
    uint8_t *stage = smem + OFF_STAGE + (warp - 2) * kStageBytes;  // this warp's
    const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
    int k = 0;
    for (int item = begin + g; item < end; item += NB, ++k) {
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[g], k & 1, abort_flag, p.status))) break;
      tc_fence_after();
      // pass 1: the row max over the keys (columns past them do not count)
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {  // 64 columns per load group, one wait each
        if (2 * hc >= nch) continue;
        uint32_t sr[64];
#pragma unroll
        for (int c = 0; c < 2; ++c)
          if (2 * hc + c < nch)
            tmem_ld32(tS + 64 * hc + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int base = 64 * hc + 32 * c;
          if (base >= p.Nkv) continue;
          if (base + 32 <= p.Nkv) {  // all keys (uniform branch): 3-input max, four chains
#pragma unroll
            for (int i = 0; i < 32; i += 8)
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4)
                m4[q4] = max3f(m4[q4], __uint_as_float(sr[32 * c + i + 2 * q4]),
                               __uint_as_float(sr[32 * c + i + 2 * q4 + 1]));
          } else {  // the chunk holding the last key
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (base + i < p.Nkv) m4[i & 3] = fmaxf(m4[i & 3], __uint_as_float(sr[32 * c + i]));
          }
        }
      }
      const float m2 = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.scale_log2;
      const float2 nm2 = make_float2(-m2, -m2);
      // pass 2, 32 keys at a time: P = 2^(s * scale - max) as fp16 pairs (ex2
      // of an fp16 pair on the special-function unit) into 16 columns over
      // the S columns already read (chunk c writes [16c, 16c + 16), below
      // the next chunk's [32(c+1), ...)); the row sum in paired fp16 adds,
      // four chains per chunk, folded into fp32
      float l = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (c >= nch) continue;
        uint32_t ch[32];
        tmem_ld32(tS + 32 * c, ch);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int key = 32 * c + 2 * i;
          if (key >= p.nkv16) {  // past the MMA's K: no exponential needed
            pk[i] = 0u;
            continue;
          }
          float s0 = __uint_as_float(ch[2 * i]), s1 = __uint_as_float(ch[2 * i + 1]);
          if (key + 2 > p.Nkv) {  // uniform: only the pairs at the end of the keys
            s0 = key < p.Nkv ? s0 : -INFINITY;
            s1 = key + 1 < p.Nkv ? s1 : -INFINITY;
          }
          const float2 x = __ffma2_rn(make_float2(s0, s1), sc2, nm2);
          pk[i] = ex2_h2(pack_half2(x.x, x.y));
        }
        __half2 acc[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j] = *reinterpret_cast<const __half2 *>(&pk[j]);
#pragma unroll
        for (int i = 4; i < 16; ++i)
          acc[i & 3] = __hadd2(acc[i & 3], *reinterpret_cast<const __half2 *>(&pk[i]));
        const float2 a0 = __half22float2(acc[0]), a1 = __half22float2(acc[1]);
        const float2 a2 = __half22float2(acc[2]), a3 = __half22float2(acc[3]);
        l += ((a0.x + a0.y) + (a1.x + a1.y)) + ((a2.x + a2.y) + (a3.x + a3.y));
        tmem_st16(tS + 16 * c, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      arrive_w(&p_full[g]);
      // epilogue: O / l to global memory (fp16), then the buffer is free
      if (!__all_sync(0xffffffffu, mbar_wait(&o_full[g], k & 1, abort_flag, p.status))) break;
      tc_fence_after();
      uint32_t o[64];
      tmem_ld32(tO, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
      tmem_ld32(tO + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
      tmem_wait_ld();
      tc_fence_before();
      arrive_w(&o_free[g]);
      const int pair = item / p.tpq, qt = item % p.tpq;
      const int b = pair / p.heads, head = pair % p.heads;
      // The warp's 32 rows x 64 fp16 go through its shared-memory staging
      // buffer (128-byte rows, 16-byte units swizzled by the row as the
      // tensor map's 128-byte swizzle does: conflict-free) and one bulk
      // tensor store; the {channel, query, batch} map clips rows past Nq.
      if (k >= 1) {  // this warp's previous store has read the buffer
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
      }
      const float inv = 1.f / l;
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        uint4 w;
        uint32_t *ww = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          ww[e] = pack_half2(__uint_as_float(o[8 * v + 2 * e]) * inv,
                             __uint_as_float(o[8 * v + 2 * e + 1]) * inv);
        *reinterpret_cast<uint4 *>(stage + lane * 128 + ((v ^ (lane & 7)) * 16)) = w;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && qt * 128 + quad * 32 < p.Nq)  // no store that starts past the end
        tma_store_3d(&tmO, stage, head * 64, qt * 128 + quad * 32, b);
    }
    if (lane == 0) bulk_wait_all();  // every bulk store has landed before the CTA exits
    __syncwarp();
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

bool xattn_tc_supported(const AttnArgs &a) {
  return a.te == E_F16 && a.C % 64 == 0 && a.heads * 64 == a.C && a.P == 1 &&
         a.kv_stale == nullptr && a.Nkv >= 1 && a.Nkv <= 128 && a.Nq > 0 && a.B > 0;
}

cudaError_t launch_xattn_tc(const AttnArgs &a, int *status, cudaStream_t s) {
  if (!xattn_tc_supported(a)) return cudaErrorNotSupported;
  const int nkv16 = (a.Nkv + 15) / 16 * 16;
  CUtensorMap mq, mkv, mo;
  {
    const uint64_t dims[2] = {(uint64_t)a.C, (uint64_t)a.B * a.Nq};
    const uint64_t str[1] = {(uint64_t)a.C * 2};
    const uint32_t box[2] = {64, 128};
    if (!encode_tiled(&mq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.q, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    // K/V [B * Nkv][K | V] viewed as {channel, key, K or V}: one box of 64
    // channels x nkv16 keys x both planes lands as K rows then V rows
    const uint64_t dims[3] = {(uint64_t)a.C, (uint64_t)a.B * a.Nkv, 2};
    const uint64_t str[2] = {(uint64_t)a.C * 4, (uint64_t)a.C * 2};
    const uint32_t box[3] = {64, (uint32_t)nkv16, 2};
    if (!encode_tiled(&mkv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, a.kv_fresh, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    // O [B][Nq][C] viewed as {channel, query, batch}: a box of 64 channels x
    // 32 queries is clipped at the end of its own batch's queries
    const uint64_t dims[3] = {(uint64_t)a.C, (uint64_t)a.Nq, (uint64_t)a.B};
    const uint64_t str[2] = {(uint64_t)a.C * 2, (uint64_t)a.Nq * a.C * 2};
    const uint32_t box[3] = {64, 32, 1};
    if (!encode_tiled(&mo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, a.o, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  const int tpq = (a.Nq + 127) / 128;
  XattnParams p{a.B, a.Nq, a.Nkv, a.C, a.heads, tpq, a.B * a.heads * tpq, nkv16, a.o, status,
                0.125f * 1.4426950408889634f};
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = p.items < sms ? p.items : sms;
  // three TMEM buffers (three softmax groups) when S fits 96 columns
  if (nkv16 <= 96) {
    cudaError_t e = cudaFuncSetAttribute(xattn_tc_kernel<3>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)XCfg<3>::kSmem);
    if (e != cudaSuccess) return e;
    xattn_tc_kernel<3><<<grid, XCfg<3>::kThreads, XCfg<3>::kSmem, s>>>(mq, mkv, mo, p);
  } else {
    cudaError_t e = cudaFuncSetAttribute(xattn_tc_kernel<2>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)XCfg<2>::kSmem);
    if (e != cudaSuccess) return e;
    xattn_tc_kernel<2><<<grid, XCfg<2>::kThreads, XCfg<2>::kSmem, s>>>(mq, mkv, mo, p);
  }
  return cudaGetLastError();
}

}  // namespace dpp

// Internal declarations shared by the translation units of libdpp.so.
// Host-side launchers (one per kernel family) and small device helpers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dpp.h"

namespace dpp {

// ---------------------------------------------------------------- constants
// Grid sizes of the reductions are fixed functions of the problem shape (not
// of the device), so every reduction order -- and therefore every bit of the
// results -- is the same on any GPU.
constexpr int kReduceBlocks = 1184;  // 148 SMs x 8

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---------------------------------------------------------------- launchers
// All return cudaSuccess or the launch error; arguments were validated.

// refresh: copy selected bands of [outer][rows][row_bytes] (row_bytes % 16 == 0)
cudaError_t launch_refresh(const void *fresh, void *stale, size_t outer, size_t rows,
                           size_t row_bytes, int P, uint64_t mask, cudaStream_t s);
// halo refresh: at each band boundary the two rows beside it (P >= 2)
cudaError_t launch_refresh_halo(const void *fresh, void *stale, size_t outer, size_t rows,
                                size_t row_bytes, int P, cudaStream_t s);

// guidance combine + discrepancy sums
size_t cfg_blocks(size_t n);
cudaError_t launch_cfg(const float *u, const float *c, float scale, size_t n, float *out,
                       double *sums3, void *ws, cudaStream_t s);

// GroupNorm: one cooperative launch (plus a counter reset), band-major, the
// second read of each chunk served from L2.  The workspace holds per-unit
// counters and fp64 totals; the grid is at most kGnMaxGrid CTAs.
constexpr int kGnMaxGrid = 592;  // 148 SMs x 4 resident CTAs
size_t gn_workspace(const dpp_gn_desc &d);
cudaError_t launch_groupnorm(const dpp_gn_desc &d, const void *x, const float *stats_prev,
                             float *stats_next, const float *gamma, const float *beta,
                             void *y, void *ws, cudaStream_t s);

// GroupNorm's single pass given the band sums of its input (from the conv
// epilogue): gn_sums fp64 [P][B][G][2].
cudaError_t launch_groupnorm_apply(const dpp_gn_desc &d, const void *x, const float *stats_prev,
                                   const double *gn_sums, float *stats_next, const float *gamma,
                                   const float *beta, void *y, cudaStream_t s);
// The band sums of x in a pass of their own (gn_sums fp64 [P][B][G][2],
// zeroed first), and the per-band affine (a, s) [P][B][C][2] fp32 that the
// normalising conv applies, with stats_next[p] = gn_sums[p] in fp32.
cudaError_t launch_groupnorm_sums(const dpp_gn_desc &d, const void *x, double *gn_sums,
                                  cudaStream_t s);
cudaError_t launch_groupnorm_affine(const dpp_gn_desc &d, const double *gn_sums,
                                    const float *stats_prev, float *stats_next,
                                    const float *gamma, const float *beta, float *affine,
                                    cudaStream_t s);

// GroupNorm with its scratch in a static device array of this many bytes
// (no workspace argument, no allocation).
constexpr size_t kGnStaticScratchBytes = DPP_GN_STATIC_SCRATCH_BYTES;
cudaError_t launch_groupnorm_static(const dpp_gn_desc &d, const void *x, const float *stats_prev,
                                    float *stats_next, const float *gamma, const float *beta,
                                    void *y, cudaStream_t s);

// SIMT implicit-GEMM conv (fp32 / bf16 storage, fp32 math)
cudaError_t launch_conv_simt(const dpp_conv_desc &d, const void *x, const void *stale,
                             const void *w, const float *bias, void *y, cudaStream_t s);

// tcgen05 implicit-GEMM conv (bf16); returns cudaErrorNotSupported when the
// shape is outside what the kernel handles
bool conv_tc_supported(const dpp_conv_desc &d);
// With gn_sums (fp64 [P][B][G][2]) the epilogue also writes, per band,
// image and group of G, the sum and sum of squares of the stored output.
cudaError_t launch_conv_tc(const dpp_conv_desc &d, const void *x, const void *stale,
                           const void *w, const float *bias, void *y, int *status,
                           cudaStream_t s, double *gn_sums = nullptr, int G = 0);
// The same conv reading act(x * a + s) (GroupNorm -> SiLU applied on load):
// affine / affine_prev [P][B][C_in][2] fp32 (scale, shift) per band of the
// row read, of this step and of the previous one (halo rows from stale).
cudaError_t launch_conv_norm_tc(const dpp_conv_desc &d, const void *x, const void *stale,
                                const float *affine, const float *affine_prev, int act,
                                const void *w, const float *bias, void *y, int *status,
                                cudaStream_t s, double *gn_sums = nullptr, int G = 0);
// zero n doubles (the fp64 totals the sum kernels add into)
cudaError_t launch_zero_f64(double *p, size_t n, cudaStream_t s);

// Element types inside the library.  Attention layers whose activations are
// bf16 keep Q, O and the K/V state in fp16: the same tensor-core rate with
// an 11-bit significand, which keeps the chained roundings of the layer
// within the bf16 error budget (bf16 intermediates alone exceed it).
enum Elem : int { E_F32 = 0, E_BF16 = 1, E_F16 = 2 };

inline Elem layer_elem(dpp_dtype t) { return t == DPP_BF16 ? E_BF16 : E_F32; }
inline Elem inter_elem(dpp_dtype t) { return t == DPP_BF16 ? E_F16 : E_F32; }
inline size_t elem_bytes(Elem e) { return e == E_F32 ? 4 : 2; }

// GEMM D = A * B^T with B given as up to 3 row blocks (weights [out, in]);
// output columns [0, split) go to out0 (leading dim ld0), the rest to out1
// (leading dim ld1, column index minus split).
struct GemmArgs {
  const void *A;      // [M, K], element type ta
  const void *B[3];   // each [b_rows, K], element type tb
  int b_rows;         // rows per B block
  int M, N, K;
  void *out0;         // element type to
  int ld0;
  int split;
  void *out1;
  int ld1;
  Elem ta, tb, to;
  const float *bias = nullptr;  // [N] fp32 added to out0's columns ([2 Nout] with geglu)
  int accumulate = 0;           // out0 += result (out0 read first)
  int geglu = 0;                // B[0] = value rows, B[1] = gate rows (b_rows = N each):
                                // out0 = value * GELU(gate), N output columns
  // optional side task of the tensor-core GEMM: a bf16 -> fp16 copy of
  // cast_n elements (a multiple of 8, 16-byte aligned), done by the
  // epilogue warps while they wait for their first accumulator
  const void *cast_src = nullptr;
  void *cast_dst = nullptr;
  size_t cast_n = 0;
};
cudaError_t launch_gemm_simt(const GemmArgs &g, cudaStream_t s);
cudaError_t launch_gemm_tc(const GemmArgs &g, int *status, cudaStream_t s);
bool gemm_tc_supported(const GemmArgs &g);
// bf16 -> fp16 element copy (weights feeding an fp16 tensor-core operand)
cudaError_t launch_cast_bf16_f16(const void *in, void *out, size_t n, cudaStream_t s);

// attention core: O = softmax(Q K^T / 8) V for head_dim 64.
// q: [B, Nq, C]; kv_fresh / kv_stale: [B, Nkv, 2, C] (kv_stale may be null:
// everything fresh).  Query band p (of P) attends over fresh keys of its own
// band and stale keys elsewhere; with Nkv != Nq (cross attention) P must be 1.
// q, kv and o share the element type `te` (fp16 or fp32).
struct AttnArgs {
  const void *q;
  const void *kv_fresh;
  const void *kv_stale;
  void *o;
  int B, Nq, Nkv, C, heads, P;
  Elem te;
  int band_local;  // queries of a band attend over that band's (fresh) keys only
};
cudaError_t launch_attn_simt(const AttnArgs &a, cudaStream_t s);
cudaError_t launch_attn_tc(const AttnArgs &a, int *status, cudaStream_t s);
bool attn_tc_supported(const AttnArgs &a);
// persistent core for keys that fit one tile (<= 128) without stale bands:
// cross-attention over the text context
cudaError_t launch_xattn_tc(const AttnArgs &a, int *status, cudaStream_t s);
bool xattn_tc_supported(const AttnArgs &a);

// token-wise LayerNorm (C <= 256 16-byte vectors)
cudaError_t launch_layernorm(const dpp_ln_desc &d, const void *x, const float *gamma,
                             const float *beta, void *y, cudaStream_t s);

// self-tests of the two bounded waits (see dpp_wait_selftest)
cudaError_t launch_wait_selftest_counter(const unsigned *counter, cudaStream_t s);
cudaError_t launch_wait_selftest_mbarrier(cudaStream_t s);

// device status word (bounded waits record DPP_ERR_TIMEOUT here)
int *device_status_ptr();

}  // namespace dpp

// Stale-buffer refresh: the all_gather of the DistriFusion developer guide
// (section 分布式通信与同步机制: each band's rows are gathered and
// concatenated along the height axis).  On one GPU every band's fresh rows
// already sit in one tensor, so the gather is a bit-exact copy of the
// selected bands into the buffer the next step reads as stale.
//
// HBM-bound: 2 bytes moved per byte of band.  16-byte vector copies, four
// independent loads in flight per thread, grid sized in multiples of the SM
// count; blockIdx.y walks the (outer slice, selected band) segments, each of
// which is contiguous in memory.
#include "dpp_internal.h"

namespace dpp {
namespace {

struct BandList {
  uint8_t band[64];
};

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads)
refresh_kernel(const uint4 *__restrict__ fresh, uint4 *__restrict__ stale, size_t rows_vec,
               size_t band_vec, int nsel, const __grid_constant__ BandList sel) {
  const size_t seg = blockIdx.y;                 // outer * nsel segments
  const size_t o = seg / nsel;
  const int p = sel.band[seg % nsel];
  const size_t base = o * rows_vec + (size_t)p * band_vec;
  const uint4 *src = fresh + base;
  uint4 *dst = stale + base;
  const size_t stride = (size_t)gridDim.x * kThreads;
  size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x;
  for (; i + (kUnroll - 1) * stride < band_vec; i += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = __ldcs(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) __stcs(dst + i + u * stride, v[u]);
  }
  for (; i < band_vec; i += stride) __stcs(dst + i, __ldcs(src + i));
}

// The rows of a displaced conv's input that another band reads as its halo:
// at every band boundary k (1 <= k < P) the last row of band k-1 and the
// first row of band k.  blockIdx.y walks (outer slice, boundary, side).
__global__ void __launch_bounds__(kThreads)
halo_kernel(const uint4 *__restrict__ fresh, uint4 *__restrict__ stale, size_t rows,
            size_t row_vec, int Hp, int nb) {
  const size_t seg = blockIdx.y;
  const size_t o = seg / nb;
  const int r = (int)(seg % nb);
  const size_t row = (size_t)(r / 2 + 1) * Hp - 1 + (r & 1);
  const size_t base = (o * rows + row) * row_vec;
  for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < row_vec;
       i += (size_t)gridDim.x * kThreads)
    __stcs(stale + base + i, __ldcs(fresh + base + i));
}

}  // namespace

cudaError_t launch_refresh(const void *fresh, void *stale, size_t outer, size_t rows,
                           size_t row_bytes, int P, uint64_t mask, cudaStream_t s) {
  BandList sel{};
  int nsel = 0;
  for (int p = 0; p < P; ++p)
    if ((mask >> p) & 1ull) sel.band[nsel++] = (uint8_t)p;
  if (nsel == 0 || outer == 0 || rows == 0 || row_bytes == 0) return cudaSuccess;
  const size_t row_vec = row_bytes / 16;
  const size_t band_vec = (rows / P) * row_vec;
  const size_t segs = outer * (size_t)nsel;
  // about 4 resident blocks of work per SM in total, at least one per segment
  size_t want = (size_t)kReduceBlocks * 2 / segs;
  size_t need = (band_vec + (size_t)kThreads * kUnroll - 1) / ((size_t)kThreads * kUnroll);
  unsigned gx = (unsigned)(want < 1 ? 1 : (want < need ? want : need));
  if (gx == 0) gx = 1;
  if (segs > 65535) return cudaErrorInvalidConfiguration;
  refresh_kernel<<<dim3(gx, (unsigned)segs), kThreads, 0, s>>>(
      (const uint4 *)fresh, (uint4 *)stale, rows * row_vec, band_vec, nsel, sel);
  return cudaGetLastError();
}

cudaError_t launch_refresh_halo(const void *fresh, void *stale, size_t outer, size_t rows,
                                size_t row_bytes, int P, cudaStream_t s) {
  if (P < 2 || outer == 0 || rows == 0 || row_bytes == 0) return cudaSuccess;
  const int nb = 2 * (P - 1);
  const size_t segs = outer * (size_t)nb;
  if (segs > 65535) return cudaErrorInvalidConfiguration;
  const size_t row_vec = row_bytes / 16;
  const unsigned gx = (unsigned)((row_vec + kThreads - 1) / kThreads);
  halo_kernel<<<dim3(gx, (unsigned)segs), kThreads, 0, s>>>(
      (const uint4 *)fresh, (uint4 *)stale, rows, row_vec, (int)(rows / P), nb);
  return cudaGetLastError();
}

}  // namespace dpp

// Row cut and scatter-back around the late layers.
//
// Entering the late layers, the per-row state of an extend (hidden rows, mHC
// streams, token ids) is cut to the tail rows, and after them the computed
// tail rows are scattered back into the full extend layout while every other
// row is left as it was ("SGLang 如何让 DeepSeek V4.1 Flash 的后半层只处理尾部
// token", sec. 2.2 and 2.7).  The row map is the tail layout's src_row (or the
// encoder replay layout's, whose replayed rows carry -1 and are skipped).
//
// Pure data movement, bound by HBM.  The work items are 4 KB pieces of rows
// (one warp each, eight 16-byte loads in flight per lane before their
// stores), so that a few thousand rows still keep every SM's memory pipeline
// full; streaming cache hints keep the one-time rows from displacing L2.  The
// row count is read on the device (the layout kernel wrote it), so nothing
// waits on the host; the grid covers the work with at most 8 CTAs of 256
// threads per SM.
#include "common.cuh"

namespace csa2 {
namespace {

constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kPieceVecs = 256;   // 16-byte vectors per work item (4 KB)

template <bool kScatter>
__global__ void __launch_bounds__(kRowThreads)
rows_copy_kernel(const int32_t *__restrict__ count, int64_t capacity,
                 const int32_t *__restrict__ row_idx, const uint4 *__restrict__ src,
                 uint4 *__restrict__ dst, int64_t other_rows, int64_t vec_per_row,
                 int64_t pieces_per_row, int32_t *__restrict__ d_err) {
  int64_t n = capacity;
  if (count) {
    const int64_t c = *count;
    n = c < 0 ? 0 : (c < n ? c : n);
  }
  const int lane = threadIdx.x & 31;
  const int64_t items = n * pieces_per_row;
  int err = 0;
  for (int64_t w = (int64_t)blockIdx.x * kRowWarps + (threadIdx.x >> 5); w < items;
       w += (int64_t)gridDim.x * kRowWarps) {
    const int64_t i = w / pieces_per_row;     // the same for the whole warp
    const int64_t piece = w - i * pieces_per_row;
    const int64_t j = row_idx[i];
    if (j < 0) continue;
    if (j >= other_rows) {
      if (piece == 0) err |= CSA2_DERR_RANGE_ROW;
      continue;
    }
    const int64_t v0 = piece * kPieceVecs;
    const uint4 *s = src + (kScatter ? i : j) * vec_per_row + v0;
    uint4 *d = dst + (kScatter ? j : i) * vec_per_row + v0;
    const int64_t nv = vec_per_row - v0 < kPieceVecs ? vec_per_row - v0 : kPieceVecs;
    if (nv == kPieceVecs) {
      uint4 r[kPieceVecs / 32];
#pragma unroll
      for (int k = 0; k < kPieceVecs / 32; ++k) r[k] = __ldcs(s + lane + 32 * k);
#pragma unroll
      for (int k = 0; k < kPieceVecs / 32; ++k) __stcs(d + lane + 32 * k, r[k]);
    } else {
      for (int64_t v = lane; v < nv; v += 32) __stcs(d + v, __ldcs(s + v));
    }
  }
  err = __reduce_or_sync(0xffffffffu, err);
  if (lane == 0) raise_err(d_err, err);
}

template <bool kScatter>
int rows_copy(const int32_t *count, int64_t capacity, const int32_t *row_idx, const void *src,
              void *dst, int64_t other_rows, int64_t row_bytes, int32_t *d_err,
              csa2_stream_t stream) {
  if (capacity < 0 || other_rows < 0 || row_bytes < 0) return CSA2_ERR_INVALID_ARG;
  if (capacity == 0 || row_bytes == 0) return CSA2_OK;
  if (!row_idx || !src || !dst) return CSA2_ERR_INVALID_ARG;
  if ((row_bytes & 15) || (((uintptr_t)src | (uintptr_t)dst) & 15u)) return CSA2_ERR_UNSUPPORTED;
  const int64_t vec_per_row = row_bytes / 16;
  const int64_t pieces = (vec_per_row + kPieceVecs - 1) / kPieceVecs;
  const int64_t want = (capacity * pieces + kRowWarps - 1) / kRowWarps;
  const int64_t cap = (int64_t)sm_count() * (2048 / kRowThreads);
  const int grid = (int)(want < cap ? want : cap);
  rows_copy_kernel<kScatter><<<grid, kRowThreads, 0, as_stream(stream)>>>(
      count, capacity, row_idx, static_cast<const uint4 *>(src), static_cast<uint4 *>(dst),
      other_rows, vec_per_row, pieces, d_err);
  return launch_status();
}

}  // namespace
}  // namespace csa2

extern "C" CSA2_API int csa2_rows_gather(const int32_t *count, int64_t capacity,
                                         const int32_t *row_idx, const void *src,
                                         int64_t src_rows, void *dst, int64_t row_bytes,
                                         int32_t *d_err, csa2_stream_t stream) {
  return csa2::rows_copy<false>(count, capacity, row_idx, src, dst, src_rows, row_bytes, d_err,
                                stream);
}

extern "C" CSA2_API int csa2_rows_scatter(const int32_t *count, int64_t capacity,
                                          const int32_t *row_idx, const void *src, void *dst,
                                          int64_t dst_rows, int64_t row_bytes, int32_t *d_err,
                                          csa2_stream_t stream) {
  return csa2::rows_copy<true>(count, capacity, row_idx, src, dst, dst_rows, row_bytes, d_err,
                               stream);
}

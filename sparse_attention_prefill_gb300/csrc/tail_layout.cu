// a1: decoder bounded-replay tail layout.
//
// Per request r (extend length E_r, sequence length S_r after the extend) the
// late layers keep the last T_r = min(window, E_r) rows of this extend, at
// their absolute positions S_r - T_r + k, each with the absolute window lower
// bound S_r - T_r ("SGLang 如何让 DeepSeek V4.1 Flash 的后半层只处理尾部 token",
// sec. 2.1 and 2.2; short extends sec. 2.6; chunked extends sec. 2.5).
//
// One CTA of 1024 threads walks the requests in chunks of 1024: a block scan
// gives each request its offset in the packed extend and in the tail, then the
// chunk's tail rows are written row-parallel (binary search of the row's
// request in the chunk's inclusive tail scan kept in shared memory).  The work
// is a few kilobytes of metadata, so one CTA on one SM is the right size.
#include "common.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 1024;

// Block-wide exclusive scan of one int64 per thread; returns the block total.
__device__ int64_t block_exclusive_scan(int64_t v, int64_t *warp_sums, int64_t &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int64_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  int64_t before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  total = warp_sums[31];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kThreads)
tail_layout_kernel(int32_t num_req, const int32_t *__restrict__ extend_len,
                   const int64_t *__restrict__ seq_len, int32_t window,
                   int32_t *__restrict__ tail_len, int32_t *__restrict__ cu_tail,
                   int32_t *__restrict__ src_row, int64_t *__restrict__ pos,
                   int64_t *__restrict__ win_lo, int32_t *__restrict__ row_req,
                   int64_t capacity, int32_t *__restrict__ d_err) {
  __shared__ int64_t warp_sums[32];
  __shared__ int64_t incl_t[kThreads];   // inclusive tail scan within the chunk
  __shared__ int64_t base_e[kThreads];   // packed-extend row of the request's first row
  __shared__ int64_t first_pos[kThreads];
  __shared__ int64_t tlen[kThreads];
  int64_t carry_e = 0, carry_t = 0;
  int err = 0;
  if (threadIdx.x == 0) cu_tail[0] = 0;
  for (int32_t c0 = 0; c0 < num_req; c0 += kThreads) {
    const int r = c0 + threadIdx.x;
    int64_t e = 0, s = 0, t = 0;
    if (r < num_req) {
      e = extend_len[r];
      s = seq_len[r];
      if (e < 0 || s < e) {
        err |= CSA2_DERR_BAD_EXTEND;
      } else {
        t = e < window ? e : window;
      }
    }
    const int64_t e_pos = e > 0 ? e : 0;
    int64_t tot_e, tot_t;
    const int64_t ex_e = block_exclusive_scan(e_pos, warp_sums, tot_e);
    const int64_t ex_t = block_exclusive_scan(t, warp_sums, tot_t);
    incl_t[threadIdx.x] = ex_t + t;
    base_e[threadIdx.x] = carry_e + ex_e + e_pos - t;
    first_pos[threadIdx.x] = s - t;
    tlen[threadIdx.x] = t;
    if (r < num_req) {
      tail_len[r] = (int32_t)t;
      cu_tail[r + 1] = (int32_t)(carry_t + ex_t + t);
    }
    __syncthreads();
    const int nreq = min(kThreads, num_req - c0);
    for (int64_t i = threadIdx.x; i < tot_t; i += kThreads) {
      // request of chunk row i: first q with incl_t[q] > i
      int lo = 0, hi = nreq - 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (incl_t[mid] > i) hi = mid; else lo = mid + 1;
      }
      const int64_t k = i - (incl_t[lo] - tlen[lo]);
      const int64_t row = carry_t + i;
      if (row >= capacity) {
        err |= CSA2_DERR_CAPACITY;
        continue;
      }
      src_row[row] = (int32_t)(base_e[lo] + k);
      pos[row] = first_pos[lo] + k;
      win_lo[row] = first_pos[lo];
      if (row_req) row_req[row] = c0 + lo;
    }
    carry_e += tot_e;
    carry_t += tot_t;
    __syncthreads();
  }
  err = __reduce_or_sync(0xffffffffu, err);
  if ((threadIdx.x & 31) == 0) raise_err(d_err, err);
}

// Encoder-side bounded replay ("DeepSeek V4.1 Flash 建模", Encoder Bounded
// Replay card; SGLang/Miles day-0 article sec. 4.1, 4.3).  Per request r with
// P_r cached tokens and E_r new ones, the rows are positions P_r - Rp_r ...
// P_r + E_r - 1 with Rp_r = min(window, P_r); replayed rows have no row in the
// packed new-token input (src_row = -1); every row carries the lower bound
// P_r - Rp_r; entry_range[r] = [floor(P_r/m), floor((P_r+E_r)/m)) are the
// global entries this extend completes (all earlier ones are cached).  Same
// one-CTA chunked scan as the tail layout.
__global__ void __launch_bounds__(kThreads)
encoder_replay_layout_kernel(int32_t num_req, const int64_t *__restrict__ prefix_len,
                             const int32_t *__restrict__ extend_len, int32_t window,
                             int32_t ratio, int32_t *__restrict__ replay_len,
                             int32_t *__restrict__ cu_rows, int32_t *__restrict__ src_row,
                             int64_t *__restrict__ pos, int64_t *__restrict__ win_lo,
                             int32_t *__restrict__ row_req, int64_t *__restrict__ entry_range,
                             int64_t capacity, int32_t *__restrict__ d_err) {
  __shared__ int64_t warp_sums[32];
  __shared__ int64_t incl_n[kThreads];   // inclusive row scan within the chunk
  __shared__ int64_t base_e[kThreads];   // packed new-token row of the request's first new row
  __shared__ int64_t first_pos[kThreads];
  __shared__ int64_t rlen[kThreads];     // replayed rows
  __shared__ int64_t nlen[kThreads];     // all rows
  int64_t carry_e = 0, carry_n = 0;
  int err = 0;
  if (threadIdx.x == 0) cu_rows[0] = 0;
  for (int32_t c0 = 0; c0 < num_req; c0 += kThreads) {
    const int r = c0 + threadIdx.x;
    int64_t p = 0, e = 0, rp = 0;
    if (r < num_req) {
      p = prefix_len[r];
      e = extend_len[r];
      if (p < 0 || e < 0) {
        err |= CSA2_DERR_BAD_EXTEND;
        p = 0;
        e = 0;
      } else {
        rp = p < window ? p : window;
      }
    }
    const int64_t n = rp + e;
    int64_t tot_e, tot_n;
    const int64_t ex_e = block_exclusive_scan(e, warp_sums, tot_e);
    const int64_t ex_n = block_exclusive_scan(n, warp_sums, tot_n);
    incl_n[threadIdx.x] = ex_n + n;
    base_e[threadIdx.x] = carry_e + ex_e;
    first_pos[threadIdx.x] = p - rp;
    rlen[threadIdx.x] = rp;
    nlen[threadIdx.x] = n;
    if (r < num_req) {
      replay_len[r] = (int32_t)rp;
      cu_rows[r + 1] = (int32_t)(carry_n + ex_n + n);
      if (entry_range) {
        entry_range[2 * r] = p / ratio;
        entry_range[2 * r + 1] = (p + e) / ratio;
      }
    }
    __syncthreads();
    const int nreq = min(kThreads, num_req - c0);
    for (int64_t i = threadIdx.x; i < tot_n; i += kThreads) {
      int lo = 0, hi = nreq - 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (incl_n[mid] > i) hi = mid; else lo = mid + 1;
      }
      const int64_t k = i - (incl_n[lo] - nlen[lo]);
      const int64_t row = carry_n + i;
      if (row >= capacity) {
        err |= CSA2_DERR_CAPACITY;
        continue;
      }
      src_row[row] = k < rlen[lo] ? -1 : (int32_t)(base_e[lo] + k - rlen[lo]);
      pos[row] = first_pos[lo] + k;
      win_lo[row] = first_pos[lo];
      if (row_req) row_req[row] = c0 + lo;
    }
    carry_e += tot_e;
    carry_n += tot_n;
    __syncthreads();
  }
  err = __reduce_or_sync(0xffffffffu, err);
  if ((threadIdx.x & 31) == 0) raise_err(d_err, err);
}

}  // namespace
}  // namespace csa2

extern "C" CSA2_API int csa2_encoder_replay_layout(
    int32_t num_req, const int64_t *prefix_len, const int32_t *extend_len, int32_t window,
    int32_t ratio, int32_t *replay_len, int32_t *cu_rows, int32_t *src_row, int64_t *pos,
    int64_t *win_lo, int32_t *row_req, int64_t *entry_range, int64_t capacity, int32_t *d_err,
    csa2_stream_t stream) {
  if (num_req < 0 || window < 1 || capacity < 0 || !cu_rows) return CSA2_ERR_INVALID_ARG;
  if (ratio != 1 && ratio != 2) return CSA2_ERR_INVALID_ARG;
  if (num_req > 0 && (!prefix_len || !extend_len || !replay_len)) return CSA2_ERR_INVALID_ARG;
  if (capacity > 0 && (!src_row || !pos || !win_lo)) return CSA2_ERR_INVALID_ARG;
  csa2::encoder_replay_layout_kernel<<<1, csa2::kThreads, 0, csa2::as_stream(stream)>>>(
      num_req, prefix_len, extend_len, window, ratio, replay_len, cu_rows, src_row, pos, win_lo,
      row_req, entry_range, capacity, d_err);
  return csa2::launch_status();
}

extern "C" CSA2_API int csa2_tail_layout(int32_t num_req, const int32_t *extend_len,
                                const int64_t *seq_len, int32_t window, int32_t *tail_len,
                                int32_t *cu_tail, int32_t *src_row, int64_t *pos,
                                int64_t *win_lo, int32_t *row_req, int64_t capacity,
                                int32_t *d_err, csa2_stream_t stream) {
  if (num_req < 0 || window < 1 || capacity < 0 || !cu_tail) return CSA2_ERR_INVALID_ARG;
  if (num_req > 0 && (!extend_len || !seq_len || !tail_len)) return CSA2_ERR_INVALID_ARG;
  if (capacity > 0 && (!src_row || !pos || !win_lo)) return CSA2_ERR_INVALID_ARG;
  csa2::tail_layout_kernel<<<1, csa2::kThreads, 0, csa2::as_stream(stream)>>>(
      num_req, extend_len, seq_len, window, tail_len, cu_tail, src_row, pos, win_lo, row_req,
      capacity, d_err);
  return csa2::launch_status();
}

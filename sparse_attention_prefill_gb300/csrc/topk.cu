// a5, a6, a7: top-K selection and hierarchical candidate blocks.
//
// Per query, the k best visible entries by the total order (score desc, entry
// id asc); NaN and -inf never selected ("DeepSeek V4.1 Flash 建模",
// Hierarchical card; SGLang/Miles day-0 article sec. 2).  The L20-style source
// also publishes at most max_blocks blocks of `block` entries ranked by their
// maximum score, always keeping the block that holds the latest position.
//
// One CTA per query row.  Scores become order-preserving uint32 keys (0 marks
// an ineligible element).  A 4-pass 8-bit radix select finds the k-th largest
// key T; keys > T are emitted directly, and the k - #(> T) keys equal to T are
// taken in index order by a block-wide ordered scan, which makes the result
// exactly the pinned total order's top k.  Rows that fit in shared memory are
// staged there once; longer rows are re-read from global memory (L2) in each
// pass.  The same selection core ranks candidate blocks by block maximum, and
// the chosen blocks are sorted ascending with a shared-memory bitonic sort.
#include "common.cuh"
#include "kernels.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 512;
constexpr int kSmemKeys = 40960;      // staged row capacity (160 KB)
constexpr int kMaxSortBlocks = 4096;  // max_blocks supported

struct SelectShared {
  uint32_t hist[256];
  uint32_t warp_tot[kThreads / 32];
  uint32_t prefix, remaining, out_count, n_elig;
  int32_t nb;
};

// Block-wide exclusive scan of one uint32 per thread (kThreads threads).
__device__ uint32_t block_scan_u32(uint32_t v, uint32_t *warp_tot, uint32_t &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = lane < kThreads / 32 ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kThreads / 32) warp_tot[lane] = s;
  }
  __syncthreads();
  total = warp_tot[kThreads / 32 - 1];
  return (warp ? warp_tot[warp - 1] : 0u) + x - v;
}

// Select the k largest keys (key 0 = ineligible) of a virtual array of n keys,
// ties by lowest index.  Calls emit(i) once for every selected index i (in no
// particular order) and returns min(k, #eligible).
template <class Keys, class Emit>
__device__ uint32_t select_topk(const Keys &keys, int64_t n, uint32_t k, SelectShared &sh,
                                Emit emit) {
  // eligible count
  uint32_t cnt = 0;
  for (int64_t i = threadIdx.x; i < n; i += kThreads) cnt += keys(i) != 0u;
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  if (threadIdx.x == 0) sh.n_elig = 0;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) atomicAdd(&sh.n_elig, cnt);
  __syncthreads();
  const uint32_t n_elig = sh.n_elig;
  if (n_elig <= k) {
    // everything eligible is selected; keep index order for determinism
    uint32_t base = 0;
    for (int64_t c0 = 0; c0 < n; c0 += kThreads) {
      const int64_t i = c0 + threadIdx.x;
      const uint32_t f = (i < n && keys(i) != 0u) ? 1u : 0u;
      uint32_t tot;
      const uint32_t ex = block_scan_u32(f, sh.warp_tot, tot);
      if (f) emit(i, base + ex);
      base += tot;
    }
    __syncthreads();
    return n_elig;
  }
  // radix select of the k-th largest key
  if (threadIdx.x == 0) {
    sh.prefix = 0;
    sh.remaining = k;
  }
  __syncthreads();
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kThreads) sh.hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = sh.prefix;
    const uint32_t hi_mask = shift == 24 ? 0u : (0xffffffffu << (shift + 8));
    // warp-aggregated increments: the lanes holding the same digit add once
    // (score keys cluster in a few exponent buckets, which would otherwise
    // serialise on a handful of shared-memory counters)
    for (int64_t i0 = 0; i0 < n; i0 += kThreads) {
      const int64_t i = i0 + threadIdx.x;
      uint32_t key = i < n ? keys(i) : 0u;
      const bool take = key != 0u && (key & hi_mask) == prefix;
      const uint32_t digit = take ? (key >> shift) & 255u : 256u;
      const uint32_t peers = __match_any_sync(0xffffffffu, digit);
      if (take && (threadIdx.x & 31) == (uint32_t)(__ffs(peers) - 1))
        atomicAdd(&sh.hist[digit], (uint32_t)__popc(peers));
    }
    __syncthreads();
    // scan bins from the top digit down
    const uint32_t remaining = sh.remaining;
    uint32_t h = threadIdx.x < 256 ? sh.hist[255 - threadIdx.x] : 0u;
    uint32_t tot;
    const uint32_t ex = block_scan_u32(h, sh.warp_tot, tot);
    if (threadIdx.x < 256 && ex < remaining && ex + h >= remaining) {
      sh.prefix = prefix | ((uint32_t)(255 - threadIdx.x) << shift);
      sh.remaining = remaining - ex;
    }
    __syncthreads();
  }
  const uint32_t T = sh.prefix;
  const uint32_t need_eq = sh.remaining;  // how many keys == T to take
  if (threadIdx.x == 0) sh.out_count = 0;
  __syncthreads();
  // keys above the threshold
  for (int64_t i = threadIdx.x; i < n; i += kThreads) {
    if (keys(i) > T) emit(i, atomicAdd(&sh.out_count, 1u));
  }
  __syncthreads();
  const uint32_t n_gt = sh.out_count;
  // keys equal to the threshold, lowest indices first
  uint32_t base = 0;
  for (int64_t c0 = 0; c0 < n && base < need_eq; c0 += kThreads) {
    const int64_t i = c0 + threadIdx.x;
    const uint32_t f = (i < n && keys(i) == T) ? 1u : 0u;
    uint32_t tot;
    const uint32_t ex = block_scan_u32(f, sh.warp_tot, tot);
    if (f && base + ex < need_eq) emit(i, n_gt + base + ex);
    base += tot;
  }
  __syncthreads();
  return k;
}

// Row view: the scores of query q as keys, in full mode (entries 0..len-1) or
// pool mode (slots, mapped to entries through the candidate blocks).
struct RowView {
  const float *row;
  const int32_t *cand;  // candidate blocks of this query or nullptr
  int block;
  int64_t n_vis;
  __device__ __forceinline__ int64_t entry(int64_t s) const {
    return cand ? (int64_t)cand[s / block] * block + s % block : s;
  }
  __device__ __forceinline__ uint32_t operator()(int64_t s) const {
    if (cand && entry(s) >= n_vis) return 0u;
    const uint32_t key = float_key(__ldg(row + s));
    return key > neg_inf_key() ? key : 0u;
  }
};

struct SmemKeys {
  const uint32_t *k;
  __device__ __forceinline__ uint32_t operator()(int64_t i) const { return k[i]; }
};

// Block view: key of block b = max key over its visible entries, plus one, so
// every block is eligible (the pool is a budget, filled whatever the scores).
struct BlockView {
  const float *row;
  int block;
  int64_t n_vis;
  __device__ __forceinline__ uint32_t operator()(int64_t b) const {
    uint32_t m = 0;
    const int64_t j1 = min((b + 1) * block, n_vis);
    for (int64_t j = b * block; j < j1; ++j) m = max(m, float_key(__ldg(row + j)));
    return m + 1u;
  }
};

__device__ void row_geometry(const Batch &b, int q, const int32_t *cand_blocks, int block,
                             int max_blocks, int64_t ld, int64_t &n_vis, int64_t &row_len,
                             int &err, SelectShared &sh) {
  const int r = b.q_req[q];
  n_vis = n_visible(b.q_pos[q], b.ratio);
  if (n_vis > b.kv_len[r]) {
    n_vis = b.kv_len[r];
    err |= CSA2_DERR_RANGE_CTX;
  }
  if (cand_blocks) {
    if (threadIdx.x == 0) sh.nb = max_blocks;
    __syncthreads();
    const int32_t *cb = cand_blocks + (int64_t)q * max_blocks;
    for (int i = threadIdx.x; i < max_blocks; i += kThreads)
      if (cb[i] < 0) atomicMin(&sh.nb, i);
    __syncthreads();
    row_len = (int64_t)sh.nb * block;
  } else {
    row_len = n_vis;
  }
  if (row_len > ld) {
    row_len = ld;
    err |= CSA2_DERR_LD;
  }
}

__global__ void __launch_bounds__(kThreads)
topk_kernel(Batch b, const float *__restrict__ scores, int64_t ld, int k,
            const int32_t *__restrict__ cand_blocks, int block, int max_blocks,
            int32_t *__restrict__ idx, int32_t *__restrict__ count, int32_t *__restrict__ d_err,
            int64_t staged) {
  extern __shared__ uint32_t smem_keys[];
  __shared__ SelectShared sh;
  const int q = blockIdx.x;
  int err = 0;
  int64_t n_vis, row_len;
  row_geometry(b, q, cand_blocks, block, max_blocks, ld, n_vis, row_len, err, sh);
  RowView view{scores + (int64_t)q * ld, cand_blocks ? cand_blocks + (int64_t)q * max_blocks : nullptr,
                block, n_vis};
  int32_t *out = idx + (int64_t)q * k;
  auto emit = [&](int64_t s, uint32_t slot) { out[slot] = (int32_t)view.entry(s); };
  uint32_t got;
  if (row_len <= staged) {
    for (int64_t s = threadIdx.x; s < row_len; s += kThreads) smem_keys[s] = view(s);
    __syncthreads();
    got = select_topk(SmemKeys{smem_keys}, row_len, (uint32_t)k, sh, emit);
  } else {
    got = select_topk(view, row_len, (uint32_t)k, sh, emit);
  }
  for (int i = (int)got + threadIdx.x; i < k; i += kThreads) out[i] = -1;
  if (threadIdx.x == 0) count[q] = (int32_t)got;
  err = __reduce_or_sync(0xffffffffu, err);
  if ((threadIdx.x & 31) == 0 && threadIdx.x == 0) raise_err(d_err, err);
}

__global__ void __launch_bounds__(kThreads)
candidate_blocks_kernel(Batch b, const float *__restrict__ scores, int64_t ld, int block,
                        int max_blocks, int32_t *__restrict__ blocks,
                        int32_t *__restrict__ nblocks, int64_t staged) {
  extern __shared__ uint32_t smem_keys[];
  __shared__ SelectShared sh;
  __shared__ int32_t chosen[kMaxSortBlocks];
  const int q = blockIdx.x;
  const int r = b.q_req[q];
  int64_t n_vis = n_visible(b.q_pos[q], b.ratio);
  if (n_vis > b.kv_len[r]) n_vis = b.kv_len[r];
  if (n_vis > ld) n_vis = ld;
  const int64_t nb_all = (n_vis + block - 1) / block;
  int32_t *out = blocks + (int64_t)q * max_blocks;
  if (nb_all <= max_blocks) {
    for (int i = threadIdx.x; i < max_blocks; i += kThreads) out[i] = i < nb_all ? i : -1;
    if (threadIdx.x == 0) nblocks[q] = (int32_t)nb_all;
    return;
  }
  const float *row = scores + (int64_t)q * ld;
  BlockView view{row, block, n_vis};
  auto emit = [&](int64_t bb, uint32_t slot) { chosen[slot] = (int32_t)bb; };
  const int64_t n = nb_all - 1;  // the latest block is kept outside the ranking
  if (n <= staged) {
    for (int64_t i = threadIdx.x; i < n; i += kThreads) smem_keys[i] = view(i);
    __syncthreads();
    select_topk(SmemKeys{smem_keys}, n, (uint32_t)(max_blocks - 1), sh, emit);
  } else {
    select_topk(view, n, (uint32_t)(max_blocks - 1), sh, emit);
  }
  // add the latest block, pad to a power of two and sort ascending
  int pow2 = 1;
  while (pow2 < max_blocks) pow2 <<= 1;
  for (int i = threadIdx.x; i < pow2; i += kThreads) {
    if (i == max_blocks - 1) chosen[i] = (int32_t)(nb_all - 1);
    else if (i >= max_blocks) chosen[i] = 0x7fffffff;
  }
  __syncthreads();
  for (int size = 2; size <= pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < pow2; i += kThreads) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;
          const int32_t a = chosen[i], c = chosen[j];
          if ((a > c) == up) {
            chosen[i] = c;
            chosen[j] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < max_blocks; i += kThreads) out[i] = chosen[i];
  if (threadIdx.x == 0) nblocks[q] = max_blocks;
}

}  // namespace

int topk_launch(const Batch &b, const float *scores, int64_t ld, int k,
                const int32_t *cand_blocks, int block, int max_blocks, int32_t *idx,
                int32_t *count, int32_t *blocks_out, int32_t *nblocks_out, int32_t *d_err,
                cudaStream_t st) {
  if (b.num_q == 0) return CSA2_OK;
  // shared memory only as large as the longest row can use (small rows then
  // leave room for several CTAs per SM); rows longer than kSmemKeys stream
  int64_t row_cap = cand_blocks ? (int64_t)max_blocks * block : ld;
  if (row_cap > ld) row_cap = ld;
  const int64_t staged = row_cap < kSmemKeys ? row_cap : kSmemKeys;
  const size_t smem = (size_t)(staged > 0 ? staged : 1) * sizeof(uint32_t);
  const int64_t nblk = (ld + block - 1) / block;
  const size_t smem_b = (size_t)(nblk < kSmemKeys ? (nblk > 0 ? nblk : 1) : kSmemKeys) *
                        sizeof(uint32_t);
  cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  topk_kernel<<<b.num_q, kThreads, smem, st>>>(b, scores, ld, k, cand_blocks, block, max_blocks,
                                               idx, count, d_err, staged);
  if (blocks_out) {
    cudaFuncSetAttribute(candidate_blocks_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem_b);
    candidate_blocks_kernel<<<b.num_q, kThreads, smem_b, st>>>(
        b, scores, ld, block, max_blocks, blocks_out, nblocks_out,
        nblk < kSmemKeys ? nblk : (int64_t)kSmemKeys);
  }
  return launch_status();
}

}  // namespace csa2

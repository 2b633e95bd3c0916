// a5, a6, a7: top-K selection and hierarchical candidate blocks.
//
// Per query, the k best visible entries by the total order (score desc, entry
// id asc); NaN and -inf never selected ("DeepSeek V4.1 Flash 建模",
// Hierarchical card; SGLang/Miles day-0 article sec. 2).  The L20-style source
// also publishes at most max_blocks blocks of `block` entries ranked by their
// maximum score, always keeping the block that holds the latest position.
//
// One CTA per query row.  Scores become order-preserving uint32 keys (0 marks
// an ineligible element); the selection is exactly the k largest keys, ties
// by lowest position, which is the pinned total order's top k.
//  - Rows of up to 16384 keys are held in registers (256 threads, KPT keys
//    each, loaded together).  A threshold guess from the mean and deviation
//    of a strided sample (the score a normal row of those moments would have
//    ~2k + 64 scores above) picks the keys that are compacted into shared
//    memory (typically ~1.1k); an 8-bit radix search finds the exact k-th key
//    on that list alone.  A guess that lists fewer than k keys or more than
//    the list holds falls back to the same search over the whole row.
//  - Longer rows (staged in shared memory, or re-read from L2): the same kind
//    of guess from every 16th key, one sweep that lists the keys at or above
//    it (up to 4096, with positions), and the exact search on the list; ties
//    at the k-th key by a second radix over inverted positions.  A guess that
//    misses falls back to a 4-pass radix select over the whole row, keys > T
//    emitted directly and the keys equal to T taken in position order by a
//    block-wide ordered scan.
// Every sweep over a row loads several elements per thread before using any,
// so that the loads overlap.  The same selection core ranks candidate blocks
// by block maximum, and the chosen blocks are sorted ascending with a
// shared-memory bitonic sort.
#include "common.cuh"
#include "kernels.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 512;        // CTA size for long rows and block ranking
constexpr int kSmemKeys = 40960;      // staged row capacity (160 KB)
constexpr int kMaxSortBlocks = 4096;  // max_blocks supported
constexpr int kBatch = 8;             // elements per thread loaded together in a sweep

// key of a score: order-preserving (larger score, larger key; -0 and +0
// share a key), 0 for NaN and -inf (never selected)
__device__ __forceinline__ uint32_t score_key(float f) {
  f += 0.0f;  // -0 + 0 = +0
  const uint32_t u = __float_as_uint(f);
  const uint32_t k = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
  return (f == f && k > neg_inf_key()) ? k : 0u;
}

template <int NT>
struct SelectShared {
  uint32_t hist[256];
  uint32_t warp_tot[NT / 32];
  uint32_t prefix, remaining, out_count, n_elig;
  int32_t nb;
};

// Block-wide exclusive scan of one uint32 per thread (NT threads).
template <int NT>
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
    uint32_t s = lane < NT / 32 ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < NT / 32) warp_tot[lane] = s;
  }
  __syncthreads();
  total = warp_tot[NT / 32 - 1];
  return (warp ? warp_tot[warp - 1] : 0u) + x - v;
}

// Warp-aggregated slot reservation: every lane with `take` gets a distinct
// slot from *counter (one shared atomic per warp).
__device__ __forceinline__ uint32_t warp_reserve(bool take, uint32_t *counter) {
  const uint32_t m = __ballot_sync(0xffffffffu, take);
  const int lane = threadIdx.x & 31;
  uint32_t base = 0;
  if (m) {
    const int leader = __ffs(m) - 1;
    if (lane == leader) base = atomicAdd(counter, (uint32_t)__popc(m));
    base = __shfl_sync(0xffffffffu, base, leader);
  }
  return base + __popc(m & ((1u << lane) - 1u));
}

// Calls f(i, key) for i = i0 + u*NT + thread over a row of n elements of a
// key source (keys.raw(i): the memory access, valid for any i < n;
// keys.key(i, raw): the key, 0 = ineligible).  Each thread loads kBatch
// elements before converting any, so their loads are in flight together.
// Every thread makes the same number of calls (i >= n gives key 0), so f may
// use warp-wide operations; per thread, i ascends.
template <int NT, class Keys, class F>
__device__ __forceinline__ void sweep(const Keys &keys, int64_t n, F f) {
  for (int64_t i0 = 0; i0 < n; i0 += (int64_t)NT * kBatch) {
    uint32_t r[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t i = i0 + u * NT + threadIdx.x;
      r[u] = keys.raw(i < n ? i : n - 1);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t i = i0 + u * NT + threadIdx.x;
      f(i, i < n ? keys.key(i, r[u]) : 0u);
    }
  }
}

// Select the k largest keys (key 0 = ineligible) of a virtual array of n keys,
// ties by lowest index.  Calls emit(i, slot) once for every selected index i
// with distinct slots 0..min(k, #eligible)-1 and returns min(k, #eligible).
template <int NT, class Keys, class Emit>
__device__ uint32_t select_topk(const Keys &keys, int64_t n, uint32_t k, SelectShared<NT> &sh,
                                Emit emit) {
  // k = 0 (candidate ranking with a one-block budget: only the latest block
  // is kept) selects nothing; the radix search below assumes k >= 1, since
  // with k = 0 no bin would ever hold the k-th key and the threshold would
  // stay at 0.  k is uniform over the block, so every thread returns here.
  static_assert(NT >= 256, "one thread per histogram bin in the scan below");
  if (k == 0u) return 0u;
  // radix select of the k-th largest key; the first pass also counts the
  // eligible keys (the histogram total)
  if (threadIdx.x == 0) {
    sh.prefix = 0;
    sh.remaining = k;
    sh.out_count = 0;
    sh.n_elig = 0;  // reused below: keys equal to the threshold
  }
  uint32_t n_elig = 0;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += NT) sh.hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = sh.prefix;
    const uint32_t hi_mask = shift == 24 ? 0u : (0xffffffffu << (shift + 8));
    // warp-aggregated increments: the lanes holding the same digit add once
    sweep<NT>(keys, n, [&](int64_t, uint32_t key) {
      const bool take = key != 0u && (key & hi_mask) == prefix;
      const uint32_t digit = take ? (key >> shift) & 255u : 256u;
      const uint32_t peers = __match_any_sync(0xffffffffu, digit);
      if (take && (threadIdx.x & 31) == (uint32_t)(__ffs(peers) - 1))
        atomicAdd(&sh.hist[digit], (uint32_t)__popc(peers));
    });
    __syncthreads();
    // scan bins from the top digit down
    const uint32_t remaining = sh.remaining;
    uint32_t h = threadIdx.x < 256 ? sh.hist[255 - threadIdx.x] : 0u;
    uint32_t tot;
    const uint32_t ex = block_scan_u32<NT>(h, sh.warp_tot, tot);
    if (shift == 24) {
      n_elig = tot;
      if (n_elig <= k) break;     // everything eligible is selected
    }
    if (threadIdx.x < 256 && ex < remaining && ex + h >= remaining) {
      sh.prefix = prefix | ((uint32_t)(255 - threadIdx.x) << shift);
      sh.remaining = remaining - ex;
    }
    __syncthreads();
  }
  if (n_elig <= k) {
    sweep<NT>(keys, n, [&](int64_t i, uint32_t key) {
      const uint32_t slot = warp_reserve(key != 0u, &sh.out_count);
      if (key != 0u) emit(i, slot);
    });
    __syncthreads();
    return n_elig;
  }
  const uint32_t T = sh.prefix;
  const uint32_t need_eq = sh.remaining;  // how many keys == T to take
  // keys above the threshold (and a count of the keys equal to it)
  uint32_t eq_local = 0;
  sweep<NT>(keys, n, [&](int64_t i, uint32_t key) {
    const uint32_t slot = warp_reserve(key > T, &sh.out_count);
    if (key > T) emit(i, slot);
    eq_local += key == T;
  });
  eq_local = __reduce_add_sync(0xffffffffu, eq_local);
  if ((threadIdx.x & 31) == 0 && eq_local) atomicAdd(&sh.n_elig, eq_local);
  __syncthreads();
  const uint32_t n_gt = sh.out_count;
  const uint32_t n_eq = sh.n_elig;
  if (n_eq == need_eq) {
    // every key equal to the threshold is selected: no ordering needed
    sweep<NT>(keys, n, [&](int64_t i, uint32_t key) {
      const uint32_t slot = warp_reserve(key == T, &sh.out_count);
      if (key == T) emit(i, slot);
    });
  } else {
    // keys equal to the threshold, lowest indices first
    uint32_t base = 0;
    for (int64_t c0 = 0; c0 < n && base < need_eq; c0 += NT) {
      const int64_t i = c0 + threadIdx.x;
      const uint32_t f = (i < n && keys.key(i, keys.raw(i)) == T) ? 1u : 0u;
      uint32_t tot;
      const uint32_t ex = block_scan_u32<NT>(f, sh.warp_tot, tot);
      if (f && base + ex < need_eq) emit(i, n_gt + base + ex);
      base += tot;
    }
  }
  __syncthreads();
  return k;
}

constexpr int kListCap = 4096;      // compacted candidates of one row (2x the largest k)
constexpr int kSampleSlots = 4;      // register slots per thread in the moment sample

template <int NT>
struct RegShared {
  uint32_t hist[256];
  uint32_t red[6][NT / 32];
  uint32_t warp_tot[NT / 32];
  uint32_t prefix, remaining, bin_count, out_count;
  uint32_t list_key[kListCap];
  int32_t list_pos[kListCap];
};

__device__ __forceinline__ uint32_t keep_above(uint32_t x, int b) {  // bits >= b of x
  return b >= 32 ? 0u : (x >> b) << b;
}

// Block-wide radix search for the k-th largest of the keys that `each` visits
// (each(f) calls f(x) on every key this thread holds; 0 = ineligible), given
// bounds mn <= x <= mx on the eligible keys and at least k of them.  The 8-bit
// digits start at the highest bit in which mn and mx differ (the bits above
// are common to every key in between) and the search stops as soon as the
// k-th key's bin is taken whole.  Result: the selection is every key >= lo,
// lo = whole ? prefix : prefix + 1, plus (if !whole) `rem` keys == prefix.
// One warp scans the 256 bins and clears them; the histogram is all zero on
// entry and on exit.
template <int NT, class Each>
__device__ void radix_kth(Each each, uint32_t mn, uint32_t mx, uint32_t k, RegShared<NT> &sh,
                          uint32_t &prefix, uint32_t &rem, bool &whole) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int hb = mx == mn ? 0 : 32 - __clz(mx ^ mn);
  prefix = keep_above(mx, hb);
  rem = k;
  whole = false;
  while (hb > 0) {
    const int width = hb < 8 ? hb : 8;
    const int shift = hb - width;
    const uint32_t dmask = (1u << width) - 1u;
    const uint32_t pre = prefix;
    each([&](uint32_t x) {
      if (x != 0u && keep_above(x, hb) == pre) atomicAdd(&sh.hist[(x >> shift) & dmask], 1u);
    });
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins top-8l .. top-8l-7 (descending key order)
      const int top = (int)dmask;
      uint32_t h[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int bin = top - (lane * 8 + i);
        h[i] = bin >= 0 ? sh.hist[bin] : 0u;
        if (bin >= 0) sh.hist[bin] = 0u;
        sum += h[i];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      uint32_t e = incl - sum;
      if (e < rem && rem <= incl) {
        bool found = false;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (!found && e + h[i] >= rem) {
            found = true;
            sh.prefix = pre | ((uint32_t)(top - (lane * 8 + i)) << shift);
            sh.remaining = rem - e;
            sh.bin_count = h[i];
          }
          e += h[i];
        }
      }
    }
    __syncthreads();
    prefix = sh.prefix;
    rem = sh.remaining;
    const uint32_t n_eq = sh.bin_count;
    hb = shift;
    if (n_eq == rem) {
      whole = true;
      break;
    }
  }
}

// Selection for a row held in registers: thread t owns positions t + j*NT
// (key[j], 0 = ineligible; slots j >= jn hold no keys).
//  1. Count the eligible keys; if at most k, all are selected.
//  2. Guess a threshold from the moments of a strided sample (kSampleSlots
//     slots per thread) and compact every key >= the guess into a
//     shared-memory list.  With between k and kListCap keys listed, the exact
//     search runs on the list alone; otherwise (a missed guess) on the whole
//     row.  Any guess is safe: only the cost depends on it.
//  3. Emit the keys >= lo; keys equal to the threshold, if only some of them
//     are taken, go in position order by a block scan over the row.
template <int NT, int KPT, class Emit>
__device__ uint32_t select_topk_regs(const uint32_t (&key)[KPT], int jn, uint32_t k,
                                     RegShared<NT> &sh, Emit emit) {
  constexpr int kStride = KPT / kSampleSlots > 0 ? KPT / kSampleSlots : 1;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  uint32_t cnt = 0, mx = 0, f_cnt = 0;
  float f_sum = 0.f, f_sq = 0.f;   // moments of a strided sample of the finite scores
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    if (j >= jn) break;
    const uint32_t x = key[j];
    cnt += x != 0u;
    mx = max(mx, x);
    if (j % kStride == 0) {
      const float f = __uint_as_float((x & 0x80000000u) ? x ^ 0x80000000u : ~x);
      const bool fin = x != 0u && fabsf(f) <= 3.0e38f;
      f_cnt += fin;
      f_sum += fin ? f : 0.f;
      f_sq += fin ? f * f : 0.f;
    }
  }
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  mx = __reduce_max_sync(0xffffffffu, mx);
  f_cnt = __reduce_add_sync(0xffffffffu, f_cnt);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    f_sum += __shfl_xor_sync(0xffffffffu, f_sum, o);
    f_sq += __shfl_xor_sync(0xffffffffu, f_sq, o);
  }
  if (lane == 0) {
    sh.red[0][warp] = cnt;
    sh.red[2][warp] = mx;
    sh.red[3][warp] = f_cnt;
    sh.red[4][warp] = __float_as_uint(f_sum);
    sh.red[5][warp] = __float_as_uint(f_sq);
  }
  for (int i = t; i < 256; i += NT) sh.hist[i] = 0;
  if (t == 0) sh.out_count = 0;
  __syncthreads();
  uint32_t n_elig = 0;
  mx = 0;
  f_cnt = 0;
  f_sum = 0.f;
  f_sq = 0.f;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    n_elig += sh.red[0][w];
    mx = max(mx, sh.red[2][w]);
    f_cnt += sh.red[3][w];
    f_sum += __uint_as_float(sh.red[4][w]);
    f_sq += __uint_as_float(sh.red[5][w]);
  }
  if (n_elig <= k) {  // everything eligible is selected
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      if (j >= jn) break;
      const bool take = key[j] != 0u;
      const uint32_t slot = warp_reserve(take, &sh.out_count);
      if (take) emit(j * NT + t, slot);
    }
    __syncthreads();
    return n_elig;
  }
  uint32_t prefix, rem;
  bool whole;
  bool listed = false;
  uint32_t n_list = 0;
  // threshold guess: the score expected to have about 2k + 64 scores above it
  // if the row were normal with its sample's mean and deviation (the same
  // value in every thread; any guess is safe, a bad one only falls through to
  // the search over the whole row)
  uint32_t t_est = 0;
  if (f_cnt > 1) {
    const float mean = f_sum / (float)f_cnt;
    const float sd = sqrtf(fmaxf(f_sq / (float)f_cnt - mean * mean, 0.f));
    const float p = (float)(2u * k + 64u) / (float)n_elig;
    if (p < 1.f && sd > 0.f) t_est = score_key(mean + 1.41421356f * erfcinvf(2.f * p) * sd);
  }
  if (t_est != 0u) {
    // keys >= t_est are counted and offset by a block scan, and written to
    // the list if at least k and at most its capacity are: the list then
    // holds the whole selection
    uint32_t mine = 0;
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      if (j >= jn) break;
      mine += key[j] >= t_est;
    }
    uint32_t off = block_scan_u32<NT>(mine, sh.warp_tot, n_list);
    if (n_list >= k && n_list <= (uint32_t)kListCap) {
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        if (j >= jn) break;
        if (key[j] >= t_est) {
          sh.list_key[off] = key[j];
          sh.list_pos[off] = j * NT + t;
          ++off;
        }
      }
      __syncthreads();
      listed = true;
      radix_kth<NT>(
          [&](auto f) {
            for (int i = t; i < (int)n_list; i += NT) f(sh.list_key[i]);
          },
          t_est, mx, k, sh, prefix, rem, whole);
    }
  }
  if (!listed) {
    // every eligible key is >= 1
    radix_kth<NT>(
        [&](auto f) {
#pragma unroll
          for (int j = 0; j < KPT; ++j)
            if (j < jn) f(key[j]);
        },
        1u, mx, k, sh, prefix, rem, whole);
  }
  const uint32_t lo = whole ? prefix : prefix + 1u;
  if (listed) {
    for (int i0 = 0; i0 < (int)n_list; i0 += NT) {
      const int i = i0 + t;
      const uint32_t x = i < (int)n_list ? sh.list_key[i] : 0u;
      const bool take = x != 0u && x >= lo;
      const uint32_t slot = warp_reserve(take, &sh.out_count);
      if (take) emit(sh.list_pos[i], slot);
    }
  } else {
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      if (j >= jn) break;
      const uint32_t x = key[j];
      const bool take = x != 0u && x >= lo;
      const uint32_t slot = warp_reserve(take, &sh.out_count);
      if (take) emit(j * NT + t, slot);
    }
  }
  if (!whole) {
    // keys equal to the threshold, lowest positions first (position order is
    // slot-major: j, then thread)
    const uint32_t base_slot = k - rem;
    uint32_t base = 0;
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      if (j >= jn || base >= rem) break;
      const uint32_t f = key[j] == prefix ? 1u : 0u;
      uint32_t tot;
      const uint32_t ex = block_scan_u32<NT>(f, sh.warp_tot, tot);
      if (f && base + ex < rem) emit(j * NT + t, base_slot + base + ex);
      base += tot;
    }
  }
  __syncthreads();
  return k;
}

// Key sources (see sweep()).  Row view: the scores of query q, in full mode
// (entries 0..len-1) or pool mode (slots, mapped to entries through the
// query's candidate blocks, read from a shared-memory copy).
struct RowView {
  const float *row;
  const int32_t *cand;  // candidate blocks of this query or nullptr
  int block;
  int64_t n_vis;
  __device__ __forceinline__ int64_t entry(int64_t s) const {
    return cand ? (int64_t)cand[s / block] * block + s % block : s;
  }
  __device__ __forceinline__ uint32_t raw(int64_t s) const {
    return __float_as_uint(__ldg(row + s));
  }
  __device__ __forceinline__ uint32_t key(int64_t s, uint32_t r) const {
    if (cand && entry(s) >= n_vis) return 0u;
    return score_key(__uint_as_float(r));
  }
};

struct SmemKeys {
  const uint32_t *k;
  __device__ __forceinline__ uint32_t raw(int64_t i) const { return k[i]; }
  __device__ __forceinline__ uint32_t key(int64_t, uint32_t r) const { return r; }
};

// Score rows read straight from memory take the vectorised listing sweep
// when they have no candidate blocks.
template <class Keys>
constexpr bool kPlainRows = false;
template <>
constexpr bool kPlainRows<RowView> = true;
template <class Keys>
__device__ __forceinline__ bool plain_rows_cand(const Keys &) { return true; }
template <>
__device__ __forceinline__ bool plain_rows_cand<RowView>(const RowView &k) {
  return k.cand != nullptr;
}

// Block view: key of block b = max key over its visible entries, plus one, so
// every block is eligible (the pool is a budget, filled whatever the scores).
struct BlockView {
  const float *row;
  int block;
  int64_t n_vis;
  __device__ __forceinline__ uint32_t raw(int64_t b) const {
    uint32_t m = 0;
    const int64_t j1 = min((b + 1) * block, n_vis);
    for (int64_t j = b * block; j < j1; ++j) m = max(m, float_key(__ldg(row + j)));
    return m + 1u;
  }
  __device__ __forceinline__ uint32_t key(int64_t, uint32_t r) const { return r; }
};

// Visible entries and row length of query q; in pool mode the query's
// candidate blocks are also copied to scand (the first -1 ends the row).
template <int NT>
__device__ void row_geometry(const Batch &b, int q, const int32_t *cand_blocks, int block,
                             int max_blocks, int64_t ld, int32_t *scand, int64_t &n_vis,
                             int64_t &row_len, int &err, SelectShared<NT> &sh) {
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
    for (int i0 = 0; i0 < max_blocks; i0 += NT * kBatch) {
      int32_t v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        v[u] = __ldg(cb + min(i0 + u * NT + (int)threadIdx.x, max_blocks - 1));
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = i0 + u * NT + threadIdx.x;
        if (i < max_blocks) {
          scand[i] = v[u];
          if (v[u] < 0) atomicMin(&sh.nb, i);
        }
      }
    }
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

// minimum residency chosen so the key registers do not spill

// Exact top k of the n listed (key, position) pairs in sh.list_key /
// sh.list_pos, given bounds mn <= key <= mx on every listed key and at least
// k listed keys: the k-th key by radix, and the keys equal to it, if only
// some are taken, by a second radix over their inverted positions (lowest
// positions first).  emit(i, slot) gets the list index i of every selected
// pair, with distinct slots 0..k-1.
template <int NT, class Emit>
__device__ void select_listed(int n_list, uint32_t mn, uint32_t mx, uint32_t k,
                              RegShared<NT> &sh, Emit emit) {
  const int t = threadIdx.x;
  if (t == 0) sh.out_count = 0;
  __syncthreads();
  uint32_t prefix, rem;
  bool whole;
  radix_kth<NT>(
      [&](auto f) {
        for (int i = t; i < n_list; i += NT) f(sh.list_key[i]);
      },
      mn, mx, k, sh, prefix, rem, whole);
  const uint32_t lo = whole ? prefix : prefix + 1u;
  for (int i0 = 0; i0 < n_list; i0 += NT) {
    const int i = i0 + t;
    const uint32_t x = i < n_list ? sh.list_key[i] : 0u;
    const bool take = x != 0u && x >= lo;
    const uint32_t slot = warp_reserve(take, &sh.out_count);
    if (take) emit(i, slot);
  }
  if (!whole) {
    // the rem lowest positions among the listed keys equal to prefix:
    // largest inverted positions (positions are below 2^31, so these keys are
    // nonzero and distinct)
    auto inv = [&](int i) -> uint32_t {
      return sh.list_key[i] == prefix ? 0xffffffffu - (uint32_t)sh.list_pos[i] : 0u;
    };
    uint32_t p2, rem2;
    bool whole2;
    radix_kth<NT>(
        [&](auto f) {
          for (int i = t; i < n_list; i += NT) f(inv(i));
        },
        0x80000000u, 0xffffffffu, rem, sh, p2, rem2, whole2);
    const uint32_t lo2 = whole2 ? p2 : p2 + 1u;
    for (int i0 = 0; i0 < n_list; i0 += NT) {
      const int i = i0 + t;
      const uint32_t y = i < n_list ? inv(i) : 0u;
      const bool take = y != 0u && (y >= lo2 || (!whole2 && y == p2));
      const uint32_t slot = warp_reserve(take, &sh.out_count);
      if (take) emit(i, slot);
    }
  }
  __syncthreads();
}

// Listing sweep over a plain score row (no candidate blocks): every score
// f >= g is appended (its key and position) to the shared list, the counter
// running on past the capacity.  Equivalent to comparing keys with
// score_key(g) when that key is nonzero: the key map is monotone, -0 and +0
// compare equal both ways, and NaN and -inf fail the float comparison.  The
// row is read 16 bytes per load, four loads per thread in flight; a thread's
// takes are placed by one warp scan per 16 scores.  Returns this thread's
// largest listed key (0 if none).
template <int NT>
__device__ uint32_t list_row_fast(const float *__restrict__ row, int64_t n, float g,
                                  RegShared<NT> &sh) {
  const int t = threadIdx.x, lane = t & 31;
  uint32_t mx = 0;
  auto put = [&](uint32_t slot, float f, int64_t i) {
    const uint32_t x = score_key(f);
    if (slot < (uint32_t)kListCap) {
      sh.list_key[slot] = x;
      sh.list_pos[slot] = (int32_t)i;
    }
    mx = max(mx, x);
  };
  // scalar edges: the scores before the first 16-byte boundary and after the
  // last whole vector (at most three each; the row is 4-byte aligned)
  const int64_t head0 = (int64_t)(((16u - ((uint32_t)(uintptr_t)row & 15u)) & 15u) >> 2);
  const int64_t head = head0 < n ? head0 : n;
  const int64_t nvec = (n - head) >> 2;
  const int64_t tail0 = head + 4 * nvec;
  if (t < 32) {
    const int64_t i = lane < head ? (int64_t)lane : tail0 + (lane - head);
    const bool in = lane < head || (lane >= head && i < n && lane - head < 3);
    const float f = in ? __ldg(row + i) : 0.f;
    const bool take = in && f >= g;
    const uint32_t slot = warp_reserve(take, &sh.out_count);
    if (take) put(slot, f, i);
  }
  const float4 *v4 = reinterpret_cast<const float4 *>(row + head);
  constexpr int kV = 4;
  for (int64_t j0 = 0; j0 < nvec; j0 += (int64_t)NT * kV) {
    float4 v[kV];
#pragma unroll
    for (int u = 0; u < kV; ++u) {
      const int64_t j = j0 + u * NT + t;
      v[u] = j < nvec ? __ldg(v4 + j) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
    uint32_t c = 0;
#pragma unroll
    for (int u = 0; u < kV; ++u)
      c += (uint32_t)(v[u].x >= g) + (uint32_t)(v[u].y >= g) + (uint32_t)(v[u].z >= g) +
           (uint32_t)(v[u].w >= g);
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
    if (tot == 0u) continue;
    uint32_t base = 0;
    if (lane == 31) base = atomicAdd(&sh.out_count, tot);
    uint32_t slot = __shfl_sync(0xffffffffu, base, 31) + incl - c;
    if (c == 0u) continue;
#pragma unroll
    for (int u = 0; u < kV; ++u) {
      const int64_t i = head + 4 * (j0 + u * NT + t);
      if (v[u].x >= g) put(slot++, v[u].x, i);
      if (v[u].y >= g) put(slot++, v[u].y, i + 1);
      if (v[u].z >= g) put(slot++, v[u].z, i + 2);
      if (v[u].w >= g) put(slot++, v[u].w, i + 3);
    }
  }
  return mx;
}

// Long rows (past the register path): a threshold guess from the moments of
// every 16th key, then one sweep that lists the keys at or above it (up to
// kListCap, with their positions).  With between k and kListCap keys listed
// the exact search runs on the list: the k-th key by radix, and the keys equal
// to it, if only some are taken, by a second radix over their inverted
// positions (lowest positions first).  Returns false, having emitted nothing,
// when the guess misses; the caller then searches the whole row.
template <int NT, class Keys, class Emit>
__device__ bool select_topk_listed(const Keys &keys, int64_t n, uint32_t k, RegShared<NT> &sh,
                                   Emit emit) {
  constexpr int kS = 16;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  uint32_t s_cnt = 0, f_cnt = 0;
  float f_sum = 0.f, f_sq = 0.f;
#pragma unroll 4
  for (int64_t i = (int64_t)t * kS; i < n; i += (int64_t)NT * kS) {
    const uint32_t x = keys.key(i, keys.raw(i));
    if (x != 0u) {
      ++s_cnt;
      const float f = __uint_as_float((x & 0x80000000u) ? x ^ 0x80000000u : ~x);
      if (fabsf(f) <= 3.0e38f) {
        ++f_cnt;
        f_sum += f;
        f_sq += f * f;
      }
    }
  }
  s_cnt = __reduce_add_sync(0xffffffffu, s_cnt);
  f_cnt = __reduce_add_sync(0xffffffffu, f_cnt);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    f_sum += __shfl_xor_sync(0xffffffffu, f_sum, o);
    f_sq += __shfl_xor_sync(0xffffffffu, f_sq, o);
  }
  if (lane == 0) {
    sh.red[0][warp] = s_cnt;
    sh.red[3][warp] = f_cnt;
    sh.red[4][warp] = __float_as_uint(f_sum);
    sh.red[5][warp] = __float_as_uint(f_sq);
  }
  for (int i = t; i < 256; i += NT) sh.hist[i] = 0;
  if (t == 0) sh.out_count = 0;
  __syncthreads();
  s_cnt = 0;
  f_cnt = 0;
  f_sum = 0.f;
  f_sq = 0.f;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    s_cnt += sh.red[0][w];
    f_cnt += sh.red[3][w];
    f_sum += __uint_as_float(sh.red[4][w]);
    f_sq += __uint_as_float(sh.red[5][w]);
  }
  // the same guess as the register path, with the eligible count estimated
  // from the sample (any guess is safe)
  if (f_cnt <= 1) return false;
  const float n_elig = (float)s_cnt * (float)kS;
  const float mean = f_sum / (float)f_cnt;
  const float sd = sqrtf(fmaxf(f_sq / (float)f_cnt - mean * mean, 0.f));
  const float p = (float)(2u * k + 64u) / n_elig;
  if (!(p < 1.f) || !(sd > 0.f)) return false;
  const float g = mean + 1.41421356f * erfcinvf(2.f * p) * sd;
  const uint32_t t_est = score_key(g);
  if (t_est == 0u) return false;
  // list the keys >= t_est; the counter runs on past the capacity
  uint32_t mx = 0;
  if constexpr (kPlainRows<Keys>) {
    if (keys.cand == nullptr) mx = list_row_fast<NT>(keys.row, n, g, sh);
  }
  if (!kPlainRows<Keys> || plain_rows_cand(keys)) {
    sweep<NT>(keys, n, [&](int64_t i, uint32_t x) {
      const bool take = x != 0u && x >= t_est;
      const uint32_t slot = warp_reserve(take, &sh.out_count);
      if (take && slot < (uint32_t)kListCap) {
        sh.list_key[slot] = x;
        sh.list_pos[slot] = (int32_t)i;
      }
      mx = max(mx, take ? x : 0u);
    });
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) sh.red[2][warp] = mx;
  __syncthreads();
  const uint32_t n_list = sh.out_count;
  mx = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) mx = max(mx, sh.red[2][w]);
  __syncthreads();
  if (t == 0) sh.out_count = 0;
  __syncthreads();
  if (n_list < k || n_list > (uint32_t)kListCap) return false;
  select_listed<NT>((int)n_list, t_est, mx, k, sh,
                    [&](int i, uint32_t slot) { emit(sh.list_pos[i], slot); });
  return true;
}

template <int NT, int KPT>
__global__ void __launch_bounds__(NT, NT >= 512 ? 1 : KPT >= 64 ? 2 : KPT >= 32 ? 3 : 4)
topk_kernel(Batch b, const float *__restrict__ scores, int64_t ld, int k,
            const int32_t *__restrict__ cand_blocks, int block, int max_blocks,
            int32_t *__restrict__ idx, int32_t *__restrict__ count, int32_t *__restrict__ d_err,
            int64_t staged) {
  // dynamic shared memory: [staged keys (staged)][candidate blocks (pool mode)]
  extern __shared__ __align__(16) uint32_t smem_dyn[];
  uint32_t *skeys = smem_dyn;
  int32_t *scand = reinterpret_cast<int32_t *>(smem_dyn + staged);
  __shared__ SelectShared<NT> sh;
  __shared__ RegShared<NT> rsh;
  const int q = blockIdx.x;
  int err = 0;
  int64_t n_vis, row_len;
  row_geometry(b, q, cand_blocks, block, max_blocks, ld, scand, n_vis, row_len, err, sh);
  RowView view{scores + (int64_t)q * ld, cand_blocks ? scand : nullptr, block, n_vis};
  int32_t *out = idx + (int64_t)q * k;
  auto emit = [&](int64_t s, uint32_t slot) { out[slot] = (int32_t)view.entry(s); };
  uint32_t got;
  if (row_len <= (int64_t)NT * KPT) {
    uint32_t key[KPT];
    const int rl = (int)row_len;
    const int jn = (rl + NT - 1) / NT;
    // every load first, at clamped (always valid) addresses, then the keys:
    // no branch separates the loads, so they are all in flight together
#pragma unroll
    for (int j = 0; j < KPT; ++j)
      key[j] = j < jn ? view.raw(min(j * NT + (int)threadIdx.x, rl - 1)) : 0u;
    if (view.cand) {
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        const int s = j * NT + threadIdx.x;
        key[j] = s < rl ? view.key(s, key[j]) : 0u;
      }
    } else {
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        const int s = j * NT + threadIdx.x;
        key[j] = s < rl ? score_key(__uint_as_float(key[j])) : 0u;
      }
    }
    got = select_topk_regs<NT, KPT>(key, jn, (uint32_t)k, rsh, emit);
  } else if (row_len <= staged) {
    sweep<NT>(view, row_len, [&](int64_t s, uint32_t x) {
      if (s < row_len) skeys[s] = x;
    });
    __syncthreads();
    if (select_topk_listed<NT>(SmemKeys{skeys}, row_len, (uint32_t)k, rsh, emit))
      got = (uint32_t)k;
    else
      got = select_topk<NT>(SmemKeys{skeys}, row_len, (uint32_t)k, sh, emit);
  } else {
    if (select_topk_listed<NT>(view, row_len, (uint32_t)k, rsh, emit))
      got = (uint32_t)k;
    else
      got = select_topk<NT>(view, row_len, (uint32_t)k, sh, emit);
  }
  for (int i = (int)got + threadIdx.x; i < k; i += NT) out[i] = -1;
  if (threadIdx.x == 0) count[q] = (int32_t)got;
  err = __reduce_or_sync(0xffffffffu, err);
  if (threadIdx.x == 0) raise_err(d_err, err);
}

// Full-visible rows of moderate length (4097 to 16384 keys) with CTAs that
// hold no row in registers (45 registers, 35 KB of shared memory: six rows in
// flight per SM instead of two): the row is read twice from L2/HBM, once for
// the strided sample that sets the threshold guess and once to list the keys
// at or above it, and the exact search runs on the list (the same selection
// as the long-row path).  A guess that misses falls back to the 4-pass radix
// select over the row.
template <int NT>
__global__ void __launch_bounds__(NT, 6)   // six CTAs per SM: 40 registers, 35 KB each
topk_list_kernel(Batch b, const float *__restrict__ scores, int64_t ld, int k,
                 int32_t *__restrict__ idx, int32_t *__restrict__ count,
                 int32_t *__restrict__ d_err) {
  __shared__ SelectShared<NT> sh;
  __shared__ RegShared<NT> rsh;
  const int q = blockIdx.x;
  int err = 0;
  int64_t n_vis, row_len;
  row_geometry(b, q, nullptr, 1, 1, ld, nullptr, n_vis, row_len, err, sh);
  RowView view{scores + (int64_t)q * ld, nullptr, 1, n_vis};
  int32_t *out = idx + (int64_t)q * k;
  auto emit = [&](int64_t s, uint32_t slot) { out[slot] = (int32_t)s; };
  uint32_t got;
  if (select_topk_listed<NT>(view, row_len, (uint32_t)k, rsh, emit))
    got = (uint32_t)k;
  else
    got = select_topk<NT>(view, row_len, (uint32_t)k, sh, emit);
  for (int i = (int)got + threadIdx.x; i < k; i += NT) out[i] = -1;
  if (threadIdx.x == 0) count[q] = (int32_t)got;
  err = __reduce_or_sync(0xffffffffu, err);
  if ((threadIdx.x & 31) == 0) raise_err(d_err, err);
}

__global__ void __launch_bounds__(kThreads)
candidate_blocks_kernel(Batch b, const float *__restrict__ scores, int64_t ld, int block,
                        int max_blocks, int32_t *__restrict__ blocks,
                        int32_t *__restrict__ nblocks, int64_t staged) {
  extern __shared__ uint32_t smem_keys[];
  __shared__ SelectShared<kThreads> sh;
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
    sweep<kThreads>(view, n, [&](int64_t i, uint32_t x) {
      if (i < n) smem_keys[i] = x;
    });
    __syncthreads();
    select_topk<kThreads>(SmemKeys{smem_keys}, n, (uint32_t)(max_blocks - 1), sh, emit);
  } else {
    select_topk<kThreads>(view, n, (uint32_t)(max_blocks - 1), sh, emit);
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

// ---------------------------------------------------------------------------
// Index score streamed into the top-K (full-visible rows): the scoring pass
// appends only the (entry, score) pairs at or above a per-query threshold to
// a bounded list, and the selection runs on that list.
//  1. sample pass (index score over every kStreamStride-th key tile)
//  2. stream_threshold_kernel: per query, the score a normal row with the
//     sample's mean and deviation would have `target` scores above; rows of at
//     most kStreamCap visible entries list everything (threshold -inf)
//  3. list pass (index score, appending epilogue)
//  4. stream_select_kernel: exact top k of the list when it holds every entry
//     at or above the threshold and at least k of them (or every visible
//     entry); any other row (a missed guess) is queued for
//  5. stream_fallback_kernel: the row rescored on the CUDA cores in blocks,
//     with the scoring epilogue's arithmetic, and an exact running top k.
// Exactness: a list holding every entry with score >= thr, with at least k of
// them, holds the k best entries and every entry tied with the k-th (all
// have score >= the k-th score >= thr); ties are broken by lowest entry.
// ---------------------------------------------------------------------------
constexpr int kStreamCap = kStreamListCap;
static_assert(kStreamCap <= kListCap, "a query's list fits the selection's shared arrays");

__device__ __forceinline__ int64_t stream_nvis(const Batch &b, int q, int64_t max_len) {
  int64_t nv = n_visible(b.q_pos[q], b.ratio);
  const int64_t kvl = b.kv_len[b.q_req[q]];
  if (nv > kvl) nv = kvl;
  return nv < max_len ? nv : max_len;
}

// One warp per query.  Also clears the list counters and the fallback queue.
__global__ void __launch_bounds__(256)
stream_threshold_kernel(Batch b, int64_t max_len, int k, int stride, StreamWs ws) {
  if (blockIdx.x == 0 && threadIdx.x < 2) ws.hdr[threadIdx.x] = 0u;
  const int lane = threadIdx.x & 31;
  const int q = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (q >= b.num_q) return;
  const int64_t nv = stream_nvis(b, q, max_len);
  float thr = -INFINITY;
  if (nv > kStreamCap) {
    const int64_t walked = ((nv + 127) / 128 + stride - 1) / stride;
    const float *row = ws.sample + (int64_t)q * ws.sample_ld;
    float n = 0.f, sum = 0.f, sq = 0.f;
    for (int64_t c = lane; c < walked * 128; c += 32) {
      const int64_t s = (c >> 7) * stride * 128 + (c & 127);
      if (s < nv) {
        const float v = row[c];
        if (fabsf(v) <= 3.0e38f) {
          n += 1.f;
          sum += v;
          sq += v * v;
        }
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      n += __shfl_xor_sync(0xffffffffu, n, o);
      sum += __shfl_xor_sync(0xffffffffu, sum, o);
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
    }
    const float target = fminf(2.f * k + 64.f, 0.5f * (k + kStreamCap));
    const float p = target / (float)nv;
    if (n > 1.f && p < 1.f) {
      const float mean = sum / n;
      const float sd = sqrtf(fmaxf(sq / n - mean * mean, 0.f));
      if (sd > 0.f) thr = mean + 1.41421356f * erfcinvf(2.f * p) * sd;
    }
  }
  if (lane == 0) {
    ws.thr[q] = thr;
    ws.cnt[q] = 0u;
  }
}

// Exact top k of a query's list, or queue the query for the fallback.
template <int NT>
__global__ void __launch_bounds__(NT)
stream_select_kernel(Batch b, int64_t max_len, int k, StreamWs ws, int32_t *__restrict__ idx,
                     int32_t *__restrict__ count) {
  __shared__ RegShared<NT> sh;
  const int q = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t c = ws.cnt[q];
  const bool all = ws.thr[q] == -INFINITY;   // every visible entry was offered
  if (c > (uint32_t)kStreamCap || (!all && c < (uint32_t)k)) {
    if (t == 0) ws.fb_rows[atomicAdd(&ws.hdr[0], 1u)] = q;
    return;
  }
  for (int i = t; i < 256; i += NT) sh.hist[i] = 0u;
  const int n = (int)c;
  uint32_t mn = 0xffffffffu, mx = 0u, ne = 0u;
  for (int i = t; i < n; i += NT) {
    const int64_t o = (int64_t)q * kStreamCap + i;
    const uint32_t key = score_key(ws.val[o]);
    sh.list_key[i] = key;
    sh.list_pos[i] = ws.ent[o];
    if (key != 0u) {
      mn = min(mn, key);
      mx = max(mx, key);
      ++ne;
    }
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  ne = __reduce_add_sync(0xffffffffu, ne);
  if (lane == 0) {
    sh.red[0][warp] = mn;
    sh.red[1][warp] = mx;
    sh.red[2][warp] = ne;
  }
  if (t == 0) sh.out_count = 0u;
  __syncthreads();
  mn = 0xffffffffu;
  mx = 0u;
  ne = 0u;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    mn = min(mn, sh.red[0][w]);
    mx = max(mx, sh.red[1][w]);
    ne += sh.red[2][w];
  }
  int32_t *out = idx + (int64_t)q * k;
  uint32_t got;
  if (ne <= (uint32_t)k) {
    for (int i0 = 0; i0 < n; i0 += NT) {
      const int i = i0 + t;
      const bool take = i < n && sh.list_key[i] != 0u;
      const uint32_t slot = warp_reserve(take, &sh.out_count);
      if (take) out[slot] = sh.list_pos[i];
    }
    got = ne;
  } else {
    select_listed<NT>(n, mn, mx, (uint32_t)k, sh,
                      [&](int i, uint32_t slot) { out[slot] = sh.list_pos[i]; });
    got = (uint32_t)k;
  }
  for (int i = (int)got + t; i < k; i += NT) out[i] = -1;
  if (t == 0) count[q] = (int32_t)got;
}

// MXFP4 row segment (32 elements = 16 bytes of codes, one power-of-two scale)
// decoded exactly to fp32
__device__ __forceinline__ void mx_decode32(const uint8_t *codes, float scale, float (&v)[32]) {
  const uint4 c = __ldg(reinterpret_cast<const uint4 *>(codes));
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h[4];
    e2m1x8_f16x8(w[i], h);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 x = *reinterpret_cast<const __half2 *>(&h[j]);
      v[8 * i + 2 * j] = __low2float(x) * scale;
      v[8 * i + 2 * j + 1] = __high2float(x) * scale;
    }
  }
}

constexpr int kFbBlock = 1024;   // entries rescored per round of the fallback

// Fallback rows: the whole row rescored on the CUDA cores in rounds of
// kFbBlock entries, each round merged with the running top k (kept in the
// list arrays) by the exact list selection.  Per-head dots in fp32 (exact for
// MXFP4 operands whose group sums fit 24 bits, as the tensor-core dots are),
// then the scoring epilogue's own head combination: (w/2) * (x + |x|) summed
// in four chains by head index mod 4, 32 heads per chain segment.
template <int HI>
__global__ void __launch_bounds__(256)
stream_fallback_kernel(Batch b, int64_t max_len, int k, const uint8_t *__restrict__ q_fp4,
                       const float *__restrict__ q_scale, const float *__restrict__ head_w,
                       const uint8_t *__restrict__ k_fp4, const float *__restrict__ k_scale,
                       StreamWs ws, int32_t *__restrict__ idx, int32_t *__restrict__ count) {
  constexpr int NT = 256;
  __shared__ RegShared<NT> sh;
  __shared__ float w2[HI];
  __shared__ int row_slot;
  // dynamic: the query dequantised [HI][128] f32, then the merge's output
  // (keys and entries of up to 2048 pairs)
  extern __shared__ __align__(16) uint32_t fb_dyn[];
  float *qv = reinterpret_cast<float *>(fb_dyn);
  uint32_t *tmp_key = fb_dyn + HI * 128;
  int32_t *tmp_ent = reinterpret_cast<int32_t *>(tmp_key + 2048);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int i = t; i < 256; i += NT) sh.hist[i] = 0u;
  while (true) {
    __syncthreads();
    if (t == 0) row_slot = (int)atomicAdd(&ws.hdr[1], 1u);
    __syncthreads();
    const int slot = row_slot;
    if (slot >= (int)ws.hdr[0]) break;
    const int q = ws.fb_rows[slot];
    const int64_t nv = stream_nvis(b, q, max_len);
    const int64_t kv0 = b.kv_start[b.q_req[q]];
    for (int i = t; i < HI * 4; i += NT) {   // 32-element segments of the query
      float v[32];
      mx_decode32(q_fp4 + ((int64_t)q * HI) * 64 + i * 16, q_scale[(int64_t)q * HI * 4 + i], v);
#pragma unroll
      for (int j = 0; j < 32; ++j) qv[i * 32 + j] = v[j];
    }
    for (int h = t; h < HI; h += NT) w2[h] = 0.5f * (head_w ? head_w[(int64_t)q * HI + h] : 1.f);
    __syncthreads();
    int n_cur = 0;
    for (int64_t s0 = 0; s0 < nv; s0 += kFbBlock) {
      const int nb = (int)min((int64_t)kFbBlock, nv - s0);
      for (int i = t; i < nb; i += NT) {
        const int64_t j = s0 + i;
        const uint8_t *kc = k_fp4 + (kv0 + j) * 64;
        const float *ks = k_scale + (kv0 + j) * 4;
        float dot[HI];
#pragma unroll
        for (int h = 0; h < HI; ++h) dot[h] = 0.f;
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          float kx[32];
          mx_decode32(kc + g * 16, __ldg(ks + g), kx);
#pragma unroll
          for (int h = 0; h < HI; ++h) {
#pragma unroll
            for (int d = 0; d < 32; ++d) dot[h] = fmaf(qv[h * 128 + g * 32 + d], kx[d], dot[h]);
          }
        }
        float acc = 0.f;
        constexpr int LW = HI < 32 ? HI : 32;
#pragma unroll
        for (int l = 0; l < HI / LW; ++l) {
          float a0 = acc, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
          for (int h = l * LW; h < l * LW + LW; h += 4) {
            a0 = fmaf(w2[h], dot[h] + fabsf(dot[h]), a0);
            a1 = fmaf(w2[h + 1], dot[h + 1] + fabsf(dot[h + 1]), a1);
            a2 = fmaf(w2[h + 2], dot[h + 2] + fabsf(dot[h + 2]), a2);
            a3 = fmaf(w2[h + 3], dot[h + 3] + fabsf(dot[h + 3]), a3);
          }
          acc = (a0 + a1) + (a2 + a3);
        }
        sh.list_key[n_cur + i] = score_key(acc);
        sh.list_pos[n_cur + i] = (int32_t)j;
      }
      __syncthreads();
      // merge: the k best of the running set and this round
      const int n = n_cur + nb;
      uint32_t mn = 0xffffffffu, mx = 0u, ne = 0u;
      for (int i = t; i < n; i += NT) {
        const uint32_t key = sh.list_key[i];
        if (key != 0u) {
          mn = min(mn, key);
          mx = max(mx, key);
          ++ne;
        }
      }
      mn = __reduce_min_sync(0xffffffffu, mn);
      mx = __reduce_max_sync(0xffffffffu, mx);
      ne = __reduce_add_sync(0xffffffffu, ne);
      if (lane == 0) {
        sh.red[0][warp] = mn;
        sh.red[1][warp] = mx;
        sh.red[2][warp] = ne;
      }
      if (t == 0) sh.out_count = 0u;
      __syncthreads();
      mn = 0xffffffffu;
      mx = 0u;
      ne = 0u;
#pragma unroll
      for (int w = 0; w < NT / 32; ++w) {
        mn = min(mn, sh.red[0][w]);
        mx = max(mx, sh.red[1][w]);
        ne += sh.red[2][w];
      }
      auto keep = [&](int i, uint32_t slot) {
        tmp_key[slot] = sh.list_key[i];
        tmp_ent[slot] = sh.list_pos[i];
      };
      if (ne <= (uint32_t)k) {
        for (int i0 = 0; i0 < n; i0 += NT) {
          const int i = i0 + t;
          const bool take = i < n && sh.list_key[i] != 0u;
          const uint32_t sl = warp_reserve(take, &sh.out_count);
          if (take) keep(i, sl);
        }
        __syncthreads();
        n_cur = (int)ne;
      } else {
        select_listed<NT>(n, mn, mx, (uint32_t)k, sh, keep);
        n_cur = k;
      }
      __syncthreads();
      for (int i = t; i < n_cur; i += NT) {
        sh.list_key[i] = tmp_key[i];
        sh.list_pos[i] = tmp_ent[i];
      }
      __syncthreads();
    }
    int32_t *out = idx + (int64_t)q * k;
    for (int i = t; i < k; i += NT) out[i] = i < n_cur ? sh.list_pos[i] : -1;
    if (t == 0) count[q] = n_cur;
  }
}

}  // namespace

int topk_launch(const Batch &b, const float *scores, int64_t ld, int k,
                const int32_t *cand_blocks, int block, int max_blocks, int32_t *idx,
                int32_t *count, int32_t *blocks_out, int32_t *nblocks_out, int32_t *d_err,
                cudaStream_t st) {
  if (b.num_q == 0) return CSA2_OK;
  // rows of up to 16384 keys are held in registers (KPT keys per thread,
  // sized to the longest possible row); longer rows are staged in shared
  // memory up to kSmemKeys, else re-read from L2 in each pass
  int64_t row_cap = cand_blocks ? (int64_t)max_blocks * block : ld;
  if (row_cap > ld) row_cap = ld;
  const int64_t nblk = (ld + block - 1) / block;
  const size_t smem_b = (size_t)(nblk < kSmemKeys ? (nblk > 0 ? nblk : 1) : kSmemKeys) *
                        sizeof(uint32_t);
  // Each kernel's shared-memory attribute is its largest request (the most
  // keys it stages plus the most candidate blocks), the same value on every
  // call, so that concurrent callers never lower it under another's launch.
  auto launch = [&](auto kern, int nt, int64_t staged, int64_t staged_max) {
    const size_t smem = (size_t)(staged + (cand_blocks ? max_blocks : 0)) * sizeof(uint32_t);
    const size_t smem_max = (size_t)(staged_max + kMaxSortBlocks) * sizeof(uint32_t);
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max);
    kern<<<b.num_q, nt, smem, st>>>(b, scores, ld, k, cand_blocks, block, max_blocks, idx, count,
                                    d_err, staged);
  };
  if (!cand_blocks && row_cap > 4096 && row_cap <= 256 * 64) {
    topk_list_kernel<256><<<b.num_q, 256, 0, st>>>(b, scores, ld, k, idx, count, d_err);
  } else if (row_cap <= 256 * 4) launch(topk_kernel<256, 4>, 256, 0, 0);
  else if (row_cap <= 256 * 8) launch(topk_kernel<256, 8>, 256, 0, 0);
  else if (row_cap <= 256 * 16) launch(topk_kernel<256, 16>, 256, 0, 0);
  else if (row_cap <= 256 * 32) launch(topk_kernel<256, 32>, 256, 0, 0);
  else if (row_cap <= 256 * 64) launch(topk_kernel<256, 64>, 256, 0, 0);
  else
    launch(topk_kernel<kThreads, 32>, kThreads, row_cap < kSmemKeys ? row_cap : kSmemKeys,
           kSmemKeys);
  if (blocks_out) {
    cudaFuncSetAttribute(candidate_blocks_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)(kSmemKeys * sizeof(uint32_t)));
    candidate_blocks_kernel<<<b.num_q, kThreads, smem_b, st>>>(
        b, scores, ld, block, max_blocks, blocks_out, nblocks_out,
        nblk < kSmemKeys ? nblk : (int64_t)kSmemKeys);
  }
  return launch_status();
}

int stream_threshold_launch(const Batch &b, int64_t max_len, int k, int stride,
                            const StreamWs &ws, cudaStream_t st) {
  stream_threshold_kernel<<<(b.num_q + 7) / 8, 256, 0, st>>>(b, max_len, k, stride, ws);
  return launch_status();
}

int stream_select_launch(const Batch &b, int64_t max_len, int k, int n_heads,
                         const uint8_t *q_fp4, const float *q_scale, const float *head_w,
                         const uint8_t *k_fp4, const float *k_scale, const StreamWs &ws,
                         int32_t *idx, int32_t *count, cudaStream_t st) {
  stream_select_kernel<256><<<b.num_q, 256, 0, st>>>(b, max_len, k, ws, idx, count);
  // the fallback: one persistent CTA per SM takes queued rows until none is left
  const int grid = sm_count();
  auto fb = [&](auto kern, int hi) {
    const int smem = (hi * 128 + 2 * 2048) * 4;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    kern<<<grid, 256, smem, st>>>(b, max_len, k, q_fp4, q_scale, head_w, k_fp4, k_scale, ws,
                                  idx, count);
  };
  switch (n_heads) {
    case 8: fb(stream_fallback_kernel<8>, 8); break;
    case 16: fb(stream_fallback_kernel<16>, 16); break;
    case 32: fb(stream_fallback_kernel<32>, 32); break;
    case 64: fb(stream_fallback_kernel<64>, 64); break;
    default: return CSA2_ERR_UNSUPPORTED;
  }
  return launch_status();
}

}  // namespace csa2

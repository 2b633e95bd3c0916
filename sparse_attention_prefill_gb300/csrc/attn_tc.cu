// a8-a10 on the 5th-generation tensor cores: sparse + sliding-window attention
// under one softmax, FP8 block-32 rows dequantised to f16 in shared memory,
// tcgen05 MMAs accumulating in TMEM.
//
// What is computed (SGLang/Miles day-0 article sec. 1; "DeepSeek V4.1 Flash
// 建模" mixed-precision card: the 512-dim latent row is key and value; window
// lower bound: "SGLang 如何让 DeepSeek V4.1 Flash 的后半层只处理尾部 token" sec. 2.3):
//   rows(q) = selected compressed rows  u  window rows [lo, t]
//   O[q,h]  = softmax_i(sm_scale <Q[q,h], row_i>) . rows
//
// Formulation.  A query has H <= 64 heads (zero-padded to 64) and up to
// k + window rows of 512 channels, processed in chunks of 64 rows.  Both
// products are written transposed:
//   S^T[r, h] = sum_d R[r, d] Q[h, d]          (M = 64 rows,   N = 64, K = 512)
//   O^T[d, h] += sum_r R[r, d] P[r, h]         (M = 128 chans, N = 64, K = 64; 4 tiles)
// One f16 copy of the chunk (SW128 layout, 8 column blocks of 64 channels) is
// the K-major A operand of the first product and the MN-major A operand of
// the second.  Chunks are double-buffered in shared memory (R and P), S^T in
// TMEM (2 x 64 columns; an M = 64 accumulator fills lanes 0-15 of each 32-lane
// sub-partition) and O^T takes 4 x 64 TMEM columns.  S^T runs one chunk ahead
// of O^T (each has its own issuing warp), so gathering, softmax and both
// products of neighbouring chunks overlap.  The softmax keeps a lazily moved reference
// maximum per head: it moves (and O^T and the row sums are rescaled) only when
// a logit exceeds it by more than 2^8, so P <= 256 always fits f16.
//
// Roles (16 warps, one CTA per SM, persistent over queries):
//   warps 0-7   softmax + epilogue; warp w reads TMEM sub-partition w%4 and
//               heads 32*(w/4) .. +31 (rows of S^T, channels of O^T); S^T is
//               read 16 lanes wide (its M = 64 rows fill lanes 0-15 of each
//               sub-partition), so every thread holds two rows x 8 heads;
//               between a query's last chunk and its epilogue the eight warps
//               load the next query's Q (bf16 rows, prefetched into L2 a query
//               ahead), convert it to f16 and store it into the operand buffer
//               the query's last S^T MMAs have released, so the next query's
//               first products overlap this query's epilogue
//   warp 8      TMEM allocation; lane 0 issues the S^T MMAs
//   warp 9      lane 0 issues the O^T MMAs (the two products of neighbouring
//               chunks are issued independently, so neither waits behind the
//               other in one issuing thread); the whole warp builds the next
//               query's row list one query ahead, while it waits for P
//   warps 10-15 producers: row gather + E4M3 -> f16 dequant in steps of 32
//               rows, loads issued one step ahead; a chunk buffer is released
//               in 32-row halves
// The per-head row sums and maxima are reduced over the 8 threads holding a
// head's columns (three butterfly steps), then across the 4 warps of a head
// half through shared memory.
// Every wait is bounded (two seconds unless csa2_set_wait_limit_ns says
// otherwise); on expiry the kernel raises CSA2_DERR_TIMEOUT, drains its MMAs
// (for at most two seconds), frees TMEM and returns.
#include "common.cuh"
#include "kernels.cuh"
#include "tcgen05.cuh"

namespace csa2 {
namespace {

using namespace tc;

constexpr int kDim = 512;
constexpr int kChunk = 64;            // rows per chunk (S^T MMA M)
constexpr int kStepRows = 32;         // rows per producer step
constexpr int kHeadsPad = 64;
constexpr int kSoftmaxWarps = 8;
constexpr int kMmaWarp = 8;            // TMEM allocation; lane 0 issues S^T
constexpr int kOWarp = 9;              // lane 0 issues O^T
constexpr int kProducerWarp0 = 10;
constexpr int kProducerWarps = 6;
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kProducerThreads = kProducerWarps * 32;
constexpr int kMaxSel = 2048;

// shared-memory map (bytes)
constexpr uint32_t kRBlock = kChunk * 128;       // 8 KB: 64 rows x 64 channels f16
constexpr uint32_t kRBuf = 8 * kRBlock;          // 64 KB per chunk buffer
constexpr uint32_t kOffR = 0;                    // 2 chunk buffers (128 KB)
constexpr uint32_t kQBlock = kHeadsPad * 128;    // 8 KB
constexpr uint32_t kOffQ = 2 * kRBuf;            // 64 KB
constexpr uint32_t kPBuf = kChunk * 128;         // 8 KB: 64 rows x 64 heads f16
constexpr uint32_t kOffP = kOffQ + 8 * kQBlock;  // 2 x 8 KB
constexpr uint32_t kOffList = kOffP + 2 * kPBuf; // 2 x int32 [kMaxSel] (16 KB)
constexpr uint32_t kOffMisc = kOffList + 2 * kMaxSel * 4;
constexpr uint32_t kSmemBytes = kOffMisc + 2048;
static_assert(kSmemBytes <= 232448, "shared memory");

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;           // 2 x 64 (M = 64 layout)
constexpr uint32_t kColO = 128;         // 4 x 64

constexpr uint64_t kWaitNs = 2000000000ull;   // drains (the pipeline waits take Params::wait_ns)
constexpr int kDerrTimeout = 128;

struct Misc {
  uint64_t q_full, q_empty, o_full, o_empty, done, done_o, sm_grp;
  uint64_t r_full[2], r_empty[2][2], s_full[2], s_empty[2], p_full[2], p_empty[2];
  uint64_t meta_full[2];
  int64_t meta[2][4];   // per query (ring of 2): selected rows, window rows, first SWA
                        // row, pool row of the request's entry 0
  uint64_t wait_ns;     // bound on every pipeline wait
  uint32_t tmem_base;
  int abort;
  int votes[2][8];      // softmax warps: "a logit exceeded the reference", by chunk parity
  alignas(16) float m_ref[64];   // reference maximum per head (log2 units)
  float alpha[64];      // rescale factors of the current slow path
  float red[4][64];     // cross-warp reductions
};
static_assert(sizeof(Misc) <= 2048, "misc region");

// 2^x on the special-function unit (ex2.approx: relative error ~2^-22)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait; on expiry raise the abort flag and report false.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, Misc *ms) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (*(volatile int *)&ms->abort) return false;
    if (globaltimer() - t0 > ms->wait_ns) {
      atomicExch(&ms->abort, 1);
      return false;
    }
  }
  return true;
}

// Group barrier among the warps of one role, on an mbarrier whose arrival
// count is the role's warp count: bounded and abort-aware, unlike bar.sync.
__device__ __forceinline__ bool group_sync(uint64_t *bar, uint32_t &phase, Misc *ms) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
  const bool ok = wait_bar(bar, phase & 1, ms);
  ++phase;
  return ok;
}

struct Rows {
  int64_t nsel;        // valid selected rows
  int64_t win_first;   // SWA row of the first window row
  int64_t nwin;        // window rows
  int err;
};

// Rows of query q, computed cooperatively by one full warp (every lane gets
// the result).  When `list` is given, the valid selected entries are
// compacted into it in idx order.
__device__ Rows query_rows(const Batch &b, int q, const int32_t *__restrict__ idx, int k,
                           const int64_t *__restrict__ win_lo, int window, int *list) {
  const int lane = threadIdx.x & 31;
  const int r = b.q_req[q];
  const int64_t t = b.q_pos[q];
  const int64_t n_vis = n_visible(t, b.ratio);
  const int64_t kvn = b.kv_len[r];
  Rows o;
  o.err = 0;
  int64_t cnt = 0;
  for (int base = 0; base < k; base += 512) {
    int32_t jv[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = base + u * 32 + lane;
      jv[u] = i < k ? __ldg(idx + (int64_t)q * k + i) : -1;
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int64_t j = jv[u];
      const bool bad = j >= 0 && (j >= n_vis || j >= kvn);
      const bool ok = j >= 0 && !bad;
      if (__any_sync(0xffffffffu, bad)) o.err |= CSA2_DERR_RANGE_IDX;
      const uint32_t m = __ballot_sync(0xffffffffu, ok);
      if (list && ok) list[cnt + __popc(m & ((1u << lane) - 1u))] = (int)j;
      cnt += __popc(m);
    }
  }
  o.nsel = cnt;
  int64_t lo = t - window + 1;
  if (win_lo && win_lo[q] > lo) lo = win_lo[q];
  if (lo < 0) lo = 0;
  const int64_t p0 = b.swa_pos0[r], pn = b.swa_len[r];
  int64_t lo_v = lo > p0 ? lo : p0;
  int64_t hi_v = t < p0 + pn - 1 ? t : p0 + pn - 1;
  if (lo <= t && (lo < p0 || t > p0 + pn - 1)) o.err |= CSA2_DERR_RANGE_WINDOW;
  o.nwin = hi_v >= lo_v ? hi_v - lo_v + 1 : 0;
  o.win_first = b.swa_start[r] + (lo_v - p0);
  return o;
}

__device__ __forceinline__ int n_chunks_of(int64_t nrows) {
  const int64_t c = (nrows + kChunk - 1) / kChunk;
  return c > 0 ? (int)c : 1;
}

struct Params {
  Batch b;
  int n_heads;
  const __nv_bfloat16 *q;
  const uint8_t *kv_fp8;     // FP8 rows, or E2M1 pairs when kv_sf is set
  const float *kv_scale;
  const uint8_t *kv_sf;      // FP4 main KV: E4M3 scale per 16 channels
  const int32_t *idx;
  int k;
  const uint8_t *swa_fp8;
  const float *swa_scale;
  const int64_t *win_lo;
  int window;
  float scale_log2;
  const float *sink;
  __nv_bfloat16 *out;
  float *lse;
  int32_t *d_err;
  uint64_t wait_ns;
};

// ---------------------------------------------------------------------------
// producers
// ---------------------------------------------------------------------------
struct Item {
  uint4 codes;
  float scale;
};

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, __half2 s) {
  __half2 x = *reinterpret_cast<__half2 *>(&a);
  x = __hmul2(x, s);
  return *reinterpret_cast<uint32_t *>(&x);
}

// four E4M3 codes -> two f16x2 (low code pair -> lo); the halves are taken
// apart by a vector move, not by shifts
__device__ __forceinline__ void e4m3x4_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
  asm("{ .reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// One producer step: 32 rows x 512 channels, as 1024 items of 16 channels.
// Producer thread p handles segment p%32 (channels 16*(p%32) ..) of rows
// p/32 + 7i: the segment is the same for every item and step of a thread (a
// warp covers whole 512-byte rows), so the per-thread address parts are fixed
// once per query and only the row changes per item.
constexpr int kRowStride = kProducerThreads / 32;   // rows between a thread's items
constexpr int kItemsPerThread = (kStepRows + kRowStride - 1) / kRowStride;
static_assert(kProducerThreads % 32 == 0, "segment fixed per thread");

// Per-thread, per-query source bases (segment offset folded in).
struct Src {
  const uint8_t *sel_b;   // row kv0 of the pool
  const float *sel_s;     // (FP8 main KV)
  const uint8_t *sel_sf;  // (FP4 main KV)
  const uint8_t *win_b;   // first window row of the SWA buffer
  const float *win_s;
  const uint8_t *dummy_b; // a readable row for rows past the end (masked when stored)
  const float *dummy_s;
  int64_t nsel, nrows;
};

// FP4 main-KV rows: 16 channels = 8 bytes of E2M1 pairs and one E4M3 scale
// byte; the item holds them in codes.x/.y and codes.z.
__device__ __forceinline__ void load_fp4(const Src &S, int64_t j, Item &it) {
  const uint2 c = __ldg(reinterpret_cast<const uint2 *>(S.sel_b + j * (kDim / 2)));
  it.codes = make_uint4(c.x, c.y, (uint32_t)__ldg(S.sel_sf + j * (kDim / 16)), 0u);
}

template <bool kFp4>
__device__ __forceinline__ void load_step(const int *list, const Src &S, int row0, int step,
                                          Item (&it)[kItemsPerThread]) {
  const int64_t r0 = (int64_t)step * kStepRows;
  if (r0 + kStepRows <= S.nsel) {            // every row selected
#pragma unroll
    for (int i = 0; i < kItemsPerThread; ++i) {
      if (row0 + i * kRowStride < kStepRows) {
        const int64_t j = list[r0 + row0 + i * kRowStride];
        if (kFp4) {
          load_fp4(S, j, it[i]);
        } else {
          it[i].codes = __ldg(reinterpret_cast<const uint4 *>(S.sel_b + j * kDim));
          it[i].scale = __ldg(S.sel_s + j * (kDim / 32));
        }
      }
    }
  } else if (r0 >= S.nsel && r0 + kStepRows <= S.nrows) {   // every row in the window
#pragma unroll
    for (int i = 0; i < kItemsPerThread; ++i) {
      if (row0 + i * kRowStride < kStepRows) {
        const int64_t w = r0 + row0 + i * kRowStride - S.nsel;
        it[i].codes = __ldg(reinterpret_cast<const uint4 *>(S.win_b + w * kDim));
        it[i].scale = __ldg(S.win_s + w * (kDim / 32));
      }
    }
  } else {                                     // boundary or last step
#pragma unroll
    for (int i = 0; i < kItemsPerThread; ++i) {
      if (row0 + i * kRowStride < kStepRows) {
        const int64_t ri = r0 + row0 + i * kRowStride;
        const uint8_t *b;
        const float *sc;
        if (kFp4 && ri < S.nsel) {   // warp-uniform: a warp's items are one row
          load_fp4(S, list[ri], it[i]);
          continue;
        }
        if (ri < S.nsel) {
          const int64_t j = list[ri];
          b = S.sel_b + j * kDim;
          sc = S.sel_s + j * (kDim / 32);
        } else if (ri < S.nrows) {
          b = S.win_b + (ri - S.nsel) * kDim;
          sc = S.win_s + (ri - S.nsel) * (kDim / 32);
        } else {
          b = S.dummy_b;
          sc = S.dummy_s;
        }
        it[i].codes = __ldg(reinterpret_cast<const uint4 *>(b));
        it[i].scale = __ldg(sc);
      }
    }
  }
}

// Dequantise a step into rows 32*half .. +31 of the chunk buffer R.
// off[i][0..1]: byte offsets (half 0) of the two 16-byte stores of item i;
// half 1 is 32 rows (4096 bytes) further.  The 8 threads of a store phase
// cover 8 consecutive segments: segments 4-7 of each group sit in the next
// column block, whose 16-byte chunk positions repeat the first block's, so
// they store their upper half first and every phase touches 8 distinct
// positions.  Rows at or past `valid_rows` (step-relative) are written as zeros.
// kKind: 0 every row FP8, 1 every row FP4 (selected rows of the FP4 layout),
// 2 rows below fp4_rows FP4 and the rest FP8 (a step that crosses from the
// selected rows into the window)
template <bool kMasked, int kKind>
__device__ __forceinline__ void store_step(uint8_t *R, int half, bool swap, int row0,
                                           const uint32_t (&off)[kItemsPerThread][2],
                                           int64_t valid_rows, int64_t fp4_rows,
                                           const Item (&it)[kItemsPerThread]) {
  uint8_t *Rb = R + half * (kStepRows / 8) * 1024;
#pragma unroll
  for (int i = 0; i < kItemsPerThread; ++i) {
    if (row0 + i * kRowStride < kStepRows) {
      uint4 cd = it[i].codes;
      float sc = it[i].scale;
      if (kMasked && row0 + i * kRowStride >= valid_rows) {
        cd = make_uint4(0, 0, 0, 0);
        sc = 0.f;
      }
      uint32_t h[8];
      __half2 s2;
      if (kKind == 1 || (kKind == 2 && row0 + i * kRowStride < fp4_rows)) {
        // E2M1 x E4M3 scale is exact in f16 (at most 5 significant bits,
        // magnitudes in [2^-10, 2688])
        uint32_t sl, sh;
        e4m3x4_f16x4(cd.z | (cd.z << 8), sl, sh);
        s2 = *reinterpret_cast<const __half2 *>(&sl);
        uint32_t lo[4], hi[4];
        e2m1x8_f16x8(swap ? cd.y : cd.x, lo);
        e2m1x8_f16x8(swap ? cd.x : cd.y, hi);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          h[j] = lo[j];
          h[4 + j] = hi[j];
        }
      } else {
        s2 = __float2half2_rn(sc);
        const uint32_t a = swap ? cd.z : cd.x, b = swap ? cd.w : cd.y;
        const uint32_t c = swap ? cd.x : cd.z, d = swap ? cd.y : cd.w;
        e4m3x4_f16x4(a, h[0], h[1]);
        e4m3x4_f16x4(b, h[2], h[3]);
        e4m3x4_f16x4(c, h[4], h[5]);
        e4m3x4_f16x4(d, h[6], h[7]);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) h[j] = hmul2_u32(h[j], s2);
      *reinterpret_cast<uint4 *>(Rb + off[i][0]) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4 *>(Rb + off[i][1]) = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
}

template <bool kFp4>
__device__ void producer_role(const Params &P, uint8_t *smem, Misc *ms) {
  const int ptid = threadIdx.x - kProducerWarp0 * 32;
  const int lane = threadIdx.x & 31;
  const int row0 = ptid >> 5, seg = lane;
  const bool swap = (seg & 4) != 0;
  uint32_t off[kItemsPerThread][2];   // R byte offsets of this thread's stores (half 0)
#pragma unroll
  for (int i = 0; i < kItemsPerThread; ++i) {
    const uint32_t row = (uint32_t)(row0 + i * kRowStride) & (kStepRows - 1);
    const uint32_t lo = sw128_offset(row, seg * 16, kRBlock);
    const uint32_t hi = sw128_offset(row, seg * 16 + 8, kRBlock);
    off[i][0] = swap ? hi : lo;
    off[i][1] = swap ? lo : hi;
  }
  const int *lists = reinterpret_cast<const int *>(smem + kOffList);
  uint32_t g = 0;  // chunks produced by this CTA
  uint32_t qi = 0;
  for (int q = blockIdx.x; q < P.b.num_q; q += gridDim.x, ++qi) {
    // ---- row list and counts of this query (built one query ahead by the
    // O^T issuer's warp)
    const uint32_t ms_slot = qi & 1;
    if (!wait_bar(&ms->meta_full[ms_slot], (qi >> 1) & 1, ms)) break;
    const int *list = lists + ms_slot * kMaxSel;
    Src S;
    S.nsel = ms->meta[ms_slot][0];
    S.nrows = S.nsel + ms->meta[ms_slot][1];
    const int64_t win_first = ms->meta[ms_slot][2];
    const int64_t kv0 = ms->meta[ms_slot][3];
    if (kFp4) {
      S.sel_b = P.kv_fp8 + kv0 * (kDim / 2) + seg * 8;
      S.sel_sf = P.kv_sf + kv0 * (kDim / 16) + seg;
      S.sel_s = nullptr;
    } else {
      S.sel_b = P.kv_fp8 + kv0 * kDim + seg * 16;
      S.sel_s = P.kv_scale + kv0 * (kDim / 32) + seg / 2;
      S.sel_sf = nullptr;
    }
    S.win_b = P.swa_fp8 + win_first * kDim + seg * 16;
    S.win_s = P.swa_scale + win_first * (kDim / 32) + seg / 2;
    S.dummy_b = P.swa_fp8 + seg * 16;
    S.dummy_s = P.swa_scale + seg / 2;
    const int nch = n_chunks_of(S.nrows);
    // ---- chunks: 2 steps of 32 rows each; the loads of the next step are
    // in flight while a step waits for its buffer and is stored
    const int nsteps = nch * 2;
    Item b0[kItemsPerThread], b1[kItemsPerThread];
    load_step<kFp4>(list, S, row0, 0, b0);
    bool ok = true;
    // one step: prefetch step st+1 into `pre`, then store step st from `use`
    auto step = [&](int st, Item(&use)[kItemsPerThread], Item(&pre)[kItemsPerThread]) -> bool {
      const uint32_t gc = g + (uint32_t)(st >> 1), buf = gc & 1;
      if (st + 1 < nsteps) load_step<kFp4>(list, S, row0, st + 1, pre);
      if (!wait_bar(&ms->r_empty[buf][st & 1], ((gc >> 1) & 1) ^ 1, ms)) return false;
      uint8_t *R = smem + kOffR + buf * kRBuf;
      const int64_t valid_rows = S.nrows - (int64_t)st * kStepRows;
      const int64_t fp4_rows = S.nsel - (int64_t)st * kStepRows;
      if (!kFp4 || fp4_rows <= 0) {             // FP8 rows only
        if (valid_rows >= kStepRows)
          store_step<false, 0>(R, st & 1, swap, row0, off, valid_rows, fp4_rows, use);
        else
          store_step<true, 0>(R, st & 1, swap, row0, off, valid_rows, fp4_rows, use);
      } else if (fp4_rows >= kStepRows) {      // FP4 rows only (valid_rows >= fp4_rows)
        store_step<false, 1>(R, st & 1, swap, row0, off, valid_rows, fp4_rows, use);
      } else {
        store_step<true, 2>(R, st & 1, swap, row0, off, valid_rows, fp4_rows, use);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms->r_full[buf]);
      return true;
    };
    // one copy of the step body: the prefetched items move into place at the
    // end of a step (their loads have had the whole store to land)
#pragma unroll 1
    for (int st = 0; st < nsteps && ok; ++st) {
      ok = step(st, b0, b1);
#pragma unroll
      for (int i = 0; i < kItemsPerThread; ++i) b0[i] = b1[i];
    }
    g += nch;
    if (!ok) break;
  }
}

// ---------------------------------------------------------------------------
// MMA issuer: lane 0 of the warp.  S^T of chunk g is issued before O^T of
// chunk g-1 (S^T runs one chunk ahead); at a query boundary the pending O^T is
// issued first so the epilogue of the finished query is not held back.
// ---------------------------------------------------------------------------
// Operand descriptors: bases (low, high words); every MMA's descriptor is
// one of these plus a compile-time offset in the low word.
struct Descs {
  uint32_t rk_lo, rk_hi, q_lo, q_hi, rm_lo, rm_hi, p_lo, p_hi;
};

__device__ __forceinline__ Descs make_descs(uint8_t *smem) {
  const uint32_t r0 = smem_u32(smem + kOffR), q0 = smem_u32(smem + kOffQ),
                 p0 = smem_u32(smem + kOffP);
  const uint64_t d_rk = make_desc_sw128(r0, 16, 1024);        // R, K-major (S)
  const uint64_t d_q = make_desc_sw128(q0, 16, 1024);         // Q, K-major (S)
  const uint64_t d_rm = make_desc_sw128(r0, kRBlock, 1024);   // R^T, MN-major (O)
  const uint64_t d_p = make_desc_sw128(p0, kRBlock, 1024);    // P^T, MN-major (O)
  return Descs{(uint32_t)d_rk, (uint32_t)(d_rk >> 32), (uint32_t)d_q, (uint32_t)(d_q >> 32),
               (uint32_t)d_rm, (uint32_t)(d_rm >> 32), (uint32_t)d_p, (uint32_t)(d_p >> 32)};
}

// bounded wait for every MMA this thread issued (TMEM is never freed under a
// running MMA)
__device__ __forceinline__ void drain(uint64_t *bar) {
  mma_commit(bar);
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, 0) && globaltimer() - t0 < kWaitNs) {
  }
}

// S^T issuer (lane 0 of warp kMmaWarp): S^T(g) = R(g) . Q^T into S buffer g&1
// as soon as chunk g is produced and the buffer is free.
__device__ void s_issuer_role(const Params &P, uint8_t *smem, Misc *ms) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    const uint32_t tmem = ms->tmem_base;
    const uint32_t id_s = make_idesc_f16(kChunk, kHeadsPad, false, false);
    const Descs D = make_descs(smem);
    bool ok = true;
    uint32_t g = 0, qi = 0;
    for (int q = blockIdx.x; q < P.b.num_q && ok; q += gridDim.x, ++qi) {
      const uint32_t slot = qi & 1;
      if (!(ok = wait_bar(&ms->meta_full[slot], (qi >> 1) & 1, ms))) break;
      const int nch = n_chunks_of(ms->meta[slot][0] + ms->meta[slot][1]);
      for (int c = 0; c < nch && ok; ++c, ++g) {
        const uint32_t sb = g & 1, ph = (g >> 1) & 1;
        ok = wait_bar(&ms->s_empty[sb], ph ^ 1, ms);
        if (ok && c == 0) ok = wait_bar(&ms->q_full, qi & 1, ms);
        if (ok) ok = wait_bar(&ms->r_full[sb], ph, ms);
        if (!ok) break;
        fence_after_sync();
        const uint32_t ra = D.rk_lo + ((sb * kRBuf) >> 4);
#pragma unroll
        for (int kk = 0; kk < 32; ++kk) {
          const int blk = kk >> 2;
          mma_f16_split(tmem + kColS + sb * 64, ra + ((blk * kRBlock + (kk & 3) * 32) >> 4),
                        D.rk_hi, D.q_lo + ((blk * kQBlock + (kk & 3) * 32) >> 4), D.q_hi, id_s,
                        kk > 0 ? 1u : 0u);
        }
        mma_commit(&ms->s_full[sb]);
        if (c == nch - 1) mma_commit(&ms->q_empty);
      }
    }
    drain(&ms->done);
  }
  __syncwarp();
}

// Row list and counts of query qn into slot qin & 1, by one whole warp
// (query_rows), then meta_full[slot] is arrived on.  The O^T issuer's warp
// builds them one query ahead of their use: at the start of its query qi it
// publishes query qi + 1 into slot (qi + 1) & 1, which was last read for
// query qi - 1 (by the producers while gathering its rows, all stored before
// its last O^T could be issued, and by every role at that query's start).
__device__ void publish_rows(const Params &P, uint8_t *smem, Misc *ms, int qn, uint32_t qin,
                             int &err) {
  if (qn >= P.b.num_q) return;
  const int lane = threadIdx.x & 31;
  int *lists = reinterpret_cast<int *>(smem + kOffList);
  const uint32_t slot = qin & 1;
  const Rows r1 = query_rows(P.b, qn, P.idx, P.k, P.win_lo, P.window, lists + slot * kMaxSel);
  err |= r1.err;
  const int64_t kv0 = P.b.kv_start[P.b.q_req[qn]];
  __syncwarp();
  if (lane == 0) {
    ms->meta[slot][0] = r1.nsel;
    ms->meta[slot][1] = r1.nwin;
    ms->meta[slot][2] = r1.win_first;
    ms->meta[slot][3] = kv0;
    mbar_arrive(&ms->meta_full[slot]);
  }
}

// O^T issuer (warp kOWarp, lane 0 issues): O^T += R(g)^T . P(g)^T as soon as P(g) is
// written.  S^T(g) has completed by then (the softmax read it), so this
// issuer's commits release R(g), half by half, for both products.
__device__ void o_issuer_role(const Params &P, uint8_t *smem, Misc *ms) {
  const int lane = threadIdx.x & 31;
  int err = 0;
  publish_rows(P, smem, ms, blockIdx.x, 0, err);
  const uint32_t tmem = ms->tmem_base;
  const uint32_t id_o = make_idesc_f16(128, kHeadsPad, true, true);
  const Descs D = make_descs(smem);
  bool ok = true;
  uint32_t g = 0, qi = 0;
  // every lane waits (each acquires what it then reads); the outcome is made
  // warp-uniform so that the whole warp leaves together on an abort
  auto wait_all = [&](uint64_t *bar, uint32_t parity) {
    const bool r = wait_bar(bar, parity, ms);
    return __all_sync(0xffffffffu, r);
  };
  for (int q = blockIdx.x; q < P.b.num_q && ok; q += gridDim.x, ++qi) {
    publish_rows(P, smem, ms, q + gridDim.x, qi + 1, err);
    const uint32_t slot = qi & 1;
    if (!(ok = wait_all(&ms->meta_full[slot], (qi >> 1) & 1))) break;
    const int nch = n_chunks_of(ms->meta[slot][0] + ms->meta[slot][1]);
    for (int c = 0; c < nch && ok; ++c, ++g) {
      const uint32_t buf = g & 1, ph = (g >> 1) & 1;
      ok = wait_all(&ms->p_full[buf], ph);
      if (ok && c == 0) ok = wait_all(&ms->o_empty, (qi & 1) ^ 1);
      if (!ok) break;
      if (lane == 0) {
        fence_after_sync();
        const uint32_t ra = D.rm_lo + ((buf * kRBuf) >> 4), pa = D.p_lo + ((buf * kPBuf) >> 4);
        // rows 0-31 of the chunk first, so the producers can refill that
        // half while the second half is still being read
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
#pragma unroll
            for (int ks = 2 * half; ks < 2 * half + 2; ++ks) {
              mma_f16_split(tmem + kColO + t * 64, ra + ((t * 2 * kRBlock + ks * 2048) >> 4),
                            D.rm_hi, pa + ((ks * 2048) >> 4), D.p_hi, id_o,
                            (c > 0 || ks > 0) ? 1u : 0u);
            }
          }
          mma_commit(&ms->r_empty[buf][half]);
        }
        mma_commit(&ms->p_empty[buf]);
        if (c == nch - 1) mma_commit(&ms->o_full);
      }
      __syncwarp();
    }
  }
  if (lane == 0) drain(&ms->done_o);
  __syncwarp();
  err = __reduce_or_sync(0xffffffffu, err);
  if (lane == 0) raise_err(P.d_err, err);
}

// ---------------------------------------------------------------------------
// softmax + epilogue (warps 0-7)
// ---------------------------------------------------------------------------
__device__ void softmax_role(const Params &P, uint8_t *smem, Misc *ms) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sp = warp & 3;          // TMEM sub-partition: lanes 32*sp ..
  const int hh = warp >> 2;         // head half: heads 32*hh ..
  const int stid = threadIdx.x;     // 0..255
  const uint32_t tmem = ms->tmem_base;
  const uint32_t lane_addr = (uint32_t)(32 * sp) << 16;
  const float NEG_INF = -INFINITY;
  float lsum[8];   // this thread's heads 32hh + 8k + hc + e, as [2k + e]
  uint32_t g = 0, qi = 0, gp = 0;
  bool ok = true;
  // Q of query qn into the f16 operand buffer: bf16 rows read 16 bytes at a
  // time (from L2: the copy was prefetched a query ahead), converted, and
  // stored at their SW128 positions; heads past n_heads stay zero (written
  // once below).  Then the S^T issuer may start the query.
  uint8_t *Qs = smem + kOffQ;
  auto load_q = [&](int qn) {
    const uint4 *src = reinterpret_cast<const uint4 *>(P.q + (int64_t)qn * P.n_heads * kDim);
    const int q_chunks = P.n_heads * (kDim / 8);
    constexpr int kQBatch = 8;
    for (int base = stid; base < q_chunks; base += kQBatch * kSoftmaxWarps * 32) {
      uint4 raw[kQBatch];
#pragma unroll
      for (int k = 0; k < kQBatch; ++k) {
        const int it = base + k * kSoftmaxWarps * 32;
        if (it < q_chunks) raw[k] = __ldg(src + it);
      }
#pragma unroll
      for (int k = 0; k < kQBatch; ++k) {
        const int it = base + k * kSoftmaxWarps * 32;
        if (it >= q_chunks) break;
        const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xffff0000u);
          __half2 h2 = __floats2half2_rn(lo, hi);
          o[j] = *reinterpret_cast<uint32_t *>(&h2);
        }
        const int h = it / (kDim / 8), d = (it % (kDim / 8)) * 8;
        *reinterpret_cast<uint4 *>(Qs + sw128_offset(h, d, kQBlock)) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ms->q_full);
  };
  auto prefetch_q = [&](int qn) {
    if (stid == 0 && qn < P.b.num_q)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                       P.q + (int64_t)qn * P.n_heads * kDim),
                   "r"((uint32_t)(P.n_heads * kDim * 2))
                   : "memory");
  };
  if (stid < 64) ms->m_ref[stid] = NEG_INF;
  for (int it = P.n_heads * (kDim / 8) + stid; it < kHeadsPad * (kDim / 8);
       it += kSoftmaxWarps * 32) {
    const int h = it / (kDim / 8), d = (it % (kDim / 8)) * 8;
    *reinterpret_cast<uint4 *>(Qs + sw128_offset(h, d, kQBlock)) = make_uint4(0, 0, 0, 0);
  }
  if (blockIdx.x < P.b.num_q) load_q(blockIdx.x);
  ok = group_sync(&ms->sm_grp, gp, ms);
  for (int q = blockIdx.x; q < P.b.num_q && ok; q += gridDim.x, ++qi) {
    const uint32_t slot = qi & 1;
    if (!(ok = wait_bar(&ms->meta_full[slot], (qi >> 1) & 1, ms))) break;
    const int64_t nrows = ms->meta[slot][0] + ms->meta[slot][1];
    const int nch = n_chunks_of(nrows);
    prefetch_q(q + gridDim.x);
#pragma unroll
    for (int j = 0; j < 8; ++j) lsum[j] = 0.f;
    for (int c = 0; c < nch; ++c, ++g) {
      const uint32_t sb = g & 1, ph = (g >> 1) & 1;
      ok = wait_bar(&ms->s_full[sb], ph, ms);
      if (!ok) break;
      fence_after_sync();
      uint32_t v[16];
      tmem_ld16x256b_x4(tmem + lane_addr + kColS + sb * 64 + 32 * hh, v);
      tmem_wait_ld();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms->s_empty[sb]);
      // M = 64 layout, read 16 lanes wide: this thread holds chunk rows crow
      // and crow + 8 (lanes t/4 and t/4 + 8 of the sub-partition) and the
      // column pairs 8k + hc, +1 (k < 4) of the warp's 32 heads:
      // v[4k + 2r + e] = row crow + 8r, head 32hh + 8k + hc + e
      const int crow = 16 * sp + (lane >> 2);
      const int hc = 2 * (lane & 3);
      const bool valid0 = (int64_t)c * kChunk + crow < nrows;
      const bool valid1 = (int64_t)c * kChunk + crow + 8 < nrows;
      float x[16], mr[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 m2 = c == 0 ? make_float2(NEG_INF, NEG_INF)
                                 : *reinterpret_cast<const float2 *>(&ms->m_ref[32 * hh + 8 * k + hc]);
        mr[2 * k] = m2.x;
        mr[2 * k + 1] = m2.y;
      }
      bool exceed = false;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const bool vr = (i & 2) ? valid1 : valid0;
        x[i] = vr ? __uint_as_float(v[i]) * P.scale_log2 : NEG_INF;
        exceed |= x[i] > mr[2 * (i >> 2) + (i & 1)] + 8.f;
      }
      // does any logit of the chunk exceed its head's reference by 2^8?
      const int vb = g & 1;
      const bool vote = __any_sync(0xffffffffu, exceed);
      if (lane == 0) ms->votes[vb][warp] = vote ? 1 : 0;
      if (!(ok = group_sync(&ms->sm_grp, gp, ms))) break;
      // the first chunk of a query always sets the reference (from an empty
      // one: -inf when no row of the chunk is valid)
      bool slow = c == 0;
#pragma unroll
      for (int w = 0; w < kSoftmaxWarps; ++w) slow |= ms->votes[vb][w] != 0;
      if (slow) {
        // per-head maximum: over this thread's two rows, then over the 8
        // threads holding the same columns, then across the 4 warps of this
        // head half
        float hm[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          hm[2 * k] = fmaxf(x[4 * k], x[4 * k + 2]);
          hm[2 * k + 1] = fmaxf(x[4 * k + 1], x[4 * k + 3]);
        }
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) {
#pragma unroll
          for (int j = 0; j < 8; ++j) hm[j] = fmaxf(hm[j], __shfl_xor_sync(0xffffffffu, hm[j], o));
        }
        if (lane < 4) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            ms->red[sp][32 * hh + 8 * k + hc] = hm[2 * k];
            ms->red[sp][32 * hh + 8 * k + hc + 1] = hm[2 * k + 1];
          }
        }
        if (!(ok = group_sync(&ms->sm_grp, gp, ms))) break;
        if (stid < 64) {
          const float old = c == 0 ? NEG_INF : ms->m_ref[stid];
          float mx = fmaxf(fmaxf(ms->red[0][stid], ms->red[1][stid]),
                           fmaxf(ms->red[2][stid], ms->red[3][stid]));
          mx = fmaxf(mx, old);
          ms->alpha[stid] = (old == NEG_INF) ? 0.f : exp2f(old - mx);
          ms->m_ref[stid] = mx;
        }
        if (!(ok = group_sync(&ms->sm_grp, gp, ms))) break;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          lsum[2 * k] *= ms->alpha[32 * hh + 8 * k + hc];
          lsum[2 * k + 1] *= ms->alpha[32 * hh + 8 * k + hc + 1];
          mr[2 * k] = ms->m_ref[32 * hh + 8 * k + hc];
          mr[2 * k + 1] = ms->m_ref[32 * hh + 8 * k + hc + 1];
        }
        if (c > 0) {
          // every earlier O^T MMA of this query must be complete: the latest
          // one issued is O^T(g-1)
          const uint32_t pb = (g - 1) & 1;
          if (!(ok = wait_bar(&ms->p_empty[pb], ((g - 1) >> 1) & 1, ms))) break;
          fence_after_sync();
#pragma unroll 1
          for (int t = 0; t < 8; ++t) {   // 4 tiles x 2 halves of this warp's 32 heads
            uint32_t o[32];
            const int hb = 32 * hh + 16 * (t & 1);
            const uint32_t a = tmem + lane_addr + kColO + (t >> 1) * 64 + 16 * (t & 1) + 32 * hh;
            tmem_ld32x32b_x16(a, o);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j)
              o[j] = __float_as_uint(__uint_as_float(o[j]) * ms->alpha[hb + j]);
            tmem_st32x32b_x16(a, o);
          }
          tmem_wait_st();
        }
      }
      // P(g) goes to buffer g&1 once O^T(g-2) has consumed it
      ok = wait_bar(&ms->p_empty[sb], ph ^ 1, ms);
      if (!ok) break;
      uint8_t *Pb = smem + kOffP + sb * kPBuf;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float m0 = mr[2 * k] == NEG_INF ? 0.f : mr[2 * k];
        const float m1 = mr[2 * k + 1] == NEG_INF ? 0.f : mr[2 * k + 1];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float p0 = ex2(x[4 * k + 2 * r] - m0);
          const float p1 = ex2(x[4 * k + 2 * r + 1] - m1);
          lsum[2 * k] += p0;
          lsum[2 * k + 1] += p1;
          __half2 h2 = __floats2half2_rn(p0, p1);
          *reinterpret_cast<uint32_t *>(Pb + sw128_offset(crow + 8 * r, 32 * hh + 8 * k + hc, 0)) =
              *reinterpret_cast<uint32_t *>(&h2);
        }
      }
      fence_proxy_async_smem();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms->p_full[sb]);
    }
    if (!ok) break;
    // ---- the next query's Q, as soon as this query's last S^T has read the
    // buffer (before this query's epilogue, so that the next query's first
    // products overlap it)
    if (q + (int)gridDim.x < P.b.num_q) {
      if (!(ok = wait_bar(&ms->q_empty, qi & 1, ms))) break;
      load_q(q + gridDim.x);
    }
    // ---- epilogue: row sums, normalisation, bf16 output, lse
    // per head: over the 8 threads holding its columns, then across the warps
    {
      const int hc = 2 * (lane & 3);
#pragma unroll
      for (int o = 4; o <= 16; o <<= 1) {
#pragma unroll
        for (int j = 0; j < 8; ++j) lsum[j] += __shfl_xor_sync(0xffffffffu, lsum[j], o);
      }
      if (lane < 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ms->red[sp][32 * hh + 8 * k + hc] = lsum[2 * k];
          ms->red[sp][32 * hh + 8 * k + hc + 1] = lsum[2 * k + 1];
        }
      }
    }
    if (!(ok = group_sync(&ms->sm_grp, gp, ms))) break;
    {
      // every warp derives the normalisers of its own head half (lane j:
      // head 32hh + j; the four warps of a half write the same values), so
      // no second barrier is needed before the output; the next query's
      // first chunk starts from an empty reference instead of a reset one
      const int h = 32 * hh + lane;
      float l = (ms->red[0][h] + ms->red[1][h]) + (ms->red[2][h] + ms->red[3][h]);
      const float m = ms->m_ref[h];
      const float mu = m == NEG_INF ? 0.f : m;
      if (P.sink && h < P.n_heads) l += exp2f(P.sink[h] * 1.4426950408889634f - mu);
      ms->alpha[h] = l > 0.f ? 1.f / l : 0.f;
      if (sp == 0 && P.lse && h < P.n_heads)
        P.lse[(int64_t)q * P.n_heads + h] =
            l > 0.f ? (mu + log2f(l)) * 0.6931471805599453f : NEG_INF;
      __syncwarp();
    }
    ok = wait_bar(&ms->o_full, qi & 1, ms);
    if (!ok) break;
    fence_after_sync();
    __nv_bfloat16 *og = P.out + (int64_t)q * P.n_heads * kDim;
    for (int t = 0; t < 4; ++t) {
      uint32_t o[32];
      tmem_ld32x32b_x32(tmem + lane_addr + kColO + t * 64 + 32 * hh, o);
      tmem_wait_ld();
      const int d = t * 128 + 32 * sp + lane;
      // two heads per conversion (one cvt.rn.bf16x2.f32), stored apart
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const int h = 32 * hh + j;
        const float2 a2 = *reinterpret_cast<const float2 *>(&ms->alpha[h]);
        const __nv_bfloat162 b2 =
            __floats2bfloat162_rn(__uint_as_float(o[j]) * a2.x, __uint_as_float(o[j + 1]) * a2.y);
        if (h < P.n_heads) og[(int64_t)h * kDim + d] = b2.x;
        if (h + 1 < P.n_heads) og[(int64_t)(h + 1) * kDim + d] = b2.y;
      }
    }
    fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ms->o_empty);
  }
}

template <bool kFp4>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(Params P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Misc *ms = reinterpret_cast<Misc *>(smem + kOffMisc);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&ms->q_full, kSoftmaxWarps);
    mbar_init(&ms->q_empty, 1);
    mbar_init(&ms->o_full, 1);
    mbar_init(&ms->o_empty, kSoftmaxWarps);
    mbar_init(&ms->done, 1);
    mbar_init(&ms->done_o, 1);
    mbar_init(&ms->sm_grp, kSoftmaxWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->r_full[i], 2 * kProducerWarps);   // two steps per chunk
      mbar_init(&ms->r_empty[i][0], 1);
      mbar_init(&ms->r_empty[i][1], 1);
      mbar_init(&ms->s_full[i], 1);
      mbar_init(&ms->s_empty[i], kSoftmaxWarps);
      mbar_init(&ms->p_full[i], kSoftmaxWarps);
      mbar_init(&ms->p_empty[i], 1);
      mbar_init(&ms->meta_full[i], 1);
    }
    ms->abort = 0;
    ms->wait_ns = P.wait_ns;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&ms->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp < kSoftmaxWarps) {
    softmax_role(P, smem, ms);
  } else if (warp == kMmaWarp) {
    s_issuer_role(P, smem, ms);
  } else if (warp == kOWarp) {
    o_issuer_role(P, smem, ms);
  } else {
    producer_role<kFp4>(P, smem, ms);
  }
  fence_before_sync();
  __syncthreads();
  if (ms->abort && threadIdx.x == 0) raise_err(P.d_err, kDerrTimeout);
  if (warp == kMmaWarp) {
    fence_after_sync();
    tmem_dealloc(ms->tmem_base, kTmemCols);
  }
}

}  // namespace

int attn_tc(const Batch &b, int n_heads, const __nv_bfloat16 *q, const uint8_t *kv_codes,
            const float *kv_scale, const uint8_t *kv_sf, const int32_t *idx, int k,
            const uint8_t *swa_fp8,
            const float *swa_scale, const int64_t *win_lo, int window, float sm_scale,
            const float *sink, __nv_bfloat16 *out, float *lse, int32_t *d_err,
            cudaStream_t st) {
  if (b.num_q == 0) return CSA2_OK;
  if (n_heads > kHeadsPad || k > kMaxSel) return CSA2_ERR_UNSUPPORTED;
  // 16-byte vector loads and asynchronous copies need 16-byte aligned rows
  // (FP4 main-KV rows are read 8 bytes at a time)
  if (((uintptr_t)q | (uintptr_t)swa_fp8) & 15u) return CSA2_ERR_UNSUPPORTED;
  if ((uintptr_t)kv_codes & (kv_sf ? 7u : 15u)) return CSA2_ERR_UNSUPPORTED;
  Params P;
  P.b = b;
  P.n_heads = n_heads;
  P.q = q;
  P.kv_fp8 = kv_codes;
  P.kv_scale = kv_scale;
  P.kv_sf = kv_sf;
  P.idx = idx;
  P.k = idx ? k : 0;
  P.swa_fp8 = swa_fp8;
  P.swa_scale = swa_scale;
  P.win_lo = win_lo;
  P.window = window;
  P.scale_log2 = sm_scale * 1.4426950408889634f;
  P.sink = sink;
  P.out = out;
  P.lse = lse;
  P.d_err = d_err;
  P.wait_ns = wait_limit_ns();
  const int grid = b.num_q < sm_count() ? b.num_q : sm_count();
  if (kv_sf) {
    cudaFuncSetAttribute(attn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)kSmemBytes);
    attn_tc_kernel<true><<<grid, kThreads, kSmemBytes, st>>>(P);
  } else {
    cudaFuncSetAttribute(attn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)kSmemBytes);
    attn_tc_kernel<false><<<grid, kThreads, kSmemBytes, st>>>(P);
  }
  return launch_status();
}

}  // namespace csa2

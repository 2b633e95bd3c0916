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
// k + window rows of 512 channels.  Rows are processed in chunks of 128 and
// every product is written transposed so that the MMA M dimension is 128:
//   S^T[r, h] = sum_d R[r, d] Q[h, d]          (M = 128 rows,  N = 64, K = 512)
//   O^T[d, h] += sum_r R[r, d] P[r, h]         (M = 128 chans, N = 64, K = 128; 4 tiles)
// One f16 copy of the chunk R (SW128 layout, 8 column blocks of 64 channels)
// is the K-major A operand of the first product and the MN-major A operand of
// the second.  S^T is double-buffered in TMEM (2 x 64 columns), O^T occupies
// 4 x 64 columns.  The softmax runs online with a lazily updated reference
// maximum per head: it is only moved (and O^T and the row sums rescaled) when
// a logit exceeds it by more than 2^8, so P <= 256 always fits f16.
//
// Roles (16 warps, one CTA per SM, persistent over queries):
//   warps 0-7   softmax + epilogue; warp w owns TMEM lanes 32*(w%4).. (rows of
//               S^T / channels of O^T) and heads 32*(w/4) .. +31
//   warp 8      TMEM allocation; lane 0 issues every MMA and commit
//   warps 9-15  producers: Q (bf16 -> f16), row gather + E4M3 -> f16 dequant,
//               in 4 pipeline steps of 128 channels per chunk
// Every wait is bounded (about two seconds); on expiry the kernel raises
// CSA2_DERR_TIMEOUT, drains and returns.
#include "common.cuh"
#include "kernels.cuh"
#include "tcgen05.cuh"

namespace csa2 {
namespace {

using namespace tc;

constexpr int kDim = 512;
constexpr int kRowsPerChunk = 128;
constexpr int kHeadsPad = 64;
constexpr int kSoftmaxWarps = 8;
constexpr int kMmaWarp = 8;
constexpr int kProducerWarp0 = 9;
constexpr int kProducerWarps = 7;
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kProducerThreads = kProducerWarps * 32;
constexpr int kMaxSel = 2048;

// shared-memory map (bytes)
constexpr uint32_t kOffR = 0;           // 8 blocks x [128 rows x 128 B]  (128 KB)
constexpr uint32_t kRBlock = 16384;
constexpr uint32_t kOffQ = 131072;      // 8 blocks x [64 heads x 128 B]  (64 KB)
constexpr uint32_t kQBlock = 8192;
constexpr uint32_t kOffP = 196608;      // [128 rows x 64 heads] f16       (16 KB)
constexpr uint32_t kOffList = 212992;   // 2 x int32 [kMaxSel]             (16 KB)
constexpr uint32_t kOffMisc = 229376;
constexpr uint32_t kSmemBytes = kOffMisc + 2048;
static_assert(kSmemBytes <= 232448, "shared memory");

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;           // 2 x 64
constexpr uint32_t kColO = 128;         // 4 x 64

constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kDerrTimeout = 128;

struct Misc {
  uint64_t q_full, q_empty, s_full[2], s_empty[2], p_full, p_empty, o_full, o_empty, done;
  uint64_t r_full[4], r_empty[4];
  uint64_t sm_grp;          // group sync of the softmax warps
  uint64_t meta_full[2];
  int64_t meta[2][4];       // per query (ring of 2): selected rows, window rows, first SWA
                            // row, pool row of the request's entry 0
  uint32_t tmem_base;
  int abort;
  int votes[2][8];      // softmax warps: "a logit exceeded the reference", by chunk parity
  float m_ref[64];      // reference maximum per head (log2 units)
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
    if (globaltimer() - t0 > kWaitNs) {
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
  const int64_t c = (nrows + kRowsPerChunk - 1) / kRowsPerChunk;
  return c > 0 ? (int)c : 1;
}

struct Params {
  Batch b;
  int n_heads;
  const __nv_bfloat16 *q;
  const uint8_t *kv_fp8;
  const float *kv_scale;
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

// One pipeline step: channels [128*pair, 128*pair+128) of the 128 rows of a
// chunk, as 1024 items of 16 channels.  Item ptid + 28*8*i of a producer
// thread is segment ptid%8 (16 channels) of row ptid/8 + 28i: the segment is
// the same for every item and step of a thread, so the per-thread address
// parts are fixed once per query and only the row changes per item.
constexpr int kRowStride = kProducerThreads / 8;   // rows between a thread's items
constexpr int kItemsPerThread = (kRowsPerChunk + kRowStride - 1) / kRowStride;
static_assert(kProducerThreads % 8 == 0, "segment fixed per thread");

// Per-thread, per-query source bases (segment offset folded in).
struct Src {
  const uint8_t *sel_b;   // row kv0 of the pool
  const float *sel_s;
  const uint8_t *win_b;   // first window row of the SWA buffer
  const float *win_s;
  const uint8_t *dummy_b; // a readable row for rows past the end (masked when stored)
  const float *dummy_s;
  int64_t nsel, nrows;
};

__device__ __forceinline__ void load_step(const int *list, const Src &S, int row0, int chunk,
                                          int pair, Item (&it)[kItemsPerThread]) {
  const int64_t r0 = (int64_t)chunk * kRowsPerChunk;
  const int cb = pair * 128, sb = pair * 4;
  if (r0 + kRowsPerChunk <= S.nsel) {          // every row selected
#pragma unroll
    for (int i = 0; i < kItemsPerThread; ++i) {
      if (row0 + i * kRowStride < kRowsPerChunk) {
        const int64_t j = list[r0 + row0 + i * kRowStride];
        it[i].codes = __ldg(reinterpret_cast<const uint4 *>(S.sel_b + j * kDim + cb));
        it[i].scale = __ldg(S.sel_s + j * (kDim / 32) + sb);
      }
    }
  } else if (r0 >= S.nsel && r0 + kRowsPerChunk <= S.nrows) {   // every row in the window
#pragma unroll
    for (int i = 0; i < kItemsPerThread; ++i) {
      if (row0 + i * kRowStride < kRowsPerChunk) {
        const int64_t w = r0 + row0 + i * kRowStride - S.nsel;
        it[i].codes = __ldg(reinterpret_cast<const uint4 *>(S.win_b + w * kDim + cb));
        it[i].scale = __ldg(S.win_s + w * (kDim / 32) + sb);
      }
    }
  } else {                                     // boundary or last chunk
#pragma unroll
    for (int i = 0; i < kItemsPerThread; ++i) {
      if (row0 + i * kRowStride < kRowsPerChunk) {
        const int64_t ri = r0 + row0 + i * kRowStride;
        const uint8_t *b;
        const float *sc;
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
        it[i].codes = __ldg(reinterpret_cast<const uint4 *>(b + cb));
        it[i].scale = __ldg(sc + sb);
      }
    }
  }
}

// Dequantise a step into R.  off[i][0..1]: byte offsets (pair 0) of the two
// 16-byte stores of item i.  The 8 threads of a store phase cover one row's 8
// segments; segments 0-3 and 4-7 fall in two column blocks whose 16-byte
// chunks share banks, so threads of segments 4-7 store their upper half
// first: every phase then touches 8 distinct chunk positions.
template <bool kMasked>
__device__ __forceinline__ void store_step(uint8_t *R, int pair, bool swap, int row0,
                                           const uint32_t (&off)[kItemsPerThread][2],
                                           int64_t valid_rows, const Item (&it)[kItemsPerThread]) {
  uint8_t *Rb = R + pair * 2 * kRBlock;
#pragma unroll
  for (int i = 0; i < kItemsPerThread; ++i) {
    if (row0 + i * kRowStride < kRowsPerChunk) {
      uint4 cd = it[i].codes;
      float sc = it[i].scale;
      if (kMasked && row0 + i * kRowStride >= valid_rows) {
        cd = make_uint4(0, 0, 0, 0);
        sc = 0.f;
      }
      const __half2 s2 = __float2half2_rn(sc);
      const uint32_t a = swap ? cd.z : cd.x, b = swap ? cd.w : cd.y;
      const uint32_t c = swap ? cd.x : cd.z, d = swap ? cd.y : cd.w;
      uint32_t h[8];
      e4m3x4_f16x4(a, h[0], h[1]);
      e4m3x4_f16x4(b, h[2], h[3]);
      e4m3x4_f16x4(c, h[4], h[5]);
      e4m3x4_f16x4(d, h[6], h[7]);
#pragma unroll
      for (int j = 0; j < 8; ++j) h[j] = hmul2_u32(h[j], s2);
      const uint4 first = make_uint4(h[0], h[1], h[2], h[3]);
      const uint4 second = make_uint4(h[4], h[5], h[6], h[7]);
      *reinterpret_cast<uint4 *>(Rb + off[i][0]) = first;
      *reinterpret_cast<uint4 *>(Rb + off[i][1]) = second;
    }
  }
}

__device__ void producer_role(const Params &P, uint8_t *smem, Misc *ms) {
  const int ptid = threadIdx.x - kProducerWarp0 * 32;
  const int lane = threadIdx.x & 31;
  const int row0 = ptid >> 3, seg = ptid & 7;
  const bool swap = (seg & 4) != 0;
  uint32_t off[kItemsPerThread][2];   // R byte offsets of this thread's stores (pair 0)
#pragma unroll
  for (int i = 0; i < kItemsPerThread; ++i) {
    const uint32_t row = (uint32_t)(row0 + i * kRowStride);
    const uint32_t lo = sw128_offset(row, seg * 16, kRBlock), hi = sw128_offset(row, seg * 16 + 8, kRBlock);
    off[i][0] = swap ? hi : lo;
    off[i][1] = swap ? lo : hi;
  }
  uint8_t *R = smem + kOffR;
  uint8_t *Qs = smem + kOffQ;
  const int *lists = reinterpret_cast<const int *>(smem + kOffList);
  uint32_t g = 0;  // chunks produced by this CTA
  uint32_t qi = 0;
  for (int q = blockIdx.x; q < P.b.num_q; q += gridDim.x, ++qi) {
    // ---- Q of this query (f16, heads zero-padded to 64)
    if (!wait_bar(&ms->q_empty, (qi & 1) ^ 1, ms)) break;
    const __nv_bfloat16 *qg = P.q + (int64_t)q * P.n_heads * kDim;
    // raw bf16 chunks land at their final swizzled place; each thread then
    // converts exactly the chunks it copied (f16 and bf16 are both 2 bytes)
    for (int it = ptid; it < kHeadsPad * (kDim / 8); it += kProducerThreads) {
      const int h = it / (kDim / 8), d = (it % (kDim / 8)) * 8;
      uint8_t *dst = Qs + sw128_offset(h, d, kQBlock);
      if (h < P.n_heads) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
                     "l"(qg + (int64_t)h * kDim + d)
                     : "memory");
      } else {
        *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    for (int it = ptid; it < P.n_heads * (kDim / 8); it += kProducerThreads) {
      const int h = it / (kDim / 8), d = (it % (kDim / 8)) * 8;
      uint4 *p4 = reinterpret_cast<uint4 *>(Qs + sw128_offset(h, d, kQBlock));
      const uint4 raw = *p4;
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xffff0000u);
        __half2 hh = __floats2half2_rn(lo, hi);
        o[j] = *reinterpret_cast<uint32_t *>(&hh);
      }
      *p4 = make_uint4(o[0], o[1], o[2], o[3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ms->q_full);
    // ---- row list (first producer warp), shared with the other producers
    // ---- row list and counts of this query (built one query ahead by the
    // first softmax warp)
    const uint32_t ms_slot = qi & 1;
    if (!wait_bar(&ms->meta_full[ms_slot], (qi >> 1) & 1, ms)) break;
    const int *list = lists + ms_slot * kMaxSel;
    Src S;
    S.nsel = ms->meta[ms_slot][0];
    S.nrows = S.nsel + ms->meta[ms_slot][1];
    const int64_t win_first = ms->meta[ms_slot][2];
    const int64_t kv0 = ms->meta[ms_slot][3];
    S.sel_b = P.kv_fp8 + kv0 * kDim + seg * 16;
    S.sel_s = P.kv_scale + kv0 * (kDim / 32) + seg / 2;
    S.win_b = P.swa_fp8 + win_first * kDim + seg * 16;
    S.win_s = P.swa_scale + win_first * (kDim / 32) + seg / 2;
    S.dummy_b = P.swa_fp8 + seg * 16;
    S.dummy_s = P.swa_scale + seg / 2;
    const int nch = n_chunks_of(S.nrows);
    // ---- chunks: 4 steps of 128 channels each; the loads of the next two
    // steps are in flight while a step waits for its buffer and is stored
    const int nsteps = nch * 4;
    Item b0[kItemsPerThread], b1[kItemsPerThread], b2[kItemsPerThread];
    load_step(list, S, row0, 0, 0, b0);
    if (nsteps > 1) load_step(list, S, row0, 0, 1, b1);
    bool ok = true;
    // one step: prefetch step st+2 into `pre`, then store step st from `use`
    auto step = [&](int st, Item(&use)[kItemsPerThread], Item(&pre)[kItemsPerThread]) -> bool {
      const int c = st >> 2, pair = st & 3;
      if (st + 2 < nsteps) load_step(list, S, row0, (st + 2) >> 2, (st + 2) & 3, pre);
      if (!wait_bar(&ms->r_empty[pair], ((g + c) & 1) ^ 1, ms)) return false;
      const int64_t valid_rows = S.nrows - (int64_t)c * kRowsPerChunk;
      if (valid_rows >= kRowsPerChunk)
        store_step<false>(R, pair, swap, row0, off, valid_rows, use);
      else
        store_step<true>(R, pair, swap, row0, off, valid_rows, use);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms->r_full[pair]);
      return true;
    };
    for (int st = 0; st < nsteps && ok; st += 3) {
      ok = step(st, b0, b2);
      if (ok && st + 1 < nsteps) ok = step(st + 1, b1, b0);
      if (ok && st + 2 < nsteps) ok = step(st + 2, b2, b1);
    }
    g += nch;
    if (!ok) break;
  }
}

// ---------------------------------------------------------------------------
// MMA issuer: the whole warp walks the queries (row counts need the warp),
// lane 0 waits on the barriers and issues every MMA and commit.
// ---------------------------------------------------------------------------
__device__ void mma_role(const Params &P, uint8_t *smem, Misc *ms) {
  const int lane = threadIdx.x & 31;
  const uint32_t tmem = ms->tmem_base;
  const uint32_t r0 = smem_u32(smem + kOffR), q0 = smem_u32(smem + kOffQ),
                 p0 = smem_u32(smem + kOffP);
  const uint32_t id_s = make_idesc_f16(128, kHeadsPad, false, false);
  const uint32_t id_o = make_idesc_f16(128, kHeadsPad, true, true);
  // base descriptors; every MMA's operand descriptor is one of these plus a
  // compile-time offset
  const uint64_t d_rk = make_desc_sw128(r0, 16, 1024);        // R, K-major (S)
  const uint64_t d_q = make_desc_sw128(q0, 16, 1024);         // Q, K-major (S)
  const uint64_t d_rm = make_desc_sw128(r0, kRBlock, 1024);   // R^T, MN-major (O)
  const uint64_t d_p = make_desc_sw128(p0, kRBlock, 1024);    // P^T, MN-major (O)
  const uint32_t rk_lo = (uint32_t)d_rk, rk_hi = (uint32_t)(d_rk >> 32);
  const uint32_t q_lo = (uint32_t)d_q, q_hi = (uint32_t)(d_q >> 32);
  const uint32_t rm_lo = (uint32_t)d_rm, rm_hi = (uint32_t)(d_rm >> 32);
  const uint32_t p_lo = (uint32_t)d_p, p_hi = (uint32_t)(d_p >> 32);
  uint32_t g = 0, qi = 0;
  int ok = 1;
  for (int q = blockIdx.x; q < P.b.num_q && lane == 0; q += gridDim.x, ++qi) {
    {
      const uint32_t slot = qi & 1;
      if (!(ok = wait_bar(&ms->meta_full[slot], (qi >> 1) & 1, ms))) break;
      const int nch = n_chunks_of(ms->meta[slot][0] + ms->meta[slot][1]);
      for (int c = 0; c < nch && ok; ++c, ++g) {
        const uint32_t sb = g & 1;
        const uint32_t s_tmem = tmem + kColS + sb * 64;
        // ---- S^T(c) = R . Q^T into S buffer sb
        ok = wait_bar(&ms->s_empty[sb], ((g >> 1) & 1) ^ 1, ms);
        if (ok && c == 0) ok = wait_bar(&ms->q_full, qi & 1, ms);
        for (int pair = 0; pair < 4 && ok; ++pair) {
          ok = wait_bar(&ms->r_full[pair], g & 1, ms);
          if (!ok) break;
          fence_after_sync();
          const uint32_t a_p = rk_lo + ((pair * 2 * kRBlock) >> 4);
          const uint32_t b_p = q_lo + ((pair * 2 * kQBlock) >> 4);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t oa = ((kk >> 2) * kRBlock + (kk & 3) * 32) >> 4;
            const uint32_t ob = ((kk >> 2) * kQBlock + (kk & 3) * 32) >> 4;
            mma_f16_split(s_tmem, a_p + oa, rk_hi, b_p + ob, q_hi, id_s,
                          (pair > 0 || kk > 0) ? 1u : 0u);
          }
        }
        if (!ok) break;
        mma_commit(&ms->s_full[sb]);
        if (c == nch - 1) mma_commit(&ms->q_empty);
        // ---- O^T += R^T . P^T, 4 tiles of 128 channels
        ok = wait_bar(&ms->p_full, g & 1, ms);
        if (ok && c == 0) ok = wait_bar(&ms->o_empty, (qi & 1) ^ 1, ms);
        if (!ok) break;
        fence_after_sync();
#pragma unroll
        for (int t = 0; t < 4; ++t) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            mma_f16_split(tmem + kColO + t * 64, rm_lo + ((t * 2 * kRBlock + ks * 2048) >> 4),
                          rm_hi, p_lo + ((ks * 2048) >> 4), p_hi, id_o,
                          (c > 0 || ks > 0) ? 1u : 0u);
          }
          mma_commit(&ms->r_empty[t]);
        }
        mma_commit(&ms->p_empty);
        if (c == nch - 1) mma_commit(&ms->o_full);
      }
    }
    if (!ok) break;
  }
  // drain: every MMA issued so far has completed once `done` flips (bounded
  // by time only, so that TMEM is never freed under a running MMA)
  if (lane == 0) {
    mma_commit(&ms->done);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&ms->done, 0) && globaltimer() - t0 < kWaitNs) {
    }
  }
  __syncwarp();
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
  uint8_t *Pbuf = smem + kOffP;
  const float NEG_INF = -INFINITY;
  float lsum[32];
  uint32_t g = 0, qi = 0, gp = 0;
  bool ok = true;
  int err = 0;
  int *lists = reinterpret_cast<int *>(smem + kOffList);
  // Row lists and counts are built by warp 0 one query ahead of their use.
  // Slot (qi+1)&1 was last read for query qi-1, whose chunks have all been
  // produced and consumed before this role reaches query qi.
  auto publish = [&](int qn, uint32_t qin) {
    if (warp != 0 || qn >= P.b.num_q) return;
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
  };
  publish(blockIdx.x, 0);
  if (stid < 64) ms->m_ref[stid] = NEG_INF;
  ok = group_sync(&ms->sm_grp, gp, ms);
  for (int q = blockIdx.x; q < P.b.num_q && ok; q += gridDim.x, ++qi) {
    const uint32_t slot = qi & 1;
    if (!(ok = wait_bar(&ms->meta_full[slot], (qi >> 1) & 1, ms))) break;
    const int64_t nrows = ms->meta[slot][0] + ms->meta[slot][1];
    const int nch = n_chunks_of(nrows);
    publish(q + gridDim.x, qi + 1);
#pragma unroll
    for (int j = 0; j < 32; ++j) lsum[j] = 0.f;
    for (int c = 0; c < nch; ++c, ++g) {
      const uint32_t sb = g & 1;
      ok = wait_bar(&ms->s_full[sb], (g >> 1) & 1, ms);
      if (!ok) break;
      fence_after_sync();
      uint32_t v[32];
      tmem_ld32x32b_x32(tmem + lane_addr + kColS + sb * 64 + 32 * hh, v);
      tmem_wait_ld();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms->s_empty[sb]);
      const int64_t row = (int64_t)c * kRowsPerChunk + 32 * sp + lane;
      const bool valid = row < nrows;
      float x[32];
      bool exceed = false;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        x[j] = valid ? __uint_as_float(v[j]) * P.scale_log2 : NEG_INF;
        exceed |= x[j] > ms->m_ref[32 * hh + j] + 8.f;
      }
      // does any logit of the chunk exceed its head's reference by 2^8?
      const int vb = g & 1;
      const bool vote = __any_sync(0xffffffffu, exceed);
      if (lane == 0) ms->votes[vb][warp] = vote ? 1 : 0;
      if (!(ok = group_sync(&ms->sm_grp, gp, ms))) break;
      bool slow = false;
#pragma unroll
      for (int w = 0; w < kSoftmaxWarps; ++w) slow |= ms->votes[vb][w] != 0;
      if (slow) {
        // per-head maximum over the warp's 32 rows (butterfly per head), then
        // across the 4 warps of this head half
        float mine = NEG_INF;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float mj = x[j];
#pragma unroll
          for (int w = 16; w >= 1; w >>= 1) mj = fmaxf(mj, __shfl_xor_sync(0xffffffffu, mj, w));
          if (lane == j) mine = mj;
        }
        ms->red[sp][32 * hh + lane] = mine;
        if (!(ok = group_sync(&ms->sm_grp, gp, ms))) break;
        if (stid < 64) {
          const float old = ms->m_ref[stid];
          float mx = fmaxf(fmaxf(ms->red[0][stid], ms->red[1][stid]),
                           fmaxf(ms->red[2][stid], ms->red[3][stid]));
          mx = fmaxf(mx, old);
          ms->alpha[stid] = (old == NEG_INF) ? 0.f : exp2f(old - mx);
          ms->m_ref[stid] = mx;
        }
        if (!(ok = group_sync(&ms->sm_grp, gp, ms))) break;
#pragma unroll
        for (int j = 0; j < 32; ++j) lsum[j] *= ms->alpha[32 * hh + j];
      }
      // P(c) may be written once O^T(c-1) has consumed P(c-1); that also
      // means every earlier O^T MMA has completed (needed for a rescale)
      ok = wait_bar(&ms->p_empty, (g & 1) ^ 1, ms);
      if (!ok) break;
      fence_after_sync();
      if (slow && c > 0) {
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
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float m0 = ms->m_ref[32 * hh + j], m1 = ms->m_ref[32 * hh + j + 1];
        const float p0 = ex2(x[j] - (m0 == NEG_INF ? 0.f : m0));
        const float p1 = ex2(x[j + 1] - (m1 == NEG_INF ? 0.f : m1));
        lsum[j] += p0;
        lsum[j + 1] += p1;
        __half2 h2 = __floats2half2_rn(p0, p1);
        pk[j / 2] = *reinterpret_cast<uint32_t *>(&h2);
      }
      const int prow = 32 * sp + lane;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint4 *>(Pbuf + sw128_offset(prow, 32 * hh + 8 * i, 0)) =
            make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      fence_proxy_async_smem();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms->p_full);
    }
    if (!ok) break;
    // ---- epilogue: row sums, normalisation, bf16 output, lse
    float lmine = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      float lj = lsum[j];
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1) lj += __shfl_xor_sync(0xffffffffu, lj, w);
      if (lane == j) lmine = lj;
    }
    ms->red[sp][32 * hh + lane] = lmine;
    if (!(ok = group_sync(&ms->sm_grp, gp, ms))) break;
    if (stid < 64) {
      float l = (ms->red[0][stid] + ms->red[1][stid]) + (ms->red[2][stid] + ms->red[3][stid]);
      const float m = ms->m_ref[stid];
      const float mu = m == NEG_INF ? 0.f : m;
      if (P.sink && stid < P.n_heads) l += exp2f(P.sink[stid] * 1.4426950408889634f - mu);
      ms->alpha[stid] = l > 0.f ? 1.f / l : 0.f;
      if (P.lse && stid < P.n_heads)
        P.lse[(int64_t)q * P.n_heads + stid] =
            l > 0.f ? (mu + log2f(l)) * 0.6931471805599453f : NEG_INF;
      ms->m_ref[stid] = NEG_INF;   // reference of the next query
    }
    if (!(ok = group_sync(&ms->sm_grp, gp, ms))) break;
    ok = wait_bar(&ms->o_full, qi & 1, ms);
    if (!ok) break;
    fence_after_sync();
    __nv_bfloat16 *og = P.out + (int64_t)q * P.n_heads * kDim;
    for (int t = 0; t < 4; ++t) {
      uint32_t o[32];
      tmem_ld32x32b_x32(tmem + lane_addr + kColO + t * 64 + 32 * hh, o);
      tmem_wait_ld();
      const int d = t * 128 + 32 * sp + lane;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int h = 32 * hh + j;
        if (h < P.n_heads)
          og[(int64_t)h * kDim + d] = __float2bfloat16_rn(__uint_as_float(o[j]) * ms->alpha[h]);
      }
    }
    fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ms->o_empty);
  }
  if (warp == 0) {
    err = __reduce_or_sync(0xffffffffu, err);
    if (lane == 0) raise_err(P.d_err, err);
  }
}

__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(Params P) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Misc *ms = reinterpret_cast<Misc *>(smem + kOffMisc);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&ms->q_full, kProducerWarps);
    mbar_init(&ms->q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->s_full[i], 1);
      mbar_init(&ms->s_empty[i], kSoftmaxWarps);
    }
    mbar_init(&ms->p_full, kSoftmaxWarps);
    mbar_init(&ms->p_empty, 1);
    mbar_init(&ms->o_full, 1);
    mbar_init(&ms->o_empty, kSoftmaxWarps);
    mbar_init(&ms->done, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&ms->r_full[i], kProducerWarps);
      mbar_init(&ms->r_empty[i], 1);
    }
    mbar_init(&ms->sm_grp, kSoftmaxWarps);
    for (int i = 0; i < 2; ++i) mbar_init(&ms->meta_full[i], 1);
    ms->abort = 0;
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
    mma_role(P, smem, ms);
  } else {
    producer_role(P, smem, ms);
  }
  fence_before_sync();
  __syncthreads();
  if (ms->abort && threadIdx.x == 0) raise_err(P.d_err, kDerrTimeout);
  if (warp == kMmaWarp) {
    fence_after_sync();
    tmem_dealloc(ms->tmem_base, kTmemCols);
  }
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

}  // namespace

int attn_tc(const Batch &b, int n_heads, const __nv_bfloat16 *q, const uint8_t *kv_fp8,
            const float *kv_scale, const int32_t *idx, int k, const uint8_t *swa_fp8,
            const float *swa_scale, const int64_t *win_lo, int window, float sm_scale,
            const float *sink, __nv_bfloat16 *out, float *lse, int32_t *d_err,
            cudaStream_t st) {
  if (b.num_q == 0) return CSA2_OK;
  if (n_heads > kHeadsPad || k > kMaxSel) return CSA2_ERR_UNSUPPORTED;
  // 16-byte vector loads and asynchronous copies need 16-byte aligned rows
  if (((uintptr_t)q | (uintptr_t)kv_fp8 | (uintptr_t)swa_fp8) & 15u) return CSA2_ERR_UNSUPPORTED;
  Params P;
  P.b = b;
  P.n_heads = n_heads;
  P.q = q;
  P.kv_fp8 = kv_fp8;
  P.kv_scale = kv_scale;
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
  cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)kSmemBytes);
  const int grid = b.num_q < sm_count() ? b.num_q : sm_count();
  attn_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(P);
  return launch_status();
}

}  // namespace csa2

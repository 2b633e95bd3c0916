// a2-a4, a7 on the 5th-generation tensor cores: index scores
//
//   s(q, j) = sum_h w[q,h] * max(0, <Qi[q,h], Ki[j]>)
//
// ("DeepSeek V4.1 Flash 建模", CSA2 and Hierarchical Sparse Indexer cards;
// SGLang/Miles day-0 article sec. 5: an MQA-shaped indexer over the FP4 keys
// of the nearest KV source, heads replicated.)
//
// Formulation.  The contraction is written with the keys as the MMA M
// dimension and (query, head) pairs as N:
//   D[j, (q,h)] = sum_d K[j, d] Qi[q, h, d]     (M = 128 keys, N <= 256, K = 128)
// so that the head reduction is a per-thread loop in the epilogue: thread j
// reads its TMEM lane (key j) and sums w[q,h] * ReLU(D[j, (q,h)]) over the
// head columns of query q.  MXFP4 operands are dequantised to f16 in shared
// memory: an E2M1 value times a power-of-two scale is exact in f16 (for
// scales in [2^-23, 2^12]), every product is exact, and so is the fp32 sum of
// one 32-channel group; the sum across the four groups of a 128-channel dot
// rounds in fp32 when their scales spread it past 24 bits (the tensor core's
// accumulation order is unspecified), and the head sum rounds.  The scores are
// held to 1e-5 of sum_h |w_h| ReLU(dot_h).
//
// Work unit (one CTA): a tile of 256/Hi consecutive query rows and a chunk of
// key tiles: 128 (16384 keys, or 128 sampled tiles) when that covers the
// longest row, else 64; 32 (4096 slots) in pool mode.
// Rows of the tile that belong to the same request share key tiles ("runs",
// full mode); in pool mode every query has its own slot list and is its own
// run, except that identity pools (blocks 0, 1, ..., nb-1: nothing excluded,
// the case when every reachable position fits the pool budget) map slot s to
// entry s and merge like full mode.  Roles (16 warps):
//   warps 0-7   epilogue (warp w: TMEM lanes 32*(w%4).., queries of parity w/4)
//   warp 8      TMEM allocation; lane 0 issues the MMAs
//   warps 9-15  producers: key gather + E2M1 -> f16 into a 4-stage ring, one
//               key tile of loads in flight ahead of the ring
// Prologue: the query operand's loads are issued first, the tile geometry is
// worked out while they are in flight, and the producers start on the key
// tiles while warps 0-8 dequantise the query operand and allocate TMEM.
// Waits are time-bounded (two seconds unless csa2_set_wait_limit_ns says
// otherwise; CSA2_DERR_TIMEOUT on expiry, after which the MMAs in flight are
// drained for at most two seconds and TMEM is freed).
#include "common.cuh"
#include "kernels.cuh"
#include "tcgen05.cuh"

namespace csa2 {
namespace {

using namespace tc;

constexpr int kKeyTile = 128;
// key tiles per CTA: over full rows 128 (16384 keys) when one chunk covers
// the longest row, so that each query tile is one CTA, else 64; in pool mode
// 32 (4096 slots), whose candidate blocks are copied to shared memory
constexpr int kTilesWhole = 128;
constexpr int kTilesFull = 64;
constexpr int kTilesPool = 32;
constexpr int kStages = 4;
constexpr int kEpiWarps = 8;
constexpr int kMmaWarp = 8;
constexpr int kProdWarp0 = 9;
constexpr int kProdWarps = 7;
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kBRows = 256 + 16;       // (query, head) rows + padding for N rounding

constexpr uint32_t kABlock = kKeyTile * 128;           // 16 KB: one 64-column block
constexpr uint32_t kAStage = 2 * kABlock;              // 32 KB: 128 keys x 128 f16
constexpr uint32_t kBBlock = kBRows * 128;             // 34 KB
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kAStage;  // 128 KB
constexpr uint32_t kOffMisc = kOffB + 2 * kBBlock;     // +68 KB
constexpr uint32_t kOffCand = kOffMisc + 4096;         // candidate blocks of the chunk
constexpr int kCandInts = 4096;                        // (16 KB; used when they fit)
constexpr uint32_t kSmemBytes = kOffCand + kCandInts * 4;

constexpr uint64_t kWaitNs = 2000000000ull;   // the MMA drain (pipeline waits: Params::wait_ns)
constexpr int kDerrTimeout = 128;
constexpr int kMaxQT = 32;

struct RunInfo {
  int64_t kv0;  // pool row of the request's entry 0
  int ql0, nq, req;
  int gather;   // 1: slots map through the query's candidate blocks
  int64_t len;  // longest row of the run
  int64_t lim;  // entries below lim hold keys (slots past it are empty)
};

struct Misc {
  uint64_t a_full[kStages], a_empty[kStages], d_full[2], d_empty[2], done;
  uint64_t wait_ns;          // bound on every pipeline wait
  uint32_t tmem_base;
  int abort;
  int nruns;
  RunInfo runs[kMaxQT];
  int64_t row_len[kMaxQT];   // per query of the tile (0 past the batch)
  int64_t n_vis[kMaxQT];
  int req[kMaxQT];           // request of each query of the tile
  int64_t kv0[kMaxQT];       // pool row of that request's entry 0
  int nb[kMaxQT];            // pool mode: candidate blocks per query
  int ident[kMaxQT];         // pool mode: blocks are 0..nb-1
  int cand_smem;             // pool mode: the chunk's candidate blocks are in shared memory
  int cand_span, b_lo;       //   as [query of the tile][block - b_lo]
  float thr[kMaxQT];         // list mode: per-query threshold
  alignas(16) float w[256];  // head weights of the tile, halved
};
static_assert(sizeof(Misc) <= 4096, "misc");

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

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

__device__ __forceinline__ bool mx_scale_ok(float s) {
  const uint32_t u = __float_as_uint(s);
  const int e = (int)((u >> 23) & 0xff) - 127;
  return (u & 0x807fffffu) == 0 && e >= -23 && e <= 12;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, __half2 s) {
  __half2 x = *reinterpret_cast<__half2 *>(&a);
  x = __hmul2(x, s);
  return *reinterpret_cast<uint32_t *>(&x);
}

// 32 E2M1 codes (16 bytes) times a power-of-two scale -> 32 f16 (4 x uint4)
__device__ __forceinline__ void dequant32(const uint4 c, float scale, uint4 (&o)[4]) {
  const __half2 s2 = __float2half2_rn(scale);
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h[4];
    e2m1x8_f16x8(w[i], h);
#pragma unroll
    for (int b = 0; b < 4; ++b) h[b] = hmul2_u32(h[b], s2);
    o[i] = make_uint4(h[0], h[1], h[2], h[3]);
  }
}

struct Params {
  Batch b;
  int hi;              // index heads
  int qt;              // queries per tile = 256 / hi
  const uint8_t *q_fp4;
  const float *q_scale;
  const float *head_w;
  const uint8_t *k_fp4;
  const float *k_scale;
  const int32_t *cand;
  int block, max_blocks;
  float *scores;
  int64_t ld;          // row capacity in entries (rows past it are cut, CSA2_DERR_LD)
  int tpc;             // key tiles per CTA chunk
  int64_t out_ld;      // row stride of `scores` (sample mode: ld / stride tiles)
  int stride;          // 1: every key tile; S: tiles 0, S, 2S, .. only, stored densely
  // list mode (list_cnt != nullptr): no dense scores; each query appends the
  // (entry, score) pairs with score >= list_thr[q] to its list of list_cap
  // slots (the counter keeps counting past the capacity)
  const float *list_thr;
  uint32_t *list_cnt;
  int32_t *list_ent;
  float *list_val;
  int list_cap;
  int32_t *d_err;
  uint64_t wait_ns;
};

// key tiles of a row of `len` keys walked by this launch (every stride-th)
template <int STRIDE>
__device__ __forceinline__ int64_t walked_tiles(int64_t len) {
  constexpr int stride = STRIDE;
  const int64_t nt = (len + kKeyTile - 1) / kKeyTile;
  return (nt + stride - 1) / stride;
}

// Candidate-block view of the tile, copied to registers once per tile: block
// of slot s (a shift for power-of-two block sizes), and the entry it holds.
struct CandView {
  const int32_t *smem;   // [query of the tile][block - b_lo], or nullptr: global
  const int32_t *glob;   // P.cand
  int span, b_lo, max_blocks, block, shift;
  __device__ __forceinline__ int blk(int s) const { return shift >= 0 ? s >> shift : s / block; }
  __device__ __forceinline__ int64_t entry(int ql, int q, int s) const {
    const int b = blk(s);
    const int64_t c = smem ? smem[ql * span + (b - b_lo)] : glob[(int64_t)q * max_blocks + b];
    return c * block + (s - b * block);
  }
};

__device__ __forceinline__ CandView cand_view(const Params &P, const Misc *ms,
                                              const uint8_t *smem) {
  CandView v;
  v.smem = ms->cand_smem ? reinterpret_cast<const int32_t *>(smem + kOffCand) : nullptr;
  v.glob = P.cand;
  v.span = ms->cand_span;
  v.b_lo = ms->b_lo;
  v.max_blocks = P.max_blocks;
  v.block = P.block;
  v.shift = (P.block & (P.block - 1)) == 0 ? __ffs(P.block) - 1 : -1;
  return v;
}

// ---------------------------------------------------------------------------
// producers: the (run, key tile) sequence of this CTA; the loads of tile i+1
// are issued before tile i is converted and stored.
// ---------------------------------------------------------------------------
constexpr int kProdItems = (kKeyTile * 4 + kProdThreads - 1) / kProdThreads;

struct KeyLoad {
  uint4 codes[kProdItems];
  float sc[kProdItems];
  uint32_t valid;  // bit i: item i holds a visible key (else zeroed when stored)
};
static_assert(kProdThreads % 4 == 0, "a thread's items share one 32-dim group");

// Key rows of tile kt of run ri: full mode, entry s of the run's request;
// pool mode, the entry of the query's candidate-block slot s.  Slots past the
// run's keys (or, in pool mode, holding no visible entry) read key row 0 and
// are zeroed when stored: every load is issued unconditionally, so no load
// waits on another.
template <int STRIDE>
__device__ __forceinline__ void load_tile(const Params &P, const Misc *ms, const CandView &cv,
                                          int ri, int64_t kt, int q0, int ptid, KeyLoad &L) {
  const RunInfo ru = ms->runs[ri];
  const int s0 = (int)kt * STRIDE * kKeyTile;
  const int lim = (int)(ru.gather ? ru.len : min(ru.len, ru.lim));
  const int64_t nvis = ms->n_vis[ru.ql0];
  L.valid = 0;
#pragma unroll
  for (int i = 0; i < kProdItems; ++i) {
    const int item = ptid + i * kProdThreads;
    const int row = item >> 2, grp = item & 3;
    const int s = s0 + row;
    bool v = item < kKeyTile * 4 && s < lim;
    int64_t j = s;
    if (ru.gather) {
      j = v ? cv.entry(ru.ql0, q0 + ru.ql0, s) : 0;
      v = v && j < nvis;
    }
    L.valid |= (v ? 1u : 0u) << i;
    const int64_t g = v ? ru.kv0 + j : 0;
    L.codes[i] = __ldg(reinterpret_cast<const uint4 *>(P.k_fp4 + g * 64) + grp);
    L.sc[i] = __ldg(P.k_scale + g * 4 + grp);
  }
}

// next (run, tile) after (ri, kt) within key chunk y; false when none is left
template <int STRIDE>
__device__ __forceinline__ bool next_item(const Misc *ms, int y, int tpc, int &ri, int64_t &kt) {
  ++kt;
  while (ri < ms->nruns) {
    const int64_t nt = walked_tiles<STRIDE>(ms->runs[ri].len);
    const int64_t hi = min(nt, (int64_t)(y + 1) * tpc);
    if (kt < hi) return true;
    ++ri;
    kt = (int64_t)y * tpc;
  }
  return false;
}

template <int STRIDE, int TPC>
__device__ void producer_role(const Params &P, uint8_t *smem, Misc *ms, int q0, int y) {
  const int ptid = threadIdx.x - kProdWarp0 * 32;
  const int lane = threadIdx.x & 31;
  int err = 0;
  uint32_t it = 0;
  int ri = 0;
  int64_t kt = (int64_t)y * TPC - 1;
  if (!next_item<STRIDE>(ms, y, TPC, ri, kt)) return;
  KeyLoad ka, kb;
  const CandView cv = cand_view(P, ms, smem);
  load_tile<STRIDE>(P, ms, cv, ri, kt, q0, ptid, ka);
  bool more = true;
  // store the tile held in `use` after issuing the loads of the next tile
  // into `pre` (two fixed buffers: no register copy waits on pending loads)
  auto step = [&](KeyLoad &use, KeyLoad &pre) -> bool {
    int ri2 = ri;
    int64_t kt2 = kt;
    more = next_item<STRIDE>(ms, y, TPC, ri2, kt2);
    if (more) load_tile<STRIDE>(P, ms, cv, ri2, kt2, q0, ptid, pre);
    const uint32_t st = it % kStages;
    if (!wait_bar(&ms->a_empty[st], ((it / kStages) & 1) ^ 1, ms)) return false;
    uint8_t *A = smem + kOffA + st * kAStage;
#pragma unroll
    for (int i = 0; i < kProdItems; ++i) {
      const int item = ptid + i * kProdThreads;
      if (item >= kKeyTile * 4) break;
      const int row = item >> 2, grp = item & 3;
      const bool v = (use.valid >> i) & 1u;
      const float sc = v ? use.sc[i] : 0.f;
      if (v && sc != 0.f && !mx_scale_ok(sc)) err |= CSA2_DERR_SCALE;
      // groups 2-3 sit in the second 64-column block, whose 16-byte chunk
      // positions repeat the first block's: they store their chunks rotated
      // by two, so the 8 threads of a store phase hit 8 distinct positions
      const bool rot = (grp & 2) != 0;
      const uint4 c0 = v ? use.codes[i] : make_uint4(0, 0, 0, 0);
      const uint4 cr = rot ? make_uint4(c0.z, c0.w, c0.x, c0.y) : c0;
      uint4 o[4];
      dequant32(cr, sc, o);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int cc = rot ? (c + 2) & 3 : c;
        *reinterpret_cast<uint4 *>(A + sw128_offset(row, grp * 32 + cc * 8, kABlock)) = o[c];
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ms->a_full[st]);
    ++it;
    ri = ri2;
    kt = kt2;
    return true;
  };
  while (true) {
    if (!step(ka, kb) || !more) break;
    if (!step(kb, ka) || !more) break;
  }
  err = __reduce_or_sync(0xffffffffu, err);
  if (lane == 0) raise_err(P.d_err, err);
}

template <int STRIDE, int TPC>
__device__ void mma_role(const Params &P, uint8_t *smem, Misc *ms, int y) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    const uint32_t tmem = ms->tmem_base;
    const uint32_t b0 = smem_u32(smem + kOffB);
    uint32_t it = 0;
    bool ok = true;
    for (int ri = 0; ri < ms->nruns && ok; ++ri) {
      const RunInfo ru = ms->runs[ri];
      const int64_t nt = walked_tiles<STRIDE>(ru.len);
      uint32_t n = (uint32_t)(ru.nq * P.hi);
      n = (n + 15u) & ~15u;
      const uint32_t idesc = make_idesc_f16(128, n, false, false);
      const uint32_t brow = (uint32_t)(ru.ql0 * P.hi) * 128u;   // byte offset of the run's rows
      for (int64_t kt = (int64_t)y * TPC;
           kt < nt && kt < (int64_t)(y + 1) * TPC; ++kt, ++it) {
        const uint32_t st = it % kStages, db = it & 1;
        if (!(ok = wait_bar(&ms->a_full[st], (it / kStages) & 1, ms))) break;
        if (!(ok = wait_bar(&ms->d_empty[db], ((it >> 1) & 1) ^ 1, ms))) break;
        fence_after_sync();
        const uint32_t a0 = smem_u32(smem + kOffA + st * kAStage);
        const uint64_t da = make_desc_sw128(a0, 16, 1024);
        const uint64_t dbq = make_desc_sw128(b0 + brow, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          mma_f16(tmem + db * 256, desc_add(da, (kk >> 2) * kABlock + (kk & 3) * 32),
                  desc_add(dbq, (kk >> 2) * kBBlock + (kk & 3) * 32), idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(&ms->a_empty[st]);
        mma_commit(&ms->d_full[db]);
      }
    }
    mma_commit(&ms->done);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&ms->done, 0) && globaltimer() - t0 < kWaitNs) {
    }
  }
  __syncwarp();
}

template <int HI, bool kList, int STRIDE, int TPC>
__device__ void epilogue_role(const Params &P, uint8_t *smem, Misc *ms, int q0, int y) {
  const CandView cv = cand_view(P, ms, smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sp = warp & 3, par = warp >> 2;
  const uint32_t tmem = ms->tmem_base;
  const uint32_t lane_addr = (uint32_t)(32 * sp) << 16;
  constexpr int LW = HI < 32 ? HI : 32;      // columns per TMEM load
  constexpr int NL = HI / LW;                // loads per query
  uint32_t it = 0;
  bool ok = true;
  // list mode in two halves: reserve() takes the warp's slots for a query
  // with one atomic whose result is only read by commit(), one round of
  // reductions later (the pending pair is carried across key tiles)
  struct Rsv {
    uint32_t m, base;
    int ql, s;
    float outv;
  };
  auto reserve = [&](int ql, int s, float acc, Rsv &r) {
    const bool in = s < ms->row_len[ql];
    r.ql = ql;
    r.s = s;
    r.outv = acc;
    r.base = 0u;
    r.m = __ballot_sync(0xffffffffu, in && acc >= ms->thr[ql]);
    if (r.m != 0u && lane == __ffs(r.m) - 1)
      r.base = atomicAdd(P.list_cnt + q0 + ql, (uint32_t)__popc(r.m));
  };
  auto commit = [&](const Rsv &r) {
    if (r.m == 0u) return;
    const uint32_t base = __shfl_sync(0xffffffffu, r.base, __ffs(r.m) - 1) +
                          __popc(r.m & ((1u << lane) - 1u));
    if (((r.m >> lane) & 1u) && base < (uint32_t)P.list_cap) {
      const int64_t o = (int64_t)(q0 + r.ql) * P.list_cap + base;
      P.list_ent[o] = r.s;
      P.list_val[o] = r.outv;
    }
  };
  Rsv p0, p1;
  bool pend0 = false, pend1 = false;
  for (int ri = 0; ri < ms->nruns && ok; ++ri) {
    const RunInfo ru = ms->runs[ri];
    const int64_t nt = walked_tiles<STRIDE>(ru.len);
    for (int64_t kt = (int64_t)y * TPC;
         kt < nt && kt < (int64_t)(y + 1) * TPC; ++kt, ++it) {
      const uint32_t db = it & 1;
      if (!(ok = wait_bar(&ms->d_full[db], (it >> 1) & 1, ms))) break;
      fence_after_sync();
      const int r = 32 * sp + lane;                       // key of the tile
      const int s = (int)kt * STRIDE * kKeyTile + r;      // its slot in the row
      const int col = (int)kt * kKeyTile + r;             // its column in `scores`
      // w . ReLU(D) over the HI head columns of query ql; store, or append to
      // the query's list (called by the whole warp: the append is
      // warp-aggregated, one counter update per warp)
      auto finish = [&](int ql, float acc) {
        const bool in = s < ms->row_len[ql];
        float outv = acc;
        if (in && P.cand) {
          const int64_t j = ru.gather ? cv.entry(ql, q0 + ql, s) : s;
          if (j >= ms->n_vis[ql]) outv = -INFINITY;
        }
        if constexpr (!kList) {
          if (in) P.scores[(int64_t)(q0 + ql) * P.out_ld + col] = outv;
          return;
        }
        const bool take = in && outv >= ms->thr[ql];
        const uint32_t m = __ballot_sync(0xffffffffu, take);
        if (m == 0u) return;
        const int leader = __ffs(m) - 1;
        uint32_t base = 0;
        if (lane == leader) base = atomicAdd(P.list_cnt + q0 + ql, (uint32_t)__popc(m));
        base = __shfl_sync(0xffffffffu, base, leader) + __popc(m & ((1u << lane) - 1u));
        if (take && base < (uint32_t)P.list_cap) {
          const int64_t o = (int64_t)(q0 + ql) * P.list_cap + base;
          P.list_ent[o] = s;
          P.list_val[o] = outv;
        }
      };
      // w * ReLU(x) as (w/2) * (x + |x|): the same value (halving and
      // doubling are exact), on the FMA pipe instead of a min/max on the ALU
      // pipe.  ms->w holds w/2.
      auto relu2 = [](uint32_t x) {
        const float f = __uint_as_float(x);
        return f + fabsf(f);
      };
      // four partial sums (heads h mod 4): independent FMA chains, two per
      // packed FP32x2 FMA
      auto dot = [&](int ql, int h0, const uint32_t *v, int n, float acc) {
        const float4 *w4 = reinterpret_cast<const float4 *>(ms->w + ql * HI + h0);
        float2 a01 = make_float2(acc, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
        for (int h = 0; h < n; h += 4) {
          const float4 wv = w4[h / 4];
          a01 = __ffma2_rn(make_float2(wv.x, wv.y), make_float2(relu2(v[h]), relu2(v[h + 1])),
                           a01);
          a23 = __ffma2_rn(make_float2(wv.z, wv.w),
                           make_float2(relu2(v[h + 2]), relu2(v[h + 3])), a23);
        }
        return (a01.x + a01.y) + (a23.x + a23.y);
      };
      if constexpr (HI == 32 && kList) {
        // as below, with the list appends of each round committed after the
        // next round's reductions (full mode: no candidate blocks)
        for (int qq = par; qq < ru.nq; qq += 4) {
          const bool two = qq + 2 < ru.nq;   // uniform across the warp
          uint32_t v0[32], v1[32];
          const uint32_t col = db * 256 + (uint32_t)(qq * HI);
          tmem_ld32x32b_x32(tmem + lane_addr + col, v0);
          if (two) tmem_ld32x32b_x32(tmem + lane_addr + col + 2 * HI, v1);
          tmem_wait_ld();
          const float a0 = dot(ru.ql0 + qq, 0, v0, 32, 0.f);
          const float a1 = two ? dot(ru.ql0 + qq + 2, 0, v1, 32, 0.f) : 0.f;
          if (pend0) commit(p0);
          if (pend1) commit(p1);
          reserve(ru.ql0 + qq, s, a0, p0);
          pend0 = true;
          pend1 = two;
          if (two) reserve(ru.ql0 + qq + 2, s, a1, p1);
        }
      } else if constexpr (HI == 32) {
        // two queries' columns in flight per TMEM wait
        for (int qq = par; qq < ru.nq; qq += 4) {
          const bool two = qq + 2 < ru.nq;   // uniform across the warp
          uint32_t v0[32], v1[32];
          const uint32_t col = db * 256 + (uint32_t)(qq * HI);
          tmem_ld32x32b_x32(tmem + lane_addr + col, v0);
          if (two) tmem_ld32x32b_x32(tmem + lane_addr + col + 2 * HI, v1);
          tmem_wait_ld();
          finish(ru.ql0 + qq, dot(ru.ql0 + qq, 0, v0, 32, 0.f));
          if (two) finish(ru.ql0 + qq + 2, dot(ru.ql0 + qq + 2, 0, v1, 32, 0.f));
        }
      } else {
        for (int qq = par; qq < ru.nq; qq += 2) {
          const int ql = ru.ql0 + qq;
          float acc = 0.f;
#pragma unroll
          for (int l = 0; l < NL; ++l) {
            uint32_t v[32];
            const uint32_t col = db * 256 + (uint32_t)(qq * HI + l * LW);
            if constexpr (LW == 32) {
              tmem_ld32x32b_x32(tmem + lane_addr + col, v);
            } else if constexpr (LW == 16) {
              tmem_ld32x32b_x16(tmem + lane_addr + col, v);
            } else {
              tmem_ld32x32b_x8(tmem + lane_addr + col, v);
            }
            tmem_wait_ld();
            acc = dot(ql, l * LW, v, LW, acc);
          }
          finish(ql, acc);
        }
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms->d_empty[db]);
    }
  }
  if (pend0) commit(p0);
  if (pend1) commit(p1);
}

// MODE 0: dense score rows; 1: sample (every kStreamStride-th key tile,
// stored densely); 2: appending lists
template <int HI, int MODE, int TPC>
__global__ void __launch_bounds__(kThreads, 1) index_score_tc_kernel(Params P) {
  constexpr int STRIDE = MODE == 1 ? kStreamStride : 1;
  constexpr bool kList = MODE == 2;
  extern __shared__ __align__(1024) uint8_t smem[];
  Misc *ms = reinterpret_cast<Misc *>(smem + kOffMisc);
  constexpr int QT = 256 / HI;
  // query tiles are taken in reverse order: in a causal batch the later
  // tiles have the longer rows, and starting those first keeps the last wave
  // of CTAs short
  const int q0 = (int)(gridDim.x - 1 - blockIdx.x) * QT;
  const int y = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  int err = 0;
  // ---- query operand loads first: they depend on nothing below, so they are
  // in flight while the tile geometry is worked out (rows past the tile read
  // query row 0 and are zeroed).  The epilogue and MMA warps build B; the
  // producer warps start on the key tiles as soon as the geometry is known.
  constexpr int kSetupThreads = kProdWarp0 * 32;
  constexpr int kBItems = (kBRows * 4 + kSetupThreads - 1) / kSetupThreads;
  uint4 bc[kBItems];
  float bsc[kBItems];
  uint32_t bvalid = 0;
  if (warp < kProdWarp0) {
#pragma unroll
    for (int k = 0; k < kBItems; ++k) {
      const int i = threadIdx.x + k * kSetupThreads;
      const int row = (i >> 2) % kBRows, grp = i & 3;
      const int ql = row / HI, h = row % HI;
      const int q = q0 + ql;
      const bool v = i < kBRows * 4 && ql < QT && q < P.b.num_q;
      bvalid |= (v ? 1u : 0u) << k;
      const int64_t base = v ? (int64_t)q * HI + h : 0;
      bc[k] = __ldg(reinterpret_cast<const uint4 *>(P.q_fp4 + base * 64) + grp);
      bsc[k] = __ldg(P.q_scale + base * 4 + grp);
    }
  }
  // ---- tile geometry -------------------------------------------------------
  // per query: visible entries and the row length seen by this key chunk.  In
  // pool mode only the candidate blocks overlapping this chunk's slots are
  // scanned: the first -1 among them ends the row (blocks are -1 padded at
  // the end), and the slots of the chunk map through an identity pool iff the
  // last present block of the range is its own index (blocks are strictly
  // ascending, so block i >= i, with equality all the way down)
  const int64_t s_lo = (int64_t)y * kKeyTile * TPC;
  const int64_t s_hi = s_lo + (int64_t)kKeyTile * TPC;
  int b_lo = 0, b_hi = 0;
  if (P.cand) {
    b_lo = (int)(s_lo / P.block);
    const int64_t bh = (s_hi + P.block - 1) / P.block;
    b_hi = (int)(bh < P.max_blocks ? bh : P.max_blocks);
    if (b_lo > b_hi) b_lo = b_hi;
  }
  if (threadIdx.x < QT) {
    ms->nb[threadIdx.x] = b_hi;
    ms->row_len[threadIdx.x] = 0;
    ms->n_vis[threadIdx.x] = 0;
  }
  if (threadIdx.x < QT)
    ms->thr[threadIdx.x] = (P.list_thr && q0 + (int)threadIdx.x < P.b.num_q)
                               ? P.list_thr[q0 + threadIdx.x] : 0.f;
  if (threadIdx.x == 0) {
    ms->abort = 0;
    ms->wait_ns = P.wait_ns;
    ms->cand_smem = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&ms->a_full[i], kProdWarps);
      mbar_init(&ms->a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->d_full[i], 1);
      mbar_init(&ms->d_empty[i], kEpiWarps);
    }
    mbar_init(&ms->done, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (P.cand) {
    const int span = b_hi - b_lo;
    const bool in_smem = QT * span <= kCandInts;
    int32_t *cand_s = reinterpret_cast<int32_t *>(smem + kOffCand);
    if (threadIdx.x == 0) {
      ms->cand_smem = in_smem ? 1 : 0;
      ms->cand_span = span;
      ms->b_lo = b_lo;
    }
    for (int i = threadIdx.x; i < QT * span; i += kThreads) {
      const int ql = i / span, bi = b_lo + i % span;
      const int q = q0 + ql;
      const int32_t v = q < P.b.num_q ? P.cand[(int64_t)q * P.max_blocks + bi] : -1;
      if (in_smem) cand_s[i] = v;
      if (q < P.b.num_q && v < 0) atomicMin(&ms->nb[ql], bi);
    }
    __syncthreads();
  }
  if (threadIdx.x < QT) {
    const int ql = threadIdx.x, q = q0 + ql;
    if (q < P.b.num_q) {
      const int r = P.b.q_req[q];
      const int64_t pos = P.b.q_pos[q];
      const int64_t kvl = P.b.kv_len[r];
      const int64_t kv0 = P.b.kv_start[r];
      int64_t nv = n_visible(pos, P.b.ratio);
      if (nv > kvl) {
        nv = kvl;
        if (y == 0) err |= CSA2_DERR_RANGE_CTX;
      }
      int64_t len = nv;
      int ident = 1;
      if (P.cand) {
        const int nb = ms->nb[ql];
        len = (int64_t)nb * P.block;
        if (len > s_hi) len = s_hi;
        ident = nb <= b_lo || P.cand[(int64_t)q * P.max_blocks + nb - 1] == nb - 1;
      }
      if (len > P.ld) {
        len = P.ld;
        if (P.cand || y == 0) err |= CSA2_DERR_LD;
      }
      ms->row_len[ql] = len;
      ms->n_vis[ql] = nv;
      ms->ident[ql] = ident;
      ms->req[ql] = r;
      ms->kv0[ql] = kv0;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // runs: consecutive queries of one request share key tiles (shared memory only)
    int nr = 0;
    for (int ql = 0; ql < QT; ++ql) {
      const int q = q0 + ql;
      if (q >= P.b.num_q) break;
      const int r = ms->req[ql];
      const int gather = P.cand && !ms->ident[ql];
      const int64_t len = ms->row_len[ql];
      const int64_t lim = len < ms->n_vis[ql] ? len : ms->n_vis[ql];
      if (!gather && nr > 0 && !ms->runs[nr - 1].gather && ms->runs[nr - 1].req == r) {
        RunInfo &ru = ms->runs[nr - 1];
        ru.nq += 1;
        if (len > ru.len) ru.len = len;
        if (lim > ru.lim) ru.lim = lim;
      } else {
        ms->runs[nr].kv0 = ms->kv0[ql];
        ms->runs[nr].ql0 = ql;
        ms->runs[nr].nq = 1;
        ms->runs[nr].req = r;
        ms->runs[nr].gather = gather;
        ms->runs[nr].len = len;
        ms->runs[nr].lim = lim;
        ++nr;
      }
    }
    ms->nruns = nr;
  }
  __syncthreads();
  // does this CTA's key chunk hold any work?
  bool any = false;
  for (int ri = 0; ri < ms->nruns; ++ri)
    any |= walked_tiles<STRIDE>(ms->runs[ri].len) > (int64_t)y * TPC;
  if (!any) {
    raise_err(P.d_err, err);
    return;
  }
  if (warp < kProdWarp0) {
    // ---- query operand B: (query, head) rows x 128 f16, and head weights ----
    uint8_t *B = smem + kOffB;
#pragma unroll
    for (int k = 0; k < kBItems; ++k) {
      const int i = threadIdx.x + k * kSetupThreads;
      if (i < kBRows * 4) {
        const int row = i >> 2, grp = i & 3;
        uint4 o[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                      make_uint4(0, 0, 0, 0)};
        if ((bvalid >> k) & 1u) {
          if (!mx_scale_ok(bsc[k]) && y == 0) err |= CSA2_DERR_SCALE;
          dequant32(bc[k], bsc[k], o);
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          *reinterpret_cast<uint4 *>(B + sw128_offset(row, grp * 32 + cc * 8, kBBlock)) = o[cc];
      }
    }
    for (int i = threadIdx.x; i < QT * HI; i += kSetupThreads) {
      const int q = q0 + i / HI;
      ms->w[i] = (q < P.b.num_q) ? 0.5f * (P.head_w ? P.head_w[(int64_t)q * HI + i % HI] : 1.f)
                                 : 0.f;
    }
    fence_proxy_async_smem();
    if (warp == kMmaWarp) {
      tmem_alloc(&ms->tmem_base, 512);
      tmem_relinquish();
    }
    // the epilogue and MMA warps wait for B, the weights and the TMEM base;
    // the producers are already on their way
    fence_before_sync();
    asm volatile("bar.sync 1, %0;" ::"n"(kSetupThreads) : "memory");
    fence_after_sync();
  }
  if (warp < kEpiWarps) {
    epilogue_role<HI, kList, STRIDE, TPC>(P, smem, ms, q0, y);
  } else if (warp == kMmaWarp) {
    mma_role<STRIDE, TPC>(P, smem, ms, y);
  } else {
    producer_role<STRIDE, TPC>(P, smem, ms, q0, y);
  }
  err = __reduce_or_sync(0xffffffffu, err);
  if ((threadIdx.x & 31) == 0) raise_err(P.d_err, err);
  fence_before_sync();
  __syncthreads();
  if (ms->abort && threadIdx.x == 0) raise_err(P.d_err, kDerrTimeout);
  if (warp == kMmaWarp) {
    fence_after_sync();
    tmem_dealloc(ms->tmem_base, 512);
  }
}

}  // namespace

namespace {

int launch(Params &P, int n_heads, cudaStream_t st) {
  P.wait_ns = wait_limit_ns();
  int64_t max_len = P.cand ? (int64_t)P.max_blocks * P.block : P.ld;
  if (max_len > P.ld) max_len = P.ld;
  const int64_t tiles_walked = (((max_len + kKeyTile - 1) / kKeyTile) + P.stride - 1) / P.stride;
  P.tpc = P.cand ? kTilesPool : tiles_walked <= kTilesWhole ? kTilesWhole : kTilesFull;
  const int64_t chunks = (tiles_walked + P.tpc - 1) / P.tpc;
  if (chunks == 0) return CSA2_OK;
  if (chunks > 65535) return CSA2_ERR_UNSUPPORTED;
  const int64_t tiles = (P.b.num_q + P.qt - 1) / P.qt;
  dim3 grid((unsigned)tiles, (unsigned)chunks);
#define CSA2_GO(H, M, T)                                                                     \
  do {                                                                                       \
    cudaFuncSetAttribute(index_score_tc_kernel<H, M, T>,                                     \
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);      \
    index_score_tc_kernel<H, M, T><<<grid, kThreads, kSmemBytes, st>>>(P);                   \
  } while (0)
#define CSA2_LAUNCH(H)                                                                       \
  do {                                                                                       \
    if (P.list_cnt && P.tpc == kTilesWhole) CSA2_GO(H, 2, kTilesWhole);                      \
    else if (P.list_cnt) CSA2_GO(H, 2, kTilesFull);                                          \
    else if (P.stride != 1 && P.tpc == kTilesWhole) CSA2_GO(H, 1, kTilesWhole);              \
    else if (P.stride != 1) CSA2_GO(H, 1, kTilesFull);                                       \
    else if (P.cand) CSA2_GO(H, 0, kTilesPool);                                              \
    else if (P.tpc == kTilesWhole) CSA2_GO(H, 0, kTilesWhole);                               \
    else CSA2_GO(H, 0, kTilesFull);                                                          \
  } while (0)
  switch (n_heads) {
    case 8: CSA2_LAUNCH(8); break;
    case 16: CSA2_LAUNCH(16); break;
    case 32: CSA2_LAUNCH(32); break;
    case 64: CSA2_LAUNCH(64); break;
    default: return CSA2_ERR_UNSUPPORTED;
  }
#undef CSA2_LAUNCH
#undef CSA2_GO
  return launch_status();
}

bool base_params(Params &P, const Batch &b, int n_heads, const uint8_t *q_fp4,
                 const float *q_scale, const float *head_w, const uint8_t *k_fp4,
                 const float *k_scale, int64_t ld, int32_t *d_err) {
  if (((uintptr_t)q_fp4 | (uintptr_t)k_fp4) & 15u) return false;
  if (((uintptr_t)q_scale | (uintptr_t)k_scale) & 15u) return false;
  P = Params{};
  P.b = b;
  P.hi = n_heads;
  P.qt = 256 / n_heads;
  P.q_fp4 = q_fp4;
  P.q_scale = q_scale;
  P.head_w = head_w;
  P.k_fp4 = k_fp4;
  P.k_scale = k_scale;
  P.cand = nullptr;
  P.block = 1;
  P.max_blocks = 1;
  P.ld = ld;
  P.out_ld = ld;
  P.stride = 1;
  P.d_err = d_err;
  return true;
}

}  // namespace

int index_score_tc(const Batch &b, int n_heads, const uint8_t *q_fp4, const float *q_scale,
                   const float *head_w, const uint8_t *k_fp4, const float *k_scale,
                   const int32_t *cand_blocks, int block, int max_blocks, float *scores,
                   int64_t ld, int32_t *d_err, cudaStream_t st) {
  if (b.num_q == 0) return CSA2_OK;
  Params P;
  if (!base_params(P, b, n_heads, q_fp4, q_scale, head_w, k_fp4, k_scale, ld, d_err))
    return CSA2_ERR_UNSUPPORTED;
  P.cand = cand_blocks;
  P.block = block;
  P.max_blocks = max_blocks;
  P.scores = scores;
  return launch(P, n_heads, st);
}

int index_score_sample(const Batch &b, int n_heads, const uint8_t *q_fp4, const float *q_scale,
                       const float *head_w, const uint8_t *k_fp4, const float *k_scale,
                       int64_t max_len, int stride, float *sample, int64_t sample_ld,
                       int32_t *d_err, cudaStream_t st) {
  if (b.num_q == 0) return CSA2_OK;
  Params P;
  if (!base_params(P, b, n_heads, q_fp4, q_scale, head_w, k_fp4, k_scale, max_len, d_err))
    return CSA2_ERR_UNSUPPORTED;
  if (stride != kStreamStride) return CSA2_ERR_UNSUPPORTED;   // the sample kernel's stride
  P.stride = stride;
  P.scores = sample;
  P.out_ld = sample_ld;
  return launch(P, n_heads, st);
}

int index_score_list(const Batch &b, int n_heads, const uint8_t *q_fp4, const float *q_scale,
                     const float *head_w, const uint8_t *k_fp4, const float *k_scale,
                     int64_t max_len, const float *thr, uint32_t *cnt, int32_t *ent, float *val,
                     int cap, int32_t *d_err, cudaStream_t st) {
  if (b.num_q == 0) return CSA2_OK;
  Params P;
  if (!base_params(P, b, n_heads, q_fp4, q_scale, head_w, k_fp4, k_scale, max_len, d_err))
    return CSA2_ERR_UNSUPPORTED;
  P.list_thr = thr;
  P.list_cnt = cnt;
  P.list_ent = ent;
  P.list_val = val;
  P.list_cap = cap;
  return launch(P, n_heads, st);
}

}  // namespace csa2

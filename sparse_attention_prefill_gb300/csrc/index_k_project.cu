// NEXT-2b: index keys projected from the compressed main KV and written as
// MXFP4 cache rows, in one kernel ("DeepSeek V4.1 Flash 建模", CSA2 card,
// compressor paragraph: index K is projected from the compressed main KV;
// SGLang/Miles day-0 article sec. 5: projection weights in BF16 with FP32
// accumulation, and a fused quantise/pack/cache write keeps the unfused
// rounding).
//
//   y[i, o] = sum_d x[i, d] W[o, d]     (x: [n, 512] bf16, W: [128, 512] bf16)
//   cache row dst_row[i] <- MXFP4(y[i, :])
//
// A CTA takes 128 source rows: D[i, o] (M = 128 rows, N = 128 outputs, K =
// 512) by tcgen05 kind::f16 with bf16 operands, fp32 accumulation in TMEM.
// The x and W blocks of 64 channels arrive by TMA (2-D tensor maps, 128-byte
// swizzle) into a 2-stage ring (three CTAs share an SM, so that the loads of
// one overlap the others' MMAs and encoding); one thread issues the loads,
// one the MMAs.
// Each of the 128 threads then owns one row: it reads its 128 fp32 values
// from TMEM and encodes them exactly as csa2_quantize_rows' MXFP4 format does
// (group scale 2^(floor(log2 amax) - 2) in fp32, x / scale in fp32, E2M1 round
// to nearest even with saturation at 6).  Waits are bounded (the library's
// wait limit); on expiry the kernel raises CSA2_DERR_TIMEOUT, lets its copies
// and MMAs in flight land (at most two seconds), frees TMEM and returns.
#include "common.cuh"
#include "kernels.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace csa2 {
namespace {

using namespace tc;

constexpr int kRows = 128;            // source rows per CTA (MMA M)
constexpr int kOut = 128;             // output channels (MMA N)
constexpr int kIn = 512;              // input channels (MMA K)
constexpr int kKBlock = 64;           // channels per TMA box (128 bytes of bf16)
constexpr int kKBlocks = kIn / kKBlock;
constexpr int kStages = 2;            // 64 KB of shared memory: three CTAs per SM
constexpr uint32_t kTile = kRows * 128;            // 16 KB per operand block
constexpr uint32_t kStage = 2 * kTile;             // x block + W block
constexpr uint32_t kOffBar = kStages * kStage;     // 64 KB
constexpr uint32_t kSmem = kOffBar + 256;
constexpr uint64_t kDrainNs = 2000000000ull;

struct Bars {
  uint64_t full[kStages], empty[kStages], done;
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, Bars *bs,
                                         uint64_t limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  while (!mbar_try_wait(bar, parity)) {
    if (*(volatile int *)&bs->abort) return false;
    if (gtimer() - t0 > limit) {
      atomicExch(&bs->abort, 1);
      return false;
    }
  }
  return true;
}

// wait (ignoring the abort flag, at most kDrainNs) for a phase to complete
__device__ __forceinline__ void drain_bar(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = gtimer();
  while (!mbar_try_wait(bar, parity) && gtimer() - t0 < kDrainNs) {
  }
}

struct Params {
  int64_t n;
  const int64_t *dst_row;
  uint8_t *codes;
  float *scales;
  int64_t rows;
  int32_t *d_err;
  uint64_t wait_ns;
};

// Warp 0 lane 0 issues the TMA loads, warp 1 lane 0 the MMAs, warp 2 owns the
// TMEM allocation; then all 128 threads encode one row each.
__global__ void __launch_bounds__(128, 1)
index_k_project_kernel(Params P, const __grid_constant__ CUtensorMap tmap_x,
                       const __grid_constant__ CUtensorMap tmap_w) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars *bs = reinterpret_cast<Bars *>(smem + kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row0 = (int64_t)blockIdx.x * kRows;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bs->full[s], 1);
      mbar_init(&bs->empty[s], 1);
    }
    mbar_init(&bs->done, 1);
    bs->abort = 0;
    mbar_fence_init();
  }
  if (warp == 2) {
    tmem_alloc(&bs->tmem, kOut);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = bs->tmem;
  if (warp == 0 && lane == 0) {
    int issued = 0;
    for (int kb = 0; kb < kKBlocks; ++kb) {
      const int s = kb % kStages;
      if (kb >= kStages &&
          !wait_bar(&bs->empty[s], ((kb / kStages) - 1) & 1, bs, P.wait_ns))
        break;
      uint8_t *st = smem + s * kStage;
      mbar_arrive_expect_tx(&bs->full[s], kStage);
      tma_load_2d(st, &tmap_x, kb * kKBlock, (int)row0, &bs->full[s]);
      tma_load_2d(st + kTile, &tmap_w, kb * kKBlock, 0, &bs->full[s]);
      ++issued;
    }
    // the copies of the stages not yet released must land before the CTA
    // exits (after an abort nobody else waits for them)
    for (int kb = issued > kStages ? issued - kStages : 0; kb < issued; ++kb)
      drain_bar(&bs->full[kb % kStages], (kb / kStages) & 1);
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = make_idesc_bf16(kRows, kOut);
    for (int kb = 0; kb < kKBlocks; ++kb) {
      const int s = kb % kStages;
      if (!wait_bar(&bs->full[s], (kb / kStages) & 1, bs, P.wait_ns)) break;
      fence_after_sync();
      const uint64_t da = make_desc_sw128(smem_u32(smem + s * kStage), 16, 1024);
      const uint64_t db = make_desc_sw128(smem_u32(smem + s * kStage + kTile), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < kKBlock / 16; ++kk)
        mma_f16(tmem, desc_add(da, kk * 32), desc_add(db, kk * 32), idesc,
                (kb > 0 || kk > 0) ? 1u : 0u);
      mma_commit(&bs->empty[s]);
    }
    mma_commit(&bs->done);   // completes once every MMA issued above has
  }
  __syncwarp();
  // every thread: the accumulator (bounded; the MMAs are always waited for,
  // since TMEM is freed below)
  drain_bar(&bs->done, 0);
  fence_after_sync();
  const bool aborted = *(volatile int *)&bs->abort != 0;
  int err = 0;
  const int64_t i = row0 + 32 * warp + lane;       // the row this thread encodes
  int64_t r = -1;
  if (!aborted && i < P.n) {
    r = P.dst_row[i];
    if (r >= P.rows) {
      err |= CSA2_DERR_RANGE_ROW;
      r = -1;
    }
  }
  const uint32_t lane_addr = (uint32_t)(32 * warp) << 16;
#pragma unroll 1
  for (int g = 0; g < kOut / 32 && !aborted; ++g) {
    uint32_t raw[32];
    tmem_ld32x32b_x32(tmem + lane_addr + 32 * g, raw);   // whole warp
    tmem_wait_ld();
    if (r < 0) continue;
    float v[32];
    float amax = 0.f;
    bool bad = false;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      v[k] = __uint_as_float(raw[k]);
      const float a = fabsf(v[k]);
      bad |= !(a <= 3.402823466e38f);   // NaN or infinity
      amax = fmaxf(amax, a);
    }
    float s = 1.0f;
    bool zero = bad;
    if (bad) {
      err |= CSA2_DERR_NONFINITE;
    } else if (amax > 0.0f) {
      int ex = 0;
      (void)frexpf(amax, &ex);
      s = ldexpf(1.0f, ex - 3);
      if (s == 0.0f || s < 0x1p-23f || s > 0x1p12f) err |= CSA2_DERR_SCALE;
      if (s == 0.0f) {
        s = 1.0f;
        zero = true;
      }
    }
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = zero ? 0.0f : v[k] / s;
    *reinterpret_cast<uint4 *>(P.codes + r * (kOut / 2) + 16 * g) =
        make_uint4(e2m1x8(v), e2m1x8(v + 8), e2m1x8(v + 16), e2m1x8(v + 24));
    P.scales[r * (kOut / 32) + g] = s;
  }
  err = __reduce_or_sync(0xffffffffu, err);
  if (lane == 0) raise_err(P.d_err, err);
  fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && bs->abort) raise_err(P.d_err, CSA2_DERR_TIMEOUT);
  if (warp == 2) {
    fence_after_sync();
    tmem_dealloc(tmem, kOut);
  }
}

// [rows, 512] bf16 as a 2-D map with 64 x 128 boxes in 128-byte swizzle (one
// box = one 64-channel block of a K-major SW128 operand tile)
bool make_map(CUtensorMap *map, const void *base, int64_t rows) {
  EncodeTiled fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kIn, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kIn * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kKBlock, (cuuint32_t)kRows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace csa2

extern "C" CSA2_API int csa2_index_k_project(int64_t n, const void *x_bf16, int32_t dim_in,
                                             const void *w_bf16, int32_t dim_out,
                                             const int64_t *dst_row, uint8_t *k_fp4,
                                             float *k_scale, int64_t rows, int32_t *d_err,
                                             csa2_stream_t stream) {
  if (n < 0 || rows < 0) return CSA2_ERR_INVALID_ARG;
  if (n > 0 && (!x_bf16 || !w_bf16 || !dst_row || !k_fp4 || !k_scale)) return CSA2_ERR_INVALID_ARG;
  if (dim_in != csa2::kIn || dim_out != csa2::kOut) return CSA2_ERR_UNSUPPORTED;
  if (n > 0x7fffffffll - csa2::kRows) return CSA2_ERR_UNSUPPORTED;
  if (n == 0) return CSA2_OK;
  if (((uintptr_t)x_bf16 | (uintptr_t)w_bf16 | (uintptr_t)k_fp4) & 15u ||
      ((uintptr_t)k_scale & 3u))
    return CSA2_ERR_UNSUPPORTED;
  CUtensorMap mx, mw;
  if (!csa2::make_map(&mx, x_bf16, n) || !csa2::make_map(&mw, w_bf16, csa2::kOut))
    return CSA2_ERR_UNSUPPORTED;
  csa2::Params P;
  P.n = n;
  P.dst_row = dst_row;
  P.codes = k_fp4;
  P.scales = k_scale;
  P.rows = rows;
  P.d_err = d_err;
  P.wait_ns = csa2::wait_limit_ns();
  const int grid = (int)((n + csa2::kRows - 1) / csa2::kRows);
  cudaFuncSetAttribute(csa2::index_k_project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)csa2::kSmem);
  csa2::index_k_project_kernel<<<grid, 128, csa2::kSmem, csa2::as_stream(stream)>>>(P, mx, mw);
  return csa2::launch_status();
}

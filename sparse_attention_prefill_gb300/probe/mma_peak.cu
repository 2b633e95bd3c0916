// Dense tensor-core throughput of one sm_103a GPU, measured with this
// library's own tcgen05 issue path (a measurement tool, not part of the layer).
//
// Every CTA (one per SM) holds one A tile (128 rows) and one B tile (256 rows)
// in shared memory, 128-byte K-major rows in the 128-byte swizzle, and one
// thread issues `iters` rounds of four M = 128, N = 256 MMAs over them into a
// TMEM accumulator (K = 16 / 32 / 64 per instruction for f16 / E4M3 / E2M1,
// i.e. 64 / 128 / 256 elements per round).  The operands never leave shared
// memory, so the rate is the tensor pipe's, not the memory system's.  With
// iters = 1 the accumulator is written out, so the host can check the
// products against its own (the kind's operand format and scale handling are
// exercised, not only its speed).  Block-scaled E2M1 (kind::mxf4) reads its
// UE8M0 scales from TMEM; every scale byte is set to 127 (= 1.0), which makes
// the result independent of how the scales are laid out there.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../csrc/tcgen05.cuh"

using namespace csa2::tc;

namespace {

constexpr int kM = 128, kN = 256;
constexpr uint32_t kATile = kM * 128;   // 16 KB
constexpr uint32_t kBTile = kN * 128;   // 32 KB
// more shared memory than the tiles need, so that no two CTAs share an SM
constexpr uint32_t kSmem = 120 * 1024;
constexpr uint64_t kWaitNs = 2000000000ull;

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// 16-byte chunk c of row r of a one-block SW128 tile
__device__ __forceinline__ uint32_t sw_off(uint32_t r, uint32_t c) {
  return (r >> 3) * 1024u + (r & 7u) * 128u + ((c ^ (r & 7u)) * 16u);
}

// kind: 0 = f16, 1 = E4M3 (kind::f8f6f4), 2 = E2M1 block-scaled (kind::mxf4)
__global__ void __launch_bounds__(128, 1)
mma_peak_kernel(int kind, int iters, const uint8_t *__restrict__ a, const uint8_t *__restrict__ b,
                float *__restrict__ d_out, int32_t *__restrict__ err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint32_t &tmem_base = *reinterpret_cast<uint32_t *>(smem + kATile + kBTile);
  uint64_t &bar = *reinterpret_cast<uint64_t *>(smem + kATile + kBTile + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t *A = smem, *B = smem + kATile;
  // rows of 128 bytes = 8 chunks of 16 bytes
  for (int i = threadIdx.x; i < kM * 8; i += blockDim.x)
    *reinterpret_cast<uint4 *>(A + sw_off(i >> 3, i & 7)) =
        reinterpret_cast<const uint4 *>(a)[i];
  for (int i = threadIdx.x; i < kN * 8; i += blockDim.x)
    *reinterpret_cast<uint4 *>(B + sw_off(i >> 3, i & 7)) =
        reinterpret_cast<const uint4 *>(b)[i];
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t lane_addr = (uint32_t)(32 * warp) << 16;
  if (kind == 2) {
    // scale factors: columns 256..511 of every lane hold UE8M0 127 (= 1.0)
    uint32_t ones[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) ones[j] = 0x7f7f7f7fu;
#pragma unroll
    for (int c = 256; c < 512; c += 32) tmem_st32x32b_x32(tmem + lane_addr + c, ones);
    tmem_wait_st();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (threadIdx.x == 0) {
    const uint64_t da = make_desc_sw128(smem_u32(A), 16, 1024);
    const uint64_t db = make_desc_sw128(smem_u32(B), 16, 1024);
    const uint32_t id16 = make_idesc_f16(kM, kN, false, false);
    const uint32_t id4 = make_idesc_mxf4(kM, kN, 0, 0);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
        const uint64_t ak = desc_add(da, kk * 32), bk = desc_add(db, kk * 32);
        if (kind == 0) mma_f16(tmem, ak, bk, id16, acc);
        else if (kind == 1) mma_f8f6f4(tmem, ak, bk, id16, acc);
        else mma_mxf4(tmem, ak, bk, id4, tmem + 256, tmem + 384, acc);
      }
    }
    mma_commit(&bar);
  }
  __syncwarp();
  // every thread waits for the MMAs (bounded)
  const uint64_t t0 = gtimer();
  bool ok = true;
  while (!mbar_try_wait(&bar, 0)) {
    if (gtimer() - t0 > kWaitNs) {
      ok = false;
      break;
    }
  }
  if (!ok && lane == 0) atomicOr(err, 1);
  fence_after_sync();
  if (ok && d_out && blockIdx.x == 0) {
    // row m = 32 * warp + lane, columns n
#pragma unroll 1
    for (int c = 0; c < kN; c += 32) {
      uint32_t v[32];
      tmem_ld32x32b_x32(tmem + lane_addr + c, v);
      tmem_wait_ld();
      for (int j = 0; j < 32; ++j)
        d_out[(int64_t)(32 * warp + lane) * kN + c + j] = __uint_as_float(v[j]);
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

// a: [128][128 bytes], b: [256][128 bytes] (K-major rows, device memory);
// d_out: [128][256] fp32 of CTA 0 or null; err: device int32, bit 0 set when a
// wait timed out.  Returns 0 on a successful launch.
extern "C" __attribute__((visibility("default"))) int csa2probe_mma(
    int kind, int iters, int ctas, const uint8_t *a, const uint8_t *b, float *d_out,
    int32_t *err, void *stream) {
  if (kind < 0 || kind > 2 || iters < 1 || ctas < 1 || !a || !b || !err) return 1;
  cudaFuncSetAttribute(mma_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  mma_peak_kernel<<<ctas, 128, kSmem, reinterpret_cast<cudaStream_t>(stream)>>>(kind, iters, a,
                                                                                  b, d_out, err);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

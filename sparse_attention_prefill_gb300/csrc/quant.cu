// Quantise-and-write of cache rows in the storage formats of the
// "DeepSeek V4.1 Flash 建模" mixed-precision card: main KV as FP8 E4M3 with an
// fp32 scale per 32 channels, or as E2M1 with an E4M3 scale per 16 channels
// (288 B per 512-channel entry); index keys as MXFP4 (E2M1, power-of-two fp32
// scale per 32).  SGLang/Miles day-0 article sec. 5: a fused quantise/pack/
// cache-write must keep the rounding and scaling sequence of the unfused
// computation.  The sequence here: the group scale in fp32 (amax / 448;
// E4M3(amax / 6); 2^(floor(log2 amax) - 2)), x / scale in fp32, then the
// hardware round-to-nearest-even conversion with saturation (cvt.rn.satfinite).
//
// One warp per source row (rows narrower than 512 channels share a warp), 16
// consecutive channels per lane and pass (a 32-channel group is a lane pair);
// rows go to dst_row[i] of the cache, so
// one launch writes the entries a step completes wherever they live.  HBM
// bound: 4 B read and 1.125 / 0.5625 B written per channel.
#include "common.cuh"

namespace csa2 {
namespace {

constexpr int kQThreads = 256;
constexpr int kQWarps = kQThreads / 32;

// 2 x fp32 -> 2 x E4M3 (x0 in the low byte), round to nearest even, saturating
__device__ __forceinline__ uint32_t e4m3x2(float x0, float x1) {
  uint32_t r;
  asm("{ .reg .b16 h;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h, %2, %1;\n\t"
      "cvt.u32.u16 %0, h; }"
      : "=r"(r) : "f"(x0), "f"(x1));
  return r;
}

// value of an E4M3 code (exact, through f16)
__device__ __forceinline__ float e4m3_to_float(uint32_t code) {
  uint32_t h;
  asm("{ .reg .b16 c; cvt.u16.u32 c, %1; cvt.rn.f16x2.e4m3x2 %0, c; }" : "=r"(h) : "r"(code));
  return __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
}

template <int kFmt>
__global__ void __launch_bounds__(kQThreads)
quantize_rows_kernel(int64_t n, const float *__restrict__ src, int dim,
                     const int64_t *__restrict__ dst_row, uint8_t *__restrict__ codes,
                     void *__restrict__ scales, int64_t rows, int32_t *__restrict__ d_err) {
  constexpr int kGroup = kFmt == CSA2_FMT_FP4KV ? 16 : 32;
  const int lane = threadIdx.x & 31;
  const int chunks = dim / 16;   // 16-channel chunks per row
  // narrow rows (a power-of-two count of chunks below 32) share a warp
  const int rpw = (chunks < 32 && (32 % chunks) == 0) ? 32 / chunks : 1;
  const int lpr = rpw > 1 ? chunks : 32;   // lanes per row
  const int sub = lane / lpr, cl = lane % lpr;
  const int passes = rpw > 1 ? 1 : (chunks + 31) / 32;
  int err = 0;
  for (int64_t base = ((int64_t)blockIdx.x * kQWarps + (threadIdx.x >> 5)) * rpw; base < n;
       base += (int64_t)gridDim.x * kQWarps * rpw) {
    const int64_t i = base + sub;
    const bool row_ok = i < n;
    const int64_t r = row_ok ? dst_row[i] : -1;
    const bool write = r >= 0 && r < rows;
    if (row_ok && r >= rows) err |= CSA2_DERR_RANGE_ROW;
    for (int p = 0; p < passes; ++p) {
      const int c = cl + 32 * p;   // chunk of 16 channels
      const bool has = write && c < chunks;
      float v[16];
      const float4 *s4 =
          reinterpret_cast<const float4 *>(src + (row_ok ? i : 0) * dim + 16 * (c < chunks ? c : 0));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 f = __ldcs(s4 + k);
        v[4 * k] = f.x;
        v[4 * k + 1] = f.y;
        v[4 * k + 2] = f.z;
        v[4 * k + 3] = f.w;
      }
      float amax = 0.f;
      bool bad = false;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float a = fabsf(v[k]);
        bad |= !(a <= 3.402823466e38f);   // NaN or infinity
        amax = fmaxf(amax, a);
      }
      if (kGroup == 32) {   // the lane pair (2j, 2j+1) holds one group
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        bad = __shfl_xor_sync(0xffffffffu, bad ? 1 : 0, 1) != 0 || bad;
      }
      if (!has) continue;
      float s = 1.0f;
      bool zero = bad;
      uint32_t sf = 0;
      if (bad) {
        err |= CSA2_DERR_NONFINITE;
      } else if (kFmt == CSA2_FMT_FP8_B32) {
        s = amax / 448.0f;
        if (s == 0.0f) s = 1.0f;
      } else if (kFmt == CSA2_FMT_FP4KV) {
        sf = e4m3x2(amax / 6.0f, 0.0f) & 0xffu;
        s = e4m3_to_float(sf);
        if (s == 0.0f) zero = true;
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
      float q[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) q[k] = zero ? 0.0f : v[k] / s;
      if (kFmt == CSA2_FMT_FP8_B32) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          w[k] = e4m3x2(q[4 * k], q[4 * k + 1]) | (e4m3x2(q[4 * k + 2], q[4 * k + 3]) << 16);
        *reinterpret_cast<uint4 *>(codes + r * dim + 16 * c) = make_uint4(w[0], w[1], w[2], w[3]);
        if ((c & 1) == 0) static_cast<float *>(scales)[r * (dim / 32) + c / 2] = s;
      } else {
        const uint2 w = make_uint2(e2m1x8(q), e2m1x8(q + 8));
        *reinterpret_cast<uint2 *>(codes + r * (dim / 2) + 8 * c) = w;
        if (kFmt == CSA2_FMT_FP4KV)
          static_cast<uint8_t *>(scales)[r * (dim / 16) + c] = bad ? 0 : (uint8_t)sf;
        else if ((c & 1) == 0)
          static_cast<float *>(scales)[r * (dim / 32) + c / 2] = s;
      }
    }
  }
  err = __reduce_or_sync(0xffffffffu, err);
  if (lane == 0) raise_err(d_err, err);
}

}  // namespace
}  // namespace csa2

extern "C" CSA2_API int csa2_quantize_rows(int32_t format, int64_t n, const float *src,
                                           int32_t dim, const int64_t *dst_row, uint8_t *codes,
                                           void *scales, int64_t rows, int32_t *d_err,
                                           csa2_stream_t stream) {
  if (n < 0 || rows < 0 || dim <= 0 || dim > 16384) return CSA2_ERR_INVALID_ARG;
  if (format != CSA2_FMT_FP8_B32 && format != CSA2_FMT_FP4KV && format != CSA2_FMT_MXFP4)
    return CSA2_ERR_INVALID_ARG;
  if (dim % (format == CSA2_FMT_FP4KV ? 16 : 32)) return CSA2_ERR_INVALID_ARG;
  if (n == 0) return CSA2_OK;
  if (!src || !dst_row || !codes || !scales) return CSA2_ERR_INVALID_ARG;
  // 16-byte source rows and code stores (8-byte for E2M1 codes)
  if (((uintptr_t)src & 15u) || ((uintptr_t)codes & (format == CSA2_FMT_FP8_B32 ? 15u : 7u)) ||
      ((uintptr_t)scales & 3u))
    return CSA2_ERR_UNSUPPORTED;
  const int chunks = dim / 16;
  const int64_t rpw = (chunks < 32 && (32 % chunks) == 0) ? 32 / chunks : 1;
  const int64_t want = (n + csa2::kQWarps * rpw - 1) / (csa2::kQWarps * rpw);
  const int64_t cap = (int64_t)csa2::sm_count() * (2048 / csa2::kQThreads);
  const int grid = (int)(want < cap ? want : cap);
  cudaStream_t st = csa2::as_stream(stream);
  switch (format) {
    case CSA2_FMT_FP8_B32:
      csa2::quantize_rows_kernel<CSA2_FMT_FP8_B32><<<grid, csa2::kQThreads, 0, st>>>(
          n, src, dim, dst_row, codes, scales, rows, d_err);
      break;
    case CSA2_FMT_FP4KV:
      csa2::quantize_rows_kernel<CSA2_FMT_FP4KV><<<grid, csa2::kQThreads, 0, st>>>(
          n, src, dim, dst_row, codes, scales, rows, d_err);
      break;
    default:
      csa2::quantize_rows_kernel<CSA2_FMT_MXFP4><<<grid, csa2::kQThreads, 0, st>>>(
          n, src, dim, dst_row, codes, scales, rows, d_err);
  }
  return csa2::launch_status();
}

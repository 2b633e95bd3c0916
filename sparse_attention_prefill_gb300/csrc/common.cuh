// Shared device helpers of libcsa2 (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/csa2.h"

namespace csa2 {

// ---------------------------------------------------------------------------
// host-side launch helpers
// ---------------------------------------------------------------------------
static inline cudaStream_t as_stream(csa2_stream_t s) {
  return reinterpret_cast<cudaStream_t>(s);
}

static inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

// SM count of the current device (cached per device; concurrent first calls
// store the same value); grids are sized by it.
static inline int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  int c = cached[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    c = n > 0 ? n : 1;
    cached[dev].store(c, std::memory_order_relaxed);
  }
  return c;
}

// Bound on the pipeline waits of the tensor-core kernels (ns of %globaltimer),
// read when a launch is issued; set by csa2_set_wait_limit_ns.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
inline std::atomic<uint64_t> &wait_limit_store() {
  static std::atomic<uint64_t> v{kDefaultWaitNs};
  return v;
}
static inline uint64_t wait_limit_ns() { return wait_limit_store().load(std::memory_order_relaxed); }

// ---------------------------------------------------------------------------
// batch view on the device (plain copy of the host struct's pointers)
// ---------------------------------------------------------------------------
struct Batch {
  int32_t num_q, num_req, ratio;
  const int32_t *q_req;
  const int64_t *q_pos;
  const int64_t *kv_start, *kv_len;
  const int64_t *swa_start, *swa_pos0, *swa_len;
};

static inline Batch to_device_view(const csa2_batch *b) {
  Batch v;
  v.num_q = b->num_q;
  v.num_req = b->num_req;
  v.ratio = b->ratio;
  v.q_req = b->q_req;
  v.q_pos = b->q_pos;
  v.kv_start = b->kv_start;
  v.kv_len = b->kv_len;
  v.swa_start = b->swa_start;
  v.swa_pos0 = b->swa_pos0;
  v.swa_len = b->swa_len;
  return v;
}

// Host-side checks common to every call taking a batch.
static inline bool batch_ok(const csa2_batch *b, bool need_swa) {
  if (!b || b->num_q < 0 || b->num_req < 0) return false;
  if (b->ratio != 1 && b->ratio != 2) return false;
  if (b->num_q > 0 && (!b->q_req || !b->q_pos || !b->kv_start || !b->kv_len)) return false;
  if (need_swa && b->num_q > 0 && (!b->swa_start || !b->swa_pos0 || !b->swa_len)) return false;
  return true;
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

// Compressed entries visible to absolute position t with non-overlapping
// groups of m tokens: entry j is complete once m*j + m - 1 <= t.
__device__ __forceinline__ int64_t n_visible(int64_t t, int m) {
  return t < 0 ? 0 : (t + 1) / m;
}

__device__ __forceinline__ void raise_err(int32_t *d_err, int bits) {
  if (d_err && bits) atomicOr(d_err, bits);
}

// E2M1 value of a 4-bit code (bit 3 sign, bits 2..1 exponent with bias 1,
// bit 0 mantissa; exponent 0 is subnormal), built directly as float bits.
__device__ __forceinline__ float e2m1_value(uint32_t nib) {
  const uint32_t m = nib & 7u;
  uint32_t bits = (m >= 2u) ? ((((m >> 1) + 126u) << 23) | ((m & 1u) << 22))
                            : (m ? 0x3F000000u : 0u);
  bits |= (nib & 8u) << 28;
  return __uint_as_float(bits);
}

// Two E4M3 codes (low byte first) -> float2, exact (hardware conversion).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
  __half2 h = *reinterpret_cast<__half2 *>(&h2);
  return __half22float2(h);
}

// Order-preserving map from float to uint32: larger float -> larger key.
// NaN maps below every number; -inf just above NaN; -0 and +0 share a key
// (they compare equal, so their order is the entry id's).
__device__ __forceinline__ uint32_t float_key(float f) {
  if (f != f) return 0u;
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// key of -inf: every eligible score has a strictly larger key
__device__ __forceinline__ uint32_t neg_inf_key() { return ~0xff800000u; }

// four bytes of E2M1 code pairs -> four f16x2 (byte b -> h[b]; low nibble in
// the low half); the bytes are taken apart by a vector move, not by shifts
__device__ __forceinline__ void e2m1x8_f16x8(uint32_t w, uint32_t (&h)[4]) {
  asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// 8 x fp32 -> 8 x E2M1 nibbles (element 2i in the low nibble of byte i),
// round to nearest even, saturating at +-6
__device__ __forceinline__ uint32_t e2m1x8(const float *x) {
  uint32_t r;
  asm("{ .reg .b8 t0, t1, t2, t3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
      "mov.b32 %0, {t0, t1, t2, t3}; }"
      : "=r"(r)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]));
  return r;
}

}  // namespace csa2

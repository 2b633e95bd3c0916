// a8-a10: sparse + sliding-window attention on CUDA cores (reference-grade
// kernel, fp32 throughout; attn_tc.cu holds the tensor-core fast path).
//
// For query q and head h, one softmax over the union of the selected
// compressed rows and the query's own window [max(win_lo, t-window+1, 0), t];
// the 512-dim latent row is both key and value (SGLang/Miles day-0 article
// sec. 1; "DeepSeek V4.1 Flash 建模" mixed-precision card; window lower bound:
// "SGLang 如何让 DeepSeek V4.1 Flash 的后半层只处理尾部 token" sec. 2.3).
//
// One CTA of 256 threads per query.  Q (fp32) lives in shared memory; every
// head is served by 256/H threads, each owning an interleaved 512*H/256-wide
// slice of the output accumulator in registers.  Rows are dequantised 16 at a
// time into shared memory; logits are reduced across a head's threads with
// warp shuffles and the softmax runs online.
#include "common.cuh"
#include "kernels.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 256;
constexpr int kDim = 512;
constexpr int kChunk = 16;
constexpr int kMaxRows = 2048 + 1024;

template <int H>
__global__ void __launch_bounds__(kThreads)
attn_simt_kernel(Batch b, const __nv_bfloat16 *__restrict__ qg, const uint8_t *__restrict__ kv_fp8,
                 const float *__restrict__ kv_scale, const int32_t *__restrict__ idx, int k,
                 const uint8_t *__restrict__ swa_fp8, const float *__restrict__ swa_scale,
                 const int64_t *__restrict__ win_lo, int window, float sm_scale,
                 const float *__restrict__ sink, __nv_bfloat16 *__restrict__ out,
                 float *__restrict__ lse, int32_t *__restrict__ d_err) {
  constexpr int TPH = kThreads / H;         // threads per head
  constexpr int V4 = kDim / 4 / TPH;        // float4 slots per thread
  extern __shared__ float4 smem4[];
  float4 *qs = smem4;                       // [H][128] float4
  float4 *rs = smem4 + H * (kDim / 4);      // [kChunk][128] float4
  __shared__ int64_t rows[kMaxRows];        // >= 0: KV pool row; < 0: -(SWA row) - 1
  __shared__ int nrows_s;
  const int q = blockIdx.x;
  const int r = b.q_req[q];
  const int64_t t = b.q_pos[q];
  const int64_t n_vis = n_visible(t, b.ratio);
  int err = 0;
  if (threadIdx.x == 0) nrows_s = 0;
  // Q -> shared fp32
  const __nv_bfloat162 *qp = reinterpret_cast<const __nv_bfloat162 *>(qg + (int64_t)q * H * kDim);
  float2 *qs2 = reinterpret_cast<float2 *>(qs);
  for (int i = threadIdx.x; i < H * kDim / 2; i += kThreads) qs2[i] = __bfloat1622float2(qp[i]);
  __syncthreads();
  // gather the row list: selected entries in idx order, then the window
  if (threadIdx.x == 0) {
    int n = 0;
    const int64_t kv0 = b.kv_start[r], kvn = b.kv_len[r];
    for (int i = 0; i < k && idx; ++i) {
      const int64_t j = idx[(int64_t)q * k + i];
      if (j < 0) continue;
      if (j >= n_vis || j >= kvn) {
        err |= CSA2_DERR_RANGE_IDX;
        continue;
      }
      rows[n++] = kv0 + j;
    }
    int64_t lo = t - window + 1;
    if (win_lo && win_lo[q] > lo) lo = win_lo[q];
    if (lo < 0) lo = 0;
    const int64_t p0 = b.swa_pos0[r], pn = b.swa_len[r], s0 = b.swa_start[r];
    for (int64_t p = lo; p <= t; ++p) {
      const int64_t off = p - p0;
      if (off < 0 || off >= pn) {
        err |= CSA2_DERR_RANGE_WINDOW;
        continue;
      }
      rows[n++] = -(s0 + off) - 1;
    }
    nrows_s = n;
  }
  __syncthreads();
  const int nrows = nrows_s;
  const int h = threadIdx.x / TPH, part = threadIdx.x % TPH;
  float4 o[V4];
#pragma unroll
  for (int i = 0; i < V4; ++i) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  float m = -INFINITY, l = 0.f;
  const float scale_log2 = sm_scale * 1.4426950408889634f;
  for (int c0 = 0; c0 < nrows; c0 += kChunk) {
    const int nc = min(kChunk, nrows - c0);
    __syncthreads();
    // dequantise nc rows: thread -> (row, 32 consecutive channels)
    {
      const int rr = threadIdx.x / 16, seg = threadIdx.x % 16;
      if (rr < nc) {
        const int64_t code = rows[c0 + rr];
        const uint8_t *src;
        float sc;
        if (code >= 0) {
          src = kv_fp8 + code * kDim;
          sc = kv_scale[code * (kDim / 32) + seg];
        } else {
          const int64_t sr = -code - 1;
          src = swa_fp8 + sr * kDim;
          sc = swa_scale[sr * (kDim / 32) + seg];
        }
        const uint4 *p = reinterpret_cast<const uint4 *>(src + seg * 32);
        const uint4 a = p[0], c = p[1];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
        float4 *dst = rs + rr * (kDim / 4) + seg * 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 lo2 = e4m3x2_to_float2((uint16_t)(w[i] & 0xffffu));
          const float2 hi2 = e4m3x2_to_float2((uint16_t)(w[i] >> 16));
          dst[i] = make_float4(lo2.x * sc, lo2.y * sc, hi2.x * sc, hi2.y * sc);
        }
      }
    }
    __syncthreads();
    float lg[kChunk];
    float cmax = -INFINITY;
#pragma unroll
    for (int rr = 0; rr < kChunk; ++rr) {
      float acc = 0.f;
      if (rr < nc) {
#pragma unroll
        for (int i = 0; i < V4; ++i) {
          const int v = part + i * TPH;
          const float4 a = qs[h * (kDim / 4) + v], c = rs[rr * (kDim / 4) + v];
          acc = fmaf(a.x, c.x, acc);
          acc = fmaf(a.y, c.y, acc);
          acc = fmaf(a.z, c.z, acc);
          acc = fmaf(a.w, c.w, acc);
        }
      }
#pragma unroll
      for (int off = TPH / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      lg[rr] = rr < nc ? acc * scale_log2 : -INFINITY;
      cmax = fmaxf(cmax, lg[rr]);
    }
    const float m_new = fmaxf(m, cmax);
    const float alpha = exp2f(m - m_new);
    l *= alpha;
#pragma unroll
    for (int i = 0; i < V4; ++i) {
      o[i].x *= alpha;
      o[i].y *= alpha;
      o[i].z *= alpha;
      o[i].w *= alpha;
    }
#pragma unroll
    for (int rr = 0; rr < kChunk; ++rr) {
      if (rr < nc) {
        const float p = exp2f(lg[rr] - m_new);
        l += p;
#pragma unroll
        for (int i = 0; i < V4; ++i) {
          const float4 c = rs[rr * (kDim / 4) + part + i * TPH];
          o[i].x = fmaf(p, c.x, o[i].x);
          o[i].y = fmaf(p, c.y, o[i].y);
          o[i].z = fmaf(p, c.z, o[i].z);
          o[i].w = fmaf(p, c.w, o[i].w);
        }
      }
    }
    m = m_new;
  }
  // sink: one more term e^{sink_h} in the denominator (natural-log units)
  float denom = l;
  float m_fin = m;
  if (sink) {
    const float sk = sink[h] * 1.4426950408889634f;
    const float mm = fmaxf(m, sk);
    denom = l * exp2f(m - mm) + exp2f(sk - mm);
    const float a = exp2f(m - mm);
#pragma unroll
    for (int i = 0; i < V4; ++i) {
      o[i].x *= a;
      o[i].y *= a;
      o[i].z *= a;
      o[i].w *= a;
    }
    m_fin = mm;
  }
  const float inv = denom > 0.f ? 1.f / denom : 0.f;
  __nv_bfloat162 *op = reinterpret_cast<__nv_bfloat162 *>(out + ((int64_t)q * H + h) * kDim);
#pragma unroll
  for (int i = 0; i < V4; ++i) {
    const int v = part + i * TPH;
    op[2 * v] = __floats2bfloat162_rn(o[i].x * inv, o[i].y * inv);
    op[2 * v + 1] = __floats2bfloat162_rn(o[i].z * inv, o[i].w * inv);
  }
  if (lse && part == 0)
    lse[(int64_t)q * H + h] = denom > 0.f ? (m_fin + log2f(denom)) * 0.6931471805599453f : -INFINITY;
  if (threadIdx.x == 0) raise_err(d_err, err);
}

}  // namespace

int attn_simt(const Batch &b, int n_heads, const __nv_bfloat16 *q, const uint8_t *kv_fp8,
              const float *kv_scale, const int32_t *idx, int k, const uint8_t *swa_fp8,
              const float *swa_scale, const int64_t *win_lo, int window, float sm_scale,
              const float *sink, __nv_bfloat16 *out, float *lse, int32_t *d_err,
              cudaStream_t st) {
  if (b.num_q == 0) return CSA2_OK;
  if (k + window > kMaxRows) return CSA2_ERR_UNSUPPORTED;
  const size_t smem = (size_t)(n_heads + kChunk) * kDim * sizeof(float);
#define CSA2_LAUNCH(HH)                                                                          \
  do {                                                                                           \
    cudaFuncSetAttribute(attn_simt_kernel<HH>, cudaFuncAttributeMaxDynamicSharedMemorySize,      \
                         (int)smem);                                                             \
    attn_simt_kernel<HH><<<b.num_q, kThreads, smem, st>>>(b, q, kv_fp8, kv_scale, idx, k,        \
                                                          swa_fp8, swa_scale, win_lo, window,    \
                                                          sm_scale, sink, out, lse, d_err);      \
  } while (0)
  switch (n_heads) {
    case 16: CSA2_LAUNCH(16); break;
    case 32: CSA2_LAUNCH(32); break;
    case 64: CSA2_LAUNCH(64); break;
    default: return CSA2_ERR_UNSUPPORTED;
  }
#undef CSA2_LAUNCH
  return launch_status();
}

}  // namespace csa2

// a2-a4, a7: index scores on CUDA cores (reference-grade kernel; the tensor-core
// kernel in index_score_tc.cu is the fast path where it applies).
//
//   s(q, j) = sum_h w[q,h] * max(0, <Qi[q,h], Ki[j]>)
//
// ("DeepSeek V4.1 Flash 建模", CSA2 and Hierarchical cards; SGLang/Miles day-0
// article sec. 5: MQA-shaped indexer over the shared FP4 keys.)
//
// Grid: (key tiles of 128, query rows).  The CTA decodes its query's Hi x 128
// MXFP4 operand into shared memory once; each thread owns one key (or pool
// slot), decodes it group by group and accumulates all Hi head dots in
// registers, then applies ReLU, the head weights and the head sum.
#include "common.cuh"
#include "kernels.cuh"

namespace csa2 {
namespace {

constexpr int kTile = 128;

__device__ __forceinline__ bool mx_scale_ok(float s) {
  const uint32_t u = __float_as_uint(s);
  const int e = (int)((u >> 23) & 0xff) - 127;
  return (u & 0x807fffffu) == 0 && e >= -23 && e <= 12;
}

template <int HI>
__global__ void __launch_bounds__(kTile)
index_score_simt_kernel(Batch b, const uint8_t *__restrict__ q_fp4,
                        const float *__restrict__ q_scale, const float *__restrict__ head_w,
                        const uint8_t *__restrict__ k_fp4, const float *__restrict__ k_scale,
                        const int32_t *__restrict__ cand_blocks, int block, int max_blocks,
                        float *__restrict__ scores, int64_t ld, int32_t *__restrict__ d_err) {
  __shared__ float qs[HI][128];
  __shared__ float ws[HI];
  __shared__ int nb_s;
  const int q = blockIdx.x;
  const int r = b.q_req[q];
  int err = 0;
  int64_t n_vis = n_visible(b.q_pos[q], b.ratio);
  const int64_t kv_len = b.kv_len[r];
  if (n_vis > kv_len) {
    n_vis = kv_len;
    if (blockIdx.y == 0 && threadIdx.x == 0) err |= CSA2_DERR_RANGE_CTX;
  }
  int64_t row_len;
  if (cand_blocks) {
    if (threadIdx.x == 0) {
      int n = 0;
      const int32_t *cb = cand_blocks + (int64_t)q * max_blocks;
      while (n < max_blocks && cb[n] >= 0) ++n;
      nb_s = n;
    }
    __syncthreads();
    row_len = (int64_t)nb_s * block;
  } else {
    row_len = n_vis;
  }
  if (row_len > ld) {
    row_len = ld;
    if (blockIdx.y == 0 && threadIdx.x == 0) err |= CSA2_DERR_LD;
  }
  const int64_t s0 = (int64_t)blockIdx.y * kTile;
  if (s0 >= row_len) {
    raise_err(d_err, err);
    return;
  }
  // decode the query's index operand
  for (int i = threadIdx.x; i < HI * 64; i += kTile) {
    const int h = i / 64, byte = i % 64;
    const uint8_t c = q_fp4[((int64_t)q * HI + h) * 64 + byte];
    const float sc = q_scale[((int64_t)q * HI + h) * 4 + byte / 16];
    if (byte % 16 == 0 && !mx_scale_ok(sc)) err |= CSA2_DERR_SCALE;
    qs[h][2 * byte] = e2m1_value(c & 15u) * sc;
    qs[h][2 * byte + 1] = e2m1_value(c >> 4) * sc;
  }
  for (int h = threadIdx.x; h < HI; h += kTile)
    ws[h] = head_w ? head_w[(int64_t)q * HI + h] : 1.0f;
  __syncthreads();
  const int64_t s = s0 + threadIdx.x;
  if (s < row_len) {
    int64_t j = s;
    bool visible = true;
    if (cand_blocks) {
      const int64_t blk = cand_blocks[(int64_t)q * max_blocks + s / block];
      j = blk * block + s % block;
      visible = j < n_vis;
    }
    float out = -INFINITY;
    if (visible) {
      const int64_t row = b.kv_start[r] + j;
      const uint4 *kp = reinterpret_cast<const uint4 *>(k_fp4 + row * 64);
      float acc[HI];
#pragma unroll
      for (int h = 0; h < HI; ++h) acc[h] = 0.f;
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        const uint4 w4 = kp[g];
        const float sc = k_scale[row * 4 + g];
        if (!mx_scale_ok(sc)) err |= CSA2_DERR_SCALE;
        const uint32_t words[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
          for (int nib = 0; nib < 8; ++nib) {
            const int d = g * 32 + wi * 8 + nib;
            const float kv = e2m1_value((words[wi] >> (4 * nib)) & 15u) * sc;
#pragma unroll
            for (int h = 0; h < HI; ++h) acc[h] = fmaf(qs[h][d], kv, acc[h]);
          }
        }
      }
      float tot = 0.f;
#pragma unroll
      for (int h = 0; h < HI; ++h) tot = fmaf(ws[h], fmaxf(acc[h], 0.f), tot);
      out = tot;
    }
    scores[(int64_t)q * ld + s] = out;
  }
  err = __reduce_or_sync(0xffffffffu, err);
  if ((threadIdx.x & 31) == 0) raise_err(d_err, err);
}

}  // namespace

int index_score_simt(const Batch &b, int n_heads, const uint8_t *q_fp4, const float *q_scale,
                     const float *head_w, const uint8_t *k_fp4, const float *k_scale,
                     const int32_t *cand_blocks, int block, int max_blocks, float *scores,
                     int64_t ld, int32_t *d_err, cudaStream_t st) {
  int64_t max_len = cand_blocks ? (int64_t)max_blocks * block : ld;
  if (max_len > ld) max_len = ld;
  const int64_t tiles = (max_len + kTile - 1) / kTile;
  if (tiles == 0 || b.num_q == 0) return CSA2_OK;
  if (tiles > 65535) return CSA2_ERR_UNSUPPORTED;
  dim3 grid((unsigned)b.num_q, (unsigned)tiles);
#define CSA2_LAUNCH(H)                                                                        \
  index_score_simt_kernel<H><<<grid, kTile, 0, st>>>(b, q_fp4, q_scale, head_w, k_fp4,      \
                                                     k_scale, cand_blocks, block, max_blocks, \
                                                     scores, ld, d_err)
  switch (n_heads) {
    case 8: CSA2_LAUNCH(8); break;
    case 16: CSA2_LAUNCH(16); break;
    case 32: CSA2_LAUNCH(32); break;
    case 64: CSA2_LAUNCH(64); break;
    default: return CSA2_ERR_UNSUPPORTED;
  }
#undef CSA2_LAUNCH
  return launch_status();
}

}  // namespace csa2

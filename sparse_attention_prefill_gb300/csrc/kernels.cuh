// Internal launchers of libcsa2 (host functions; one per kernel family).
#pragma once
#include "common.cuh"

namespace csa2 {

int index_score_tc(const Batch &b, int n_heads, const uint8_t *q_fp4, const float *q_scale,
                   const float *head_w, const uint8_t *k_fp4, const float *k_scale,
                   const int32_t *cand_blocks, int block, int max_blocks, float *scores,
                   int64_t ld, int32_t *d_err, cudaStream_t st);

// Streamed index score -> top-K: views into the caller's workspace.
struct StreamWs {
  uint32_t *hdr;        // [0] rows queued for the fallback, [1] next queued row to take
  float *thr;           // [Nq] per-query threshold
  uint32_t *cnt;        // [Nq] pairs offered to the query's list (may exceed the capacity)
  int32_t *fb_rows;     // [Nq] queued rows
  float *sample;        // [Nq, sample_ld] sampled scores
  int64_t sample_ld;
  int32_t *ent;         // [Nq, cap] listed entries
  float *val;           // [Nq, cap] listed scores
};
constexpr int kStreamListCap = 4096;   // listed pairs per query
constexpr int kStreamStride = 8;       // the sample pass scores every 8th key tile of 128

int index_score_sample(const Batch &b, int n_heads, const uint8_t *q_fp4, const float *q_scale,
                       const float *head_w, const uint8_t *k_fp4, const float *k_scale,
                       int64_t max_len, int stride, float *sample, int64_t sample_ld,
                       int32_t *d_err, cudaStream_t st);
int index_score_list(const Batch &b, int n_heads, const uint8_t *q_fp4, const float *q_scale,
                     const float *head_w, const uint8_t *k_fp4, const float *k_scale,
                     int64_t max_len, const float *thr, uint32_t *cnt, int32_t *ent, float *val,
                     int cap, int32_t *d_err, cudaStream_t st);
int stream_threshold_launch(const Batch &b, int64_t max_len, int k, int stride,
                            const StreamWs &ws, cudaStream_t st);
int stream_select_launch(const Batch &b, int64_t max_len, int k, int n_heads,
                         const uint8_t *q_fp4, const float *q_scale, const float *head_w,
                         const uint8_t *k_fp4, const float *k_scale, const StreamWs &ws,
                         int32_t *idx, int32_t *count, cudaStream_t st);

int topk_launch(const Batch &b, const float *scores, int64_t ld, int k,
                const int32_t *cand_blocks, int block, int max_blocks, int32_t *idx,
                int32_t *count, int32_t *blocks_out, int32_t *nblocks_out, int32_t *d_err,
                cudaStream_t st);

// kv_sf == nullptr: selected rows are FP8 block-32 (kv_codes [Nkv,512] E4M3 +
// kv_scale fp32 [Nkv,16]); otherwise FP4 (kv_codes [Nkv,256] E2M1 pairs +
// kv_sf [Nkv,32] E4M3, one scale per 16 channels).  Window rows are FP8.
int attn_tc(const Batch &b, int n_heads, const __nv_bfloat16 *q, const uint8_t *kv_codes,
            const float *kv_scale, const uint8_t *kv_sf, const int32_t *idx, int k,
            const uint8_t *swa_fp8,
            const float *swa_scale, const int64_t *win_lo, int window, float sm_scale,
            const float *sink, __nv_bfloat16 *out, float *lse, int32_t *d_err,
            cudaStream_t st);

}  // namespace csa2

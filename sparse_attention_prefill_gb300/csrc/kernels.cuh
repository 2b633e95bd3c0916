// Internal launchers of libcsa2 (host functions; one per kernel family).
#pragma once
#include "common.cuh"

namespace csa2 {

int index_score_tc(const Batch &b, int n_heads, const uint8_t *q_fp4, const float *q_scale,
                   const float *head_w, const uint8_t *k_fp4, const float *k_scale,
                   const int32_t *cand_blocks, int block, int max_blocks, float *scores,
                   int64_t ld, int32_t *d_err, cudaStream_t st);

int topk_launch(const Batch &b, const float *scores, int64_t ld, int k,
                const int32_t *cand_blocks, int block, int max_blocks, int32_t *idx,
                int32_t *count, int32_t *blocks_out, int32_t *nblocks_out, int32_t *d_err,
                cudaStream_t st);

int attn_tc(const Batch &b, int n_heads, const __nv_bfloat16 *q, const uint8_t *kv_fp8,
            const float *kv_scale, const int32_t *idx, int k, const uint8_t *swa_fp8,
            const float *swa_scale, const int64_t *win_lo, int window, float sm_scale,
            const float *sink, __nv_bfloat16 *out, float *lse, int32_t *d_err,
            cudaStream_t st);

}  // namespace csa2

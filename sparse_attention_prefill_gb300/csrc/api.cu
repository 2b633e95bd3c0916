// extern "C" entry points of libcsa2: host-side argument checks, then dispatch
// to the kernels.  Everything on the data path runs on the GPU; nothing here
// reads device memory or synchronises the host.
#include "common.cuh"
#include "kernels.cuh"

extern "C" CSA2_API const char *csa2_status_string(int status) {
  switch (status) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument";
    case CSA2_ERR_UNSUPPORTED: return "unsupported configuration";
    case CSA2_ERR_CUDA: return "CUDA launch failure";
    case CSA2_ERR_TIMEOUT: return "timeout";
    case CSA2_ERR_TOO_LARGE: return "request exceeds the fixed scratch of the allocation-free call";
    default: return "unknown status";
  }
}

extern "C" CSA2_API int csa2_set_wait_limit_ns(uint64_t ns) {
  csa2::wait_limit_store().store(ns ? ns : csa2::kDefaultWaitNs, std::memory_order_relaxed);
  return CSA2_OK;
}

extern "C" CSA2_API int csa2_index_score(const csa2_batch *b, int32_t n_heads, int32_t head_dim,
                                const uint8_t *q_fp4, const float *q_scale, const float *head_w,
                                const uint8_t *k_fp4, const float *k_scale,
                                const int32_t *cand_blocks, int32_t block, int32_t max_blocks,
                                float *scores, int64_t ld, int32_t *d_err, csa2_stream_t stream) {
  if (!csa2::batch_ok(b, false) || ld < 0) return CSA2_ERR_INVALID_ARG;
  if (b->num_q > 0 && (!q_fp4 || !q_scale || !k_fp4 || !k_scale || !scores))
    return CSA2_ERR_INVALID_ARG;
  if (cand_blocks && (block < 1 || max_blocks < 1)) return CSA2_ERR_INVALID_ARG;
  if (head_dim != 128) return CSA2_ERR_UNSUPPORTED;
  if (n_heads != 8 && n_heads != 16 && n_heads != 32 && n_heads != 64) return CSA2_ERR_UNSUPPORTED;
  if (cand_blocks && (block > 64 || max_blocks > 4096)) return CSA2_ERR_UNSUPPORTED;
  const csa2::Batch v = csa2::to_device_view(b);
  return csa2::index_score_tc(v, n_heads, q_fp4, q_scale, head_w, k_fp4, k_scale, cand_blocks,
                              block, max_blocks, scores, ld, d_err, csa2::as_stream(stream));
}

extern "C" CSA2_API int csa2_topk(const csa2_batch *b, const float *scores, int64_t ld, int32_t k,
                         const int32_t *cand_blocks, int32_t block, int32_t max_blocks,
                         int32_t *idx, int32_t *count, int32_t *d_err, csa2_stream_t stream) {
  if (!csa2::batch_ok(b, false) || ld < 0 || k < 1) return CSA2_ERR_INVALID_ARG;
  if (b->num_q > 0 && (!scores || !idx || !count)) return CSA2_ERR_INVALID_ARG;
  if (cand_blocks && (block < 1 || max_blocks < 1)) return CSA2_ERR_INVALID_ARG;
  if (k > 2048) return CSA2_ERR_UNSUPPORTED;
  if (cand_blocks && (block > 64 || max_blocks > 4096)) return CSA2_ERR_UNSUPPORTED;
  const csa2::Batch v = csa2::to_device_view(b);
  return csa2::topk_launch(v, scores, ld, k, cand_blocks, block, max_blocks, idx, count, nullptr,
                           nullptr, d_err, csa2::as_stream(stream));
}

extern "C" CSA2_API int csa2_topk_candidates(const csa2_batch *b, const float *scores, int64_t ld,
                                    int32_t k, int32_t block, int32_t max_blocks, int32_t *idx,
                                    int32_t *count, int32_t *blocks, int32_t *nblocks,
                                    int32_t *d_err, csa2_stream_t stream) {
  if (!csa2::batch_ok(b, false) || ld < 0 || k < 1 || block < 1 || max_blocks < 1)
    return CSA2_ERR_INVALID_ARG;
  if (b->num_q > 0 && (!scores || !idx || !count || !blocks || !nblocks))
    return CSA2_ERR_INVALID_ARG;
  if (k > 2048 || block > 64 || max_blocks > 4096) return CSA2_ERR_UNSUPPORTED;
  const csa2::Batch v = csa2::to_device_view(b);
  return csa2::topk_launch(v, scores, ld, k, nullptr, block, max_blocks, idx, count, blocks,
                           nblocks, d_err, csa2::as_stream(stream));
}

extern "C" CSA2_API int csa2_sparse_swa_attn(const csa2_batch *b, int32_t n_heads, int32_t dim,
                                    const void *q_bf16, const uint8_t *kv_fp8,
                                    const float *kv_scale, const int32_t *idx, int32_t k,
                                    const uint8_t *swa_fp8, const float *swa_scale,
                                    const int64_t *win_lo, int32_t window, float sm_scale,
                                    const float *sink, void *out_bf16, float *lse,
                                    int32_t *d_err, csa2_stream_t stream) {
  if (!csa2::batch_ok(b, true) || window < 1) return CSA2_ERR_INVALID_ARG;
  if (!idx) k = 0;
  if (k < 0) return CSA2_ERR_INVALID_ARG;
  if (b->num_q > 0 && (!q_bf16 || !swa_fp8 || !swa_scale || !out_bf16)) return CSA2_ERR_INVALID_ARG;
  if (b->num_q > 0 && k > 0 && (!kv_fp8 || !kv_scale)) return CSA2_ERR_INVALID_ARG;
  if (dim != 512) return CSA2_ERR_UNSUPPORTED;
  if (n_heads != 16 && n_heads != 32 && n_heads != 64) return CSA2_ERR_UNSUPPORTED;
  if (k > 2048 || window > 1024) return CSA2_ERR_UNSUPPORTED;
  const csa2::Batch v = csa2::to_device_view(b);
  return csa2::attn_tc(v, n_heads, reinterpret_cast<const __nv_bfloat16 *>(q_bf16), kv_fp8,
                         kv_scale, nullptr, idx, k, swa_fp8, swa_scale, win_lo, window, sm_scale,
                         sink, reinterpret_cast<__nv_bfloat16 *>(out_bf16), lse, d_err,
                         csa2::as_stream(stream));
}

extern "C" CSA2_API int csa2_sparse_swa_attn_fp4kv(
    const csa2_batch *b, int32_t n_heads, int32_t dim, const void *q_bf16, const uint8_t *kv_fp4,
    const uint8_t *kv_sf, const int32_t *idx, int32_t k, const uint8_t *swa_fp8,
    const float *swa_scale, const int64_t *win_lo, int32_t window, float sm_scale,
    const float *sink, void *out_bf16, float *lse, int32_t *d_err, csa2_stream_t stream) {
  if (!csa2::batch_ok(b, true) || window < 1) return CSA2_ERR_INVALID_ARG;
  if (!idx) k = 0;
  if (k < 0) return CSA2_ERR_INVALID_ARG;
  if (b->num_q > 0 && (!q_bf16 || !swa_fp8 || !swa_scale || !out_bf16)) return CSA2_ERR_INVALID_ARG;
  if (b->num_q > 0 && k > 0 && (!kv_fp4 || !kv_sf)) return CSA2_ERR_INVALID_ARG;
  if (dim != 512) return CSA2_ERR_UNSUPPORTED;
  if (n_heads != 16 && n_heads != 32 && n_heads != 64) return CSA2_ERR_UNSUPPORTED;
  if (k > 2048 || window > 1024) return CSA2_ERR_UNSUPPORTED;
  const csa2::Batch v = csa2::to_device_view(b);
  // a null scale pointer selects the FP8 pool, so with no selected rows any
  // readable byte stands in for it
  const uint8_t *sf = kv_sf ? kv_sf : swa_fp8;
  return csa2::attn_tc(v, n_heads, reinterpret_cast<const __nv_bfloat16 *>(q_bf16),
                       kv_fp4 ? kv_fp4 : swa_fp8, nullptr, sf, idx, k, swa_fp8, swa_scale,
                       win_lo, window, sm_scale, sink,
                       reinterpret_cast<__nv_bfloat16 *>(out_bf16), lse, d_err,
                       csa2::as_stream(stream));
}

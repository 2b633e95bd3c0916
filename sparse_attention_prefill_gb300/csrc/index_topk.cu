// Index score streamed into the top-K for full-visible rows (Full and
// Reindex layers scoring every visible entry): no score row is written; the
// scoring pass appends only the pairs at or above a per-query threshold to a
// bounded list, and the exact selection runs on that list ("DeepSeek V4.1
// Flash 建模", Hierarchical Sparse Indexer card: the data movement of the
// Top-K is a cost of its own).  Four steps on the caller's stream:
//   1. index score over every 8th key tile of 128 (the sample)
//   2. per-query threshold from the sample's moments
//   3. index score with the appending epilogue
//   4. exact selection from the lists; rows whose list misses (fewer than k
//      listed, or more than the capacity) are rescored on the CUDA cores by a
//      persistent fallback kernel with an exact running top-k
// The selected set is the same as csa2_index_score + csa2_topk's whenever the
// list holds the row's k best (the threshold is a guess; the fallback keeps
// the result exact when it misses).
#include "common.cuh"
#include "kernels.cuh"

namespace csa2 {

namespace {

constexpr int64_t kAlign = 256;

int64_t round_up(int64_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int64_t sample_ld_of(int64_t max_len) {
  const int64_t tiles = (max_len + 127) / 128;
  return (tiles + kStreamStride - 1) / kStreamStride * 128;
}

// Byte offsets of the workspace's arrays for num_q rows of at most max_len
// visible entries; returns the total size.  With base != nullptr the views
// are filled in.
int64_t layout(int64_t num_q, int64_t max_len, uint8_t *base, StreamWs *ws) {
  const int64_t sld = sample_ld_of(max_len);
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    const int64_t o = off;
    off += round_up(bytes);
    return o;
  };
  const int64_t o_hdr = take(8);
  const int64_t o_thr = take(num_q * 4);
  const int64_t o_cnt = take(num_q * 4);
  const int64_t o_fb = take(num_q * 4);
  const int64_t o_smp = take(num_q * sld * 4);
  const int64_t o_ent = take(num_q * kStreamListCap * 4);
  const int64_t o_val = take(num_q * kStreamListCap * 4);
  if (base && ws) {
    ws->hdr = reinterpret_cast<uint32_t *>(base + o_hdr);
    ws->thr = reinterpret_cast<float *>(base + o_thr);
    ws->cnt = reinterpret_cast<uint32_t *>(base + o_cnt);
    ws->fb_rows = reinterpret_cast<int32_t *>(base + o_fb);
    ws->sample = reinterpret_cast<float *>(base + o_smp);
    ws->sample_ld = sld;
    ws->ent = reinterpret_cast<int32_t *>(base + o_ent);
    ws->val = reinterpret_cast<float *>(base + o_val);
  }
  return off;
}

}  // namespace

int64_t index_topk_workspace_bytes(int64_t num_q, int64_t max_len) {
  return layout(num_q, max_len, nullptr, nullptr);
}

int index_topk(const Batch &b, int n_heads, const uint8_t *q_fp4, const float *q_scale,
               const float *head_w, const uint8_t *k_fp4, const float *k_scale,
               int64_t max_len, int k, int32_t *idx, int32_t *count, void *workspace,
               int64_t workspace_bytes, int32_t *d_err, cudaStream_t st) {
  if (b.num_q == 0) return CSA2_OK;
  if (workspace_bytes < index_topk_workspace_bytes(b.num_q, max_len))
    return CSA2_ERR_INVALID_ARG;
  if ((uintptr_t)workspace & (kAlign - 1)) return CSA2_ERR_UNSUPPORTED;
  StreamWs ws;
  layout(b.num_q, max_len, static_cast<uint8_t *>(workspace), &ws);
  int st1 = index_score_sample(b, n_heads, q_fp4, q_scale, head_w, k_fp4, k_scale, max_len,
                               kStreamStride, ws.sample, ws.sample_ld, d_err, st);
  if (st1 != CSA2_OK) return st1;
  st1 = stream_threshold_launch(b, max_len, k, kStreamStride, ws, st);
  if (st1 != CSA2_OK) return st1;
  st1 = index_score_list(b, n_heads, q_fp4, q_scale, head_w, k_fp4, k_scale, max_len, ws.thr,
                         ws.cnt, ws.ent, ws.val, kStreamListCap, d_err, st);
  if (st1 != CSA2_OK) return st1;
  return stream_select_launch(b, max_len, k, n_heads, q_fp4, q_scale, head_w, k_fp4, k_scale,
                              ws, idx, count, st);
}

}  // namespace csa2

extern "C" CSA2_API int csa2_index_topk_workspace(int32_t num_q, int64_t max_len,
                                                  int64_t *bytes) {
  if (num_q < 0 || max_len < 0 || !bytes) return CSA2_ERR_INVALID_ARG;
  *bytes = csa2::index_topk_workspace_bytes(num_q, max_len);
  return CSA2_OK;
}

extern "C" CSA2_API int csa2_index_topk(const csa2_batch *b, int32_t n_heads, int32_t head_dim,
                                        const uint8_t *q_fp4, const float *q_scale,
                                        const float *head_w, const uint8_t *k_fp4,
                                        const float *k_scale, int64_t max_len, int32_t k,
                                        int32_t *idx, int32_t *count, void *workspace,
                                        int64_t workspace_bytes, int32_t *d_err,
                                        csa2_stream_t stream) {
  if (!csa2::batch_ok(b, false) || max_len < 0 || k < 1) return CSA2_ERR_INVALID_ARG;
  if (b->num_q > 0 && (!q_fp4 || !q_scale || !k_fp4 || !k_scale || !idx || !count ||
                       !workspace))
    return CSA2_ERR_INVALID_ARG;
  if (head_dim != 128) return CSA2_ERR_UNSUPPORTED;
  if (n_heads != 8 && n_heads != 16 && n_heads != 32 && n_heads != 64)
    return CSA2_ERR_UNSUPPORTED;
  if (k > 2048) return CSA2_ERR_UNSUPPORTED;
  const csa2::Batch v = csa2::to_device_view(b);
  return csa2::index_topk(v, n_heads, q_fp4, q_scale, head_w, k_fp4, k_scale, max_len, k, idx,
                          count, workspace, workspace_bytes, d_err, csa2::as_stream(stream));
}

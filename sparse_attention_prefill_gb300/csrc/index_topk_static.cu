// csa2_index_topk_static: the streamed index score -> top-K of
// csa2_index_topk for callers that cannot allocate device memory, such as
// code running inside a CUDA graph capture, a custom allocator's own
// initialisation, or an embedding runtime that forbids cudaMalloc once it has
// started.  Their scratch lives in one fixed array of this file, reserved on
// every GPU that loads the library, instead of a caller-provided workspace.
//
// The pages have no counterpart to this call; it is a packaging variant of
// csa2_index_topk and runs exactly its kernels.
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace csa2 {

int64_t index_topk_workspace_bytes(int64_t num_q, int64_t max_len);
int index_topk(const Batch &b, int n_heads, const uint8_t *q_fp4, const float *q_scale,
               const float *head_w, const uint8_t *k_fp4, const float *k_scale,
               int64_t max_len, int k, int32_t *idx, int32_t *count, void *workspace,
               int64_t workspace_bytes, int32_t *d_err, cudaStream_t st);

namespace {

// 64 MiB: about 1600 queries of rows up to 16384 entries (40 KB each), or
// 2000 queries of rows up to 4096 entries
constexpr int64_t kStaticScratchBytes = 64ll << 20;

// The scratch itself.  In host code this name is only a stand-in for the
// device array: its device address is looked up per device below.
static __device__ __align__(256) uint8_t g_topk_scratch[kStaticScratchBytes];

std::mutex g_mu;
void *g_addr[64];   // device address of g_topk_scratch, per device (nullptr: not looked up)

// Device address of the scratch on the current device, looked up once per
// device with that device current.
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CSA2_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || !p) return CSA2_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return CSA2_OK;
}

}  // namespace
}  // namespace csa2

extern "C" CSA2_API int csa2_index_topk_static_capacity(int64_t *bytes) {
  if (!bytes) return CSA2_ERR_INVALID_ARG;
  *bytes = csa2::kStaticScratchBytes;
  return CSA2_OK;
}

extern "C" CSA2_API int csa2_index_topk_static(const csa2_batch *b, int32_t n_heads,
                                               int32_t head_dim, const uint8_t *q_fp4,
                                               const float *q_scale, const float *head_w,
                                               const uint8_t *k_fp4, const float *k_scale,
                                               int64_t max_len, int32_t k, int32_t *idx,
                                               int32_t *count, int32_t *d_err,
                                               csa2_stream_t stream) {
  if (!csa2::batch_ok(b, false) || max_len < 0 || k < 1) return CSA2_ERR_INVALID_ARG;
  if (b->num_q > 0 && (!q_fp4 || !q_scale || !k_fp4 || !k_scale || !idx || !count))
    return CSA2_ERR_INVALID_ARG;
  if (head_dim != 128) return CSA2_ERR_UNSUPPORTED;
  if (n_heads != 8 && n_heads != 16 && n_heads != 32 && n_heads != 64)
    return CSA2_ERR_UNSUPPORTED;
  if (k > 2048) return CSA2_ERR_UNSUPPORTED;
  if (csa2::index_topk_workspace_bytes(b->num_q, max_len) > csa2::kStaticScratchBytes)
    return CSA2_ERR_TOO_LARGE;
  if (b->num_q == 0) return CSA2_OK;
  void *scratch = nullptr;
  const int st = csa2::scratch_address(&scratch);
  if (st != CSA2_OK) return st;
  const csa2::Batch v = csa2::to_device_view(b);
  return csa2::index_topk(v, n_heads, q_fp4, q_scale, head_w, k_fp4, k_scale, max_len, k, idx,
                          count, scratch, csa2::kStaticScratchBytes, d_err,
                          csa2::as_stream(stream));
}

// noalloc.cu -- csa2_index_score_topk_reindex_noalloc: the Reindex mode of
// csa2_index_score_topk for callers that cannot hand the library any device memory beyond
// their inputs and outputs.  Its scratch (the fp32 score of every candidate slot) lives in the
// file-scope device array below, which every GPU that loads this library keeps until the
// process exits.
#include <mutex>

#include "common.cuh"

namespace csa2 {

// Scratch capacity in candidate slots: nq * n_cand_blocks * 8 must not exceed it (4 MiB).
constexpr int64_t kNoAllocSlots = (int64_t)1 << 20;

static __device__ __align__(256) float g_reindex_scratch[kNoAllocSlots];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
float *g_noalloc_ptr[kMaxDevices];  // device address of g_reindex_scratch, per device

// Device address of the scratch array on the current device.  The first call on a device looks
// it up with cudaGetSymbolAddress (host code cannot use the array's name as a device pointer).
cudaError_t noalloc_scratch(float **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_reindex_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<float *>(p);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}
}  // namespace

}  // namespace csa2

extern "C" int csa2_index_score_topk_reindex_noalloc(
    const void *q_idx, int q_dtype, const float *w, int nq, int Hi, int Di, const void *k_idx,
    int k_dtype, int64_t k_rows, const float *k_scale, const int64_t *cu_ctx, int B,
    const int32_t *q_seq, const int32_t *q_vis, int64_t max_vis, const int32_t *cand_blocks,
    int n_cand_blocks, int topk, int32_t *out_idx, void *stream) {
  using namespace csa2;
  // the same checks as csa2_index_score_topk in Reindex mode
  if (n_cand_blocks < 1) return CSA2_ERR_INVALID_ARG;
  if (int r = index_args_ok(q_idx, q_dtype, w, nq, Hi, Di, k_idx, k_dtype, k_rows, k_scale, cu_ctx,
                            B, q_seq, q_vis, max_vis, cand_blocks, n_cand_blocks, topk, out_idx,
                            nullptr, 0, nullptr))
    return r;
  if (nq == 0) return CSA2_OK;
  const int64_t slots = (int64_t)nq * n_cand_blocks * kBlock;
  if (slots > kNoAllocSlots) return CSA2_ERR_WORKSPACE;  // beyond the static scratch
  if (int r = check_device()) return r;
  float *scores = nullptr;
  if (noalloc_scratch(&scores) != cudaSuccess) return CSA2_ERR_CUDA;
  // Every slot the selection reads is written by the scoring kernel of the same call, so the
  // scratch needs no clearing between calls.  The selection runs without a workspace: for
  // pools over 2,048 blocks it takes the one-CTA-per-query path, which selects exactly the set
  // the workspace version's two-kernel path selects.
  return cuda_status(reindex_launch(q_idx, q_dtype, w, nq, Hi, Di, k_idx, k_rows, k_scale, cu_ctx,
                                    q_seq, q_vis, cand_blocks, n_cand_blocks, topk, out_idx,
                                    scores, nullptr, static_cast<cudaStream_t>(stream)));
}

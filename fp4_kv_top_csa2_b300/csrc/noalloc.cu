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
  if (nq < 0 || nq > 65535 || B < 1 || Hi < 1 || Hi > 16 || topk < 1 || topk > 4096 ||
      max_vis < 0 || max_vis > (int64_t)1 << 30 || k_rows < 0 || k_rows > INT32_MAX ||
      n_cand_blocks < 1 || n_cand_blocks > 65536)
    return CSA2_ERR_INVALID_ARG;
  if (q_dtype != k_dtype) return CSA2_ERR_INVALID_ARG;
  if (!((q_dtype == CSA2_BF16 && Di == 64) || (q_dtype == CSA2_E4M3 && Di == 128)))
    return CSA2_ERR_INVALID_ARG;
  if (nq == 0) return CSA2_OK;
  if (!q_idx || !w || !k_idx || !cu_ctx || !q_seq || !q_vis || !cand_blocks || !out_idx)
    return CSA2_ERR_INVALID_ARG;
  const void *ptrs[] = {q_idx, w, k_idx, k_scale, cu_ctx, q_seq, q_vis, cand_blocks, out_idx};
  for (const void *p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) & 15u) return CSA2_ERR_INVALID_ARG;
  const int64_t slots = (int64_t)nq * n_cand_blocks * kBlock;
  if (slots > kNoAllocSlots) return CSA2_ERR_WORKSPACE;  // beyond the static scratch
  {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return CSA2_ERR_CUDA;
    if (major != 10 || minor != 3) return CSA2_ERR_UNSUPPORTED;
  }
  float *scores = nullptr;
  if (noalloc_scratch(&scores) != cudaSuccess) return CSA2_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Every slot the selection reads is written by the scoring kernel of the same call, so the
  // scratch needs no clearing between calls.
  cudaError_t e = index_mma_supported(nq)
                      ? launch_score_cand_mma(q_idx, q_dtype, w, nq, Hi, k_idx, k_rows, k_scale,
                                              cu_ctx, q_seq, q_vis, cand_blocks, n_cand_blocks,
                                              scores, st)
                      : launch_score_cand(q_idx, q_dtype, w, nq, Hi, Di, k_idx, k_scale, cu_ctx,
                                          q_seq, q_vis, cand_blocks, n_cand_blocks, scores, st);
  if (e == cudaSuccess)
    e = launch_topk(scores, (int64_t)n_cand_blocks * kBlock, (int64_t)n_cand_blocks * kBlock,
                    cand_blocks, n_cand_blocks, 1, q_vis, nq, topk, out_idx, st);
  return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

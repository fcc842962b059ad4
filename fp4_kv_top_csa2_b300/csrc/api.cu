// api.cu -- the extern "C" entry points declared in include/csa2.h: host-side validation,
// workspace carving and kernel launches.  Nothing here allocates device memory.
#include <atomic>

#include "common.cuh"

using namespace csa2;

namespace {

constexpr size_t kWsAlign = 256;

size_t align_up(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device "is sm_103" cache: 0 unknown, 1 yes, 2 no.  Idempotent writes, so a benign race.
std::atomic<int> g_arch_ok[64];

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSA2_ERR_CUDA;
  if (dev < 0 || dev >= 64) return CSA2_ERR_UNSUPPORTED;
  int st = g_arch_ok[dev].load(std::memory_order_relaxed);
  if (st == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return CSA2_ERR_CUDA;
    st = (major == 10 && minor == 3) ? 1 : 2;
    g_arch_ok[dev].store(st, std::memory_order_relaxed);
  }
  return st == 1 ? CSA2_OK : CSA2_ERR_UNSUPPORTED;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA; }

struct WsCursor {
  char *p;
  size_t used = 0;
  explicit WsCursor(void *base) : p(static_cast<char *>(base)) {}
  template <class T>
  T *take(size_t count) {
    T *r = p ? reinterpret_cast<T *>(p + used) : nullptr;
    used += align_up(count * sizeof(T));
    return r;
  }
};

// Workspace layout of csa2_index_score_topk (also used to size it).
//   Reindex: scores of the candidate slots.
//   Full:    block maxima (unless the caller passes out_block_max, the region stays reserved),
//            the Top-K block list, and either the score of every visible position (tensor-core
//            path while that array stays small: the final selection reads it by position) or
//            the scores of the positions of the selected blocks (rescored).
constexpr int64_t kKeepScoresMax = (int64_t)1 << 27;  // elements (one-query-per-MMA scan)
// Chunked prefill (more than 1,024 queries, the 32-queries-per-MMA scan): keeping every score
// (4 B per visible pair, 4.4 GB at 4,096 x 266,240) costs one write pass instead of rescoring
// 16,384 candidates per query.
constexpr int64_t kKeepScoresMaxMulti = (int64_t)1 << 31;

struct ScoreWs {
  float *bm = nullptr;
  int32_t *blocks = nullptr;
  float *scores = nullptr;      // candidate-slot scores
  float *pos_scores = nullptr;  // per-position scores (Full, tensor-core path)
  void *topk = nullptr;         // scratch of the Top-K selections (shared: they run in turn)
  size_t bytes = 0;
  int64_t nb_max = 0;
  int kb = 0;         // blocks the Full selection needs: min(topk, blocks)
  bool pool_list = false;  // Full with a pool of >= kb blocks: the pool is the block list
  int nl = 0;         // length of the block list the positions are drawn from
};

ScoreWs score_ws(void *base, int nq, int64_t max_vis, int n_cand_blocks, int topk,
                 int n_pool = 0) {
  ScoreWs w;
  WsCursor c(base);
  if (n_cand_blocks > 0) {
    w.scores = c.take<float>((size_t)nq * n_cand_blocks * kBlock);
    w.topk = c.take<char>(topk_workspace_bytes(nq, (int64_t)n_cand_blocks * kBlock));
  } else {
    w.nb_max = (max_vis + kBlock - 1) / kBlock;
    w.kb = (int)std::min<int64_t>(topk, w.nb_max);
    w.pool_list = n_pool > 0 && n_pool >= w.kb;
    w.nl = w.pool_list ? n_pool : w.kb;
    w.bm = c.take<float>((size_t)nq * w.nb_max);
    if (!w.pool_list) w.blocks = c.take<int32_t>((size_t)nq * w.kb);
    const bool keep_mma = index_mma_supported(nq) && (int64_t)nq * max_vis <= kKeepScoresMax;
    const bool keep_multi = nq > kMaxScanQueries && (int64_t)nq * max_vis <= kKeepScoresMaxMulti;
    if (keep_mma || keep_multi) w.pos_scores = c.take<float>((size_t)nq * max_vis);
    // rescoring scratch: always when no score array is kept; with the prefill array too, for
    // calls that take the CUDA-core scan (several sequences, or not 8 indexer heads)
    if (!keep_mma) w.scores = c.take<float>((size_t)nq * w.nl * kBlock);
    w.topk = c.take<char>(std::max(topk_workspace_bytes(nq, w.nb_max),
                                   topk_workspace_bytes(nq, (int64_t)w.nl * kBlock)));
  }
  w.bytes = c.used;
  return w;
}

// Argument checks shared by every indexer entry point (with or without a workspace): ranges,
// dtype / Di pairs, the Reindex / Full / pool combinations, null and 16-byte alignment checks.
// CSA2_OK with nq == 0 means "nothing to enqueue".
int index_args_ok(const void *q_idx, int q_dtype, const float *w, int nq, int Hi, int Di,
                  const void *k_idx, int k_dtype, int64_t k_rows, const float *k_scale,
                  const int64_t *cu_ctx, int B, const int32_t *q_seq, const int32_t *q_vis,
                  int64_t max_vis, const int32_t *cand_blocks, int n_cand_blocks, int topk,
                  const int32_t *out_idx, const float *out_block_max, int n_pool,
                  const int32_t *out_pool) {
  if (nq < 0 || nq > 65535 || B < 1 || Hi < 1 || Hi > 16 || topk < 1 || topk > 4096 ||
      max_vis < 0 || max_vis > (int64_t)1 << 30 || k_rows < 0 || k_rows > INT32_MAX)
    return CSA2_ERR_INVALID_ARG;
  if (q_dtype != k_dtype) return CSA2_ERR_INVALID_ARG;
  if (!((q_dtype == CSA2_BF16 && Di == 64) || (q_dtype == CSA2_E4M3 && Di == 128)))
    return CSA2_ERR_INVALID_ARG;
  if (cand_blocks ? (n_cand_blocks < 1 || n_cand_blocks > 65536 || out_block_max)
                  : (n_cand_blocks != 0))
    return CSA2_ERR_INVALID_ARG;
  if (n_pool < 0 || n_pool > 4096 || (n_pool > 0 && cand_blocks)) return CSA2_ERR_INVALID_ARG;
  if (nq == 0) return CSA2_OK;
  if (!q_idx || !w || !k_idx || !cu_ctx || !q_seq || !q_vis || !out_idx ||
      (n_pool > 0 && !out_pool))
    return CSA2_ERR_INVALID_ARG;
  const void *ptrs[] = {q_idx, w, k_idx, k_scale, cu_ctx, q_seq, q_vis,
                        cand_blocks, out_idx, out_block_max, out_pool};
  for (const void *p : ptrs)
    if (!aligned16(p)) return CSA2_ERR_INVALID_ARG;
  return CSA2_OK;
}

// Reindex mode: score the listed blocks' positions into `scores` ([nq, n_cand_blocks * 8]),
// then select.  topk_ws may be null (the selection then takes its one-CTA-per-query path,
// which selects exactly the same set).  Shared by csa2_index_score_topk and the entry point
// without a workspace, so both score and select the same way.
cudaError_t reindex_launch(const void *q_idx, int q_dtype, const float *w, int nq, int Hi,
                           int Di, const void *k_idx, int64_t k_rows, const float *k_scale,
                           const int64_t *cu_ctx, const int32_t *q_seq, const int32_t *q_vis,
                           const int32_t *cand_blocks, int n_cand_blocks, int topk,
                           int32_t *out_idx, float *scores, void *topk_ws, cudaStream_t st) {
  cudaError_t e =
      cand_mma_supported()
          ? launch_score_cand_mma(q_idx, q_dtype, w, nq, Hi, k_idx, k_rows, k_scale, cu_ctx,
                                  q_seq, q_vis, cand_blocks, n_cand_blocks, scores, st)
          : launch_score_cand(q_idx, q_dtype, w, nq, Hi, Di, k_idx, k_scale, cu_ctx, q_seq,
                              q_vis, cand_blocks, n_cand_blocks, scores, st);
  if (e == cudaSuccess)
    e = launch_topk(scores, (int64_t)n_cand_blocks * kBlock, (int64_t)n_cand_blocks * kBlock,
                    cand_blocks, n_cand_blocks, 1, q_vis, nq, topk, out_idx, st, nullptr, 0,
                    topk_ws);
  return e;
}

// csa2_index_score_topk and csa2_index_score_topk_pool (n_pool > 0: Full mode with the pool).
int index_score_topk_impl(const void *q_idx, int q_dtype, const float *w, int nq, int Hi, int Di,
                          const void *k_idx, int k_dtype, int64_t k_rows, const float *k_scale,
                          const int64_t *cu_ctx, int B, const int32_t *q_seq,
                          const int32_t *q_vis, int64_t max_vis, const int32_t *cand_blocks,
                          int n_cand_blocks, int topk, int32_t *out_idx, float *out_block_max,
                          int n_pool, int32_t *out_pool, void *workspace, size_t ws_bytes,
                          void *stream, void *pool_event = nullptr) {
  if (int r = index_args_ok(q_idx, q_dtype, w, nq, Hi, Di, k_idx, k_dtype, k_rows, k_scale, cu_ctx,
                            B, q_seq, q_vis, max_vis, cand_blocks, n_cand_blocks, topk, out_idx,
                            out_block_max, n_pool, out_pool))
    return r;
  if (nq == 0)  // nothing to select; the (empty) pool is complete
    return pool_event ? cuda_status(cudaEventRecord(static_cast<cudaEvent_t>(pool_event),
                                                    static_cast<cudaStream_t>(stream)))
                      : CSA2_OK;
  if (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) return CSA2_ERR_INVALID_ARG;
  ScoreWs need = score_ws(nullptr, nq, max_vis, n_cand_blocks, topk, n_pool);
  if (ws_bytes < need.bytes || (need.bytes && !workspace)) return CSA2_ERR_WORKSPACE;
  if (int r = check_device()) return r;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ScoreWs ws = score_ws(workspace, nq, max_vis, n_cand_blocks, topk, n_pool);
  const bool mma = index_mma_supported(nq);
  const bool multi = !mma && index_multi_supported(nq, Hi, B);
  cudaError_t e;
  if (cand_blocks)  // Reindex: score the listed blocks, select
    return cuda_status(reindex_launch(q_idx, q_dtype, w, nq, Hi, Di, k_idx, k_rows, k_scale,
                                      cu_ctx, q_seq, q_vis, cand_blocks, n_cand_blocks, topk,
                                      out_idx, ws.scores, ws.topk, st));
  // Full: block maxima over every visible position; the Top-K positions lie inside the Top-K
  // blocks by block maximum (each block ahead of a selected position's block holds a position
  // ranked ahead of it), so select those blocks first, then select among their positions.  A
  // candidate pool of at least that many blocks (the top blocks by block maximum, the same
  // selection) serves as the block list itself.
  float *bm = out_block_max ? out_block_max : ws.bm;
  float *pos_scores = (mma || multi) ? ws.pos_scores : nullptr;  // written by the scan
  if (mma) {
    e = launch_score_scan_mma(q_idx, q_dtype, w, nq, Hi, k_idx, k_rows, k_scale, cu_ctx, q_seq,
                              q_vis, max_vis, bm, ws.nb_max, pos_scores, max_vis, st);
  } else if (multi) {  // chunked prefill over one sequence: 32 queries per key tile
    e = launch_score_scan_multi(q_idx, q_dtype, w, nq, k_idx, k_rows, k_scale, q_vis, max_vis,
                                bm, ws.nb_max, pos_scores, max_vis, st);
  } else {
    e = launch_score_scan(q_idx, q_dtype, w, nq, Hi, Di, k_idx, k_scale, cu_ctx, q_seq, q_vis,
                          max_vis, bm, ws.nb_max, st);
  }
  int32_t *list = ws.pool_list ? out_pool : ws.blocks;
  if (e == cudaSuccess)
    e = launch_topk(bm, ws.nb_max, ws.nb_max, nullptr, 0, kBlock, q_vis, nq, ws.nl, list, st,
                    nullptr, 0, ws.topk);
  if (e == cudaSuccess && n_pool > 0 && !ws.pool_list)  // a pool smaller than the block list
    e = launch_topk(bm, ws.nb_max, ws.nb_max, nullptr, 0, kBlock, q_vis, nq, n_pool, out_pool, st,
                    nullptr, 0, ws.topk);
  if (e == cudaSuccess && pool_event)  // the pool is complete: let its consumers start
    e = cudaEventRecord(static_cast<cudaEvent_t>(pool_event), st);
  if (pos_scores) {  // the scan kept every score: select among the blocks' positions
    if (e == cudaSuccess)
      e = launch_topk(nullptr, 0, (int64_t)ws.nl * kBlock, list, ws.nl, 1, q_vis, nq, topk,
                      out_idx, st, pos_scores, max_vis, ws.topk);
    return cuda_status(e);
  }
  if (e == cudaSuccess)
    e = (mma || multi) ? launch_score_cand_mma(q_idx, q_dtype, w, nq, Hi, k_idx, k_rows, k_scale,
                                               cu_ctx, q_seq, q_vis, list, ws.nl, ws.scores, st)
            : launch_score_cand(q_idx, q_dtype, w, nq, Hi, Di, k_idx, k_scale, cu_ctx, q_seq,
                                q_vis, list, ws.nl, ws.scores, st);
  if (e == cudaSuccess)
    e = launch_topk(ws.scores, (int64_t)ws.nl * kBlock, (int64_t)ws.nl * kBlock, list, ws.nl, 1,
                    q_vis, nq, topk, out_idx, st, nullptr, 0, ws.topk);
  return cuda_status(e);
}

}  // namespace

extern "C" {

const char *csa2_error_string(int status) {
  switch (status) {
    case CSA2_OK: return "CSA2_OK";
    case CSA2_ERR_INVALID_ARG: return "CSA2_ERR_INVALID_ARG: invalid argument";
    case CSA2_ERR_UNSUPPORTED: return "CSA2_ERR_UNSUPPORTED: device is not sm_103";
    case CSA2_ERR_CUDA: return "CSA2_ERR_CUDA: CUDA runtime or launch failure";
    case CSA2_ERR_WORKSPACE: return "CSA2_ERR_WORKSPACE: workspace too small";
    case CSA2_ERR_TIMEOUT: return "CSA2_ERR_TIMEOUT: bounded device wait expired";
    default: return "unknown CSA2 status";
  }
}

int csa2_kv_quant_fp4(const void *x_bf16, int64_t n_rows, int d, const int64_t *out_rows,
                      uint8_t *codes, uint8_t *sf, void *stream) {
  if (n_rows < 0 || d < 32 || d > 4096 || d % 32 != 0) return CSA2_ERR_INVALID_ARG;
  if (n_rows == 0) return CSA2_OK;
  if (!x_bf16 || !codes || !sf) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(codes) || !aligned16(sf) || !aligned16(out_rows))
    return CSA2_ERR_INVALID_ARG;
  if (int r = check_device()) return r;
  return cuda_status(launch_kv_quant(x_bf16, n_rows, d, out_rows, codes, sf,
                                     static_cast<cudaStream_t>(stream)));
}

size_t csa2_index_score_topk_workspace_size(int nq, int64_t max_vis, int n_cand_blocks,
                                            int topk) {
  if (nq < 0 || max_vis < 0 || n_cand_blocks < 0 || topk < 1) return 0;
  return score_ws(nullptr, nq, max_vis, n_cand_blocks, topk).bytes;
}

int csa2_index_score_topk(const void *q_idx, int q_dtype, const float *w, int nq, int Hi, int Di,
                          const void *k_idx, int k_dtype, int64_t k_rows, const float *k_scale,
                          const int64_t *cu_ctx, int B, const int32_t *q_seq,
                          const int32_t *q_vis, int64_t max_vis, const int32_t *cand_blocks,
                          int n_cand_blocks, int topk, int32_t *out_idx, float *out_block_max,
                          void *workspace, size_t ws_bytes, void *stream) {
  return index_score_topk_impl(q_idx, q_dtype, w, nq, Hi, Di, k_idx, k_dtype, k_rows, k_scale,
                               cu_ctx, B, q_seq, q_vis, max_vis, cand_blocks, n_cand_blocks, topk,
                               out_idx, out_block_max, 0, nullptr, workspace, ws_bytes, stream);
}

size_t csa2_index_score_topk_pool_workspace_size(int nq, int64_t max_vis, int topk,
                                                 int n_pool_blocks) {
  if (nq < 0 || max_vis < 0 || topk < 1 || n_pool_blocks < 1) return 0;
  return score_ws(nullptr, nq, max_vis, 0, topk, n_pool_blocks).bytes;
}

int csa2_index_score_topk_pool(const void *q_idx, int q_dtype, const float *w, int nq, int Hi,
                               int Di, const void *k_idx, int k_dtype, int64_t k_rows,
                               const float *k_scale, const int64_t *cu_ctx, int B,
                               const int32_t *q_seq, const int32_t *q_vis, int64_t max_vis,
                               int topk, int32_t *out_idx, float *out_block_max,
                               int block_size, int n_pool_blocks, int32_t *out_pool_blocks,
                               void *workspace, size_t ws_bytes, void *stream, void *pool_event) {
  if (block_size != kBlock || n_pool_blocks < 1) return CSA2_ERR_INVALID_ARG;
  return index_score_topk_impl(q_idx, q_dtype, w, nq, Hi, Di, k_idx, k_dtype, k_rows, k_scale,
                               cu_ctx, B, q_seq, q_vis, max_vis, nullptr, 0, topk, out_idx,
                               out_block_max, n_pool_blocks, out_pool_blocks, workspace, ws_bytes,
                               stream, pool_event);
}

int csa2_index_block_max(const void *q_idx, int q_dtype, const float *w, int nq, int Hi, int Di,
                         const void *k_idx, int k_dtype, int64_t k_rows, const float *k_scale,
                         const int64_t *cu_ctx, int B, const int32_t *q_seq, const int32_t *q_vis,
                         int64_t max_vis, float *out_block_max, void *stream) {
  // the Full-mode checks of csa2_index_score_topk; topk plays no part here (1), and the block
  // maxima, this call's only output, take the place of out_idx in the presence checks
  if (nq > 0 && !out_block_max) return CSA2_ERR_INVALID_ARG;
  if (int r = index_args_ok(q_idx, q_dtype, w, nq, Hi, Di, k_idx, k_dtype, k_rows, k_scale, cu_ctx,
                            B, q_seq, q_vis, max_vis, nullptr, 0, 1,
                            reinterpret_cast<const int32_t *>(out_block_max), out_block_max, 0,
                            nullptr))
    return r;
  if (nq == 0 || max_vis == 0) return CSA2_OK;
  if (int r = check_device()) return r;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t nb = (max_vis + kBlock - 1) / kBlock;
  cudaError_t e;
  if (index_mma_supported(nq))
    e = launch_score_scan_mma(q_idx, q_dtype, w, nq, Hi, k_idx, k_rows, k_scale, cu_ctx, q_seq,
                              q_vis, max_vis, out_block_max, nb, nullptr, 0, st);
  else if (index_multi_supported(nq, Hi, B))
    e = launch_score_scan_multi(q_idx, q_dtype, w, nq, k_idx, k_rows, k_scale, q_vis, max_vis,
                                out_block_max, nb, nullptr, 0, st);
  else
    e = launch_score_scan(q_idx, q_dtype, w, nq, Hi, Di, k_idx, k_scale, cu_ctx, q_seq, q_vis,
                          max_vis, out_block_max, nb, st);
  return cuda_status(e);
}

size_t csa2_hier_candidate_pool_workspace_size(int nq, int64_t max_blocks, int n_pool_blocks) {
  (void)n_pool_blocks;
  if (nq < 0 || max_blocks < 0) return 0;
  return align_up(topk_workspace_bytes(nq, max_blocks));
}

int csa2_hier_candidate_pool(const float *block_max, int nq, const int32_t *q_vis,
                             int64_t max_blocks, int block_size, int n_pool_blocks,
                             int32_t *out_pool_blocks, void *workspace, size_t ws_bytes,
                             void *stream) {
  if (nq < 0 || nq > 65535 || max_blocks < 0 || max_blocks > (int64_t)1 << 27 ||
      block_size != kBlock || n_pool_blocks < 1 || n_pool_blocks > 4096)
    return CSA2_ERR_INVALID_ARG;
  if (nq == 0) return CSA2_OK;
  if (!block_max || !q_vis || !out_pool_blocks) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(block_max) || !aligned16(q_vis) || !aligned16(out_pool_blocks))
    return CSA2_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) return CSA2_ERR_INVALID_ARG;
  const size_t need = csa2_hier_candidate_pool_workspace_size(nq, max_blocks, n_pool_blocks);
  if (ws_bytes < need || (need && !workspace)) return CSA2_ERR_WORKSPACE;
  if (int r = check_device()) return r;
  return cuda_status(launch_topk(block_max, max_blocks, max_blocks, nullptr, 0, block_size, q_vis,
                                 nq, n_pool_blocks, out_pool_blocks,
                                 static_cast<cudaStream_t>(stream), nullptr, 0,
                                 need ? workspace : nullptr));
}

size_t csa2_sparse_attn_decode_workspace_size(int B, int H, int topk) {
  if (B < 0 || H < 1 || topk < 1) return 0;
  return align_up(attn_mma_supported(H, topk) ? attn_mma_workspace_bytes(B, H, topk)
                                              : attn_workspace_bytes(B, H, topk));
}

static int attn_args_ok(int nq, int H, const uint8_t *codes, const uint8_t *sf,
                        const int64_t *cu_ctx, const int32_t *idx, int topk, float scale,
                        const void *q, const void *out, const float *lse, const void *ws) {
  if (nq < 0 || nq > 65535 || H < 1 || H > 128 || topk < 1 || topk > 16384 || !(scale > 0.0f))
    return CSA2_ERR_INVALID_ARG;
  if (nq == 0) return CSA2_OK;
  if (!q || !codes || !sf || !cu_ctx || !idx || !out) return CSA2_ERR_INVALID_ARG;
  const void *ptrs[] = {q, codes, sf, cu_ctx, idx, out, lse};
  for (const void *p : ptrs)
    if (!aligned16(p)) return CSA2_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) % kWsAlign) return CSA2_ERR_INVALID_ARG;
  return CSA2_OK;
}

int csa2_sparse_attn_decode(const void *q_bf16, int B, int H, const uint8_t *codes,
                            const uint8_t *sf, const int64_t *cu_ctx, const int32_t *idx, int topk,
                            float softmax_scale, void *out_bf16, float *lse, void *workspace,
                            size_t ws_bytes, void *stream) {
  if (int r = attn_args_ok(B, H, codes, sf, cu_ctx, idx, topk, softmax_scale, q_bf16, out_bf16,
                           lse, workspace))
    return r;
  if (B == 0) return CSA2_OK;
  const size_t need = csa2_sparse_attn_decode_workspace_size(B, H, topk);
  if (ws_bytes < need || (need && !workspace)) return CSA2_ERR_WORKSPACE;
  if (int r = check_device()) return r;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (attn_mma_supported(H, topk))
    return cuda_status(launch_attn_mma(q_bf16, B, H, codes, sf, cu_ctx, idx, topk, softmax_scale,
                                       out_bf16, lse, workspace, st));
  return cuda_status(launch_attn(q_bf16, nullptr, nullptr, B, H, nullptr, codes, sf, cu_ctx, idx,
                                 topk, softmax_scale, out_bf16, lse, workspace, st));
}

size_t csa2_sparse_attn_prefill_workspace_size(int T, int H, int topk) {
  if (T < 0 || H < 1 || topk < 1) return 0;
  if (attn_prefill_supported(H)) return 0;  // the tensor-core kernel quantises the query itself
  const size_t rows = (size_t)T * H;
  return align_up(rows * kCodeBytes) + align_up(rows * kSfBytes) +
         align_up(attn_workspace_bytes(T, H, topk));
}

int csa2_sparse_attn_prefill(const void *q_bf16, int T, int H, const int32_t *q_seq,
                             const uint8_t *codes, const uint8_t *sf, const int64_t *cu_ctx,
                             int B, const int32_t *idx, int topk, float softmax_scale,
                             void *out_bf16, float *lse, void *workspace, size_t ws_bytes,
                             void *stream) {
  if (int r = attn_args_ok(T, H, codes, sf, cu_ctx, idx, topk, softmax_scale, q_bf16, out_bf16,
                           lse, workspace))
    return r;
  if (B < 1) return CSA2_ERR_INVALID_ARG;
  if (T == 0) return CSA2_OK;
  if (!q_seq || !aligned16(q_seq)) return CSA2_ERR_INVALID_ARG;
  const size_t need = csa2_sparse_attn_prefill_workspace_size(T, H, topk);
  if (ws_bytes < need || (need && !workspace)) return CSA2_ERR_WORKSPACE;
  if (int r = check_device()) return r;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the query is quantised per (token, head) row with the main-KV FP4 rule: inside the
  // tensor-core kernel, or by the quantisation kernel ahead of the CUDA-core one
  if (attn_prefill_supported(H))
    return cuda_status(launch_attn_prefill(q_bf16, T, H, q_seq, codes, sf, cu_ctx, idx, topk,
                                           softmax_scale, out_bf16, lse, st));
  WsCursor c(workspace);
  const size_t rows = (size_t)T * H;
  uint8_t *q_codes = c.take<uint8_t>(rows * kCodeBytes);
  uint8_t *q_sf = c.take<uint8_t>(rows * kSfBytes);
  void *attn_ws = c.take<char>(attn_workspace_bytes(T, H, topk));
  cudaError_t e = launch_kv_quant(q_bf16, (int64_t)rows, kD, nullptr, q_codes, q_sf, st);
  if (e == cudaSuccess)
    e = launch_attn(nullptr, q_codes, q_sf, T, H, q_seq, codes, sf, cu_ctx, idx, topk,
                    softmax_scale, out_bf16, lse, attn_ws, st);
  return cuda_status(e);
}

// ---- the full-FP4 PV variant of prefill attention -----------------------------------------

int csa2_sparse_attn_prefill_fp4pv(const void *q_bf16, int T, int H, const int32_t *q_seq,
                                   const uint8_t *codes, const uint8_t *sf, const int64_t *cu_ctx,
                                   int B, const int32_t *idx, int topk, float softmax_scale,
                                   void *out_bf16, float *lse, void *stream) {
  if (int r = attn_args_ok(T, H, codes, sf, cu_ctx, idx, topk, softmax_scale, q_bf16, out_bf16,
                           lse, nullptr))
    return r;
  if (B < 1) return CSA2_ERR_INVALID_ARG;
  if (T == 0) return CSA2_OK;
  if (!q_seq || !aligned16(q_seq)) return CSA2_ERR_INVALID_ARG;
  if (!attn_prefill_supported(H)) return CSA2_ERR_UNSUPPORTED;
  if (int r = check_device()) return r;
  return cuda_status(launch_attn_fp4pv(q_bf16, T, H, q_seq, codes, sf, cu_ctx, idx, topk,
                                       softmax_scale, out_bf16, lse,
                                       static_cast<cudaStream_t>(stream)));
}

// ---- index keys derived from main-KV rows -------------------------------------------------

int csa2_index_keys_from_kv(const uint8_t *codes, const uint8_t *sf, int64_t n_rows,
                            const int64_t *rows, const void *w_bf16, int Di, uint8_t *k_idx,
                            float *k_scale, void *stream) {
  if (n_rows < 0 || n_rows > ((int64_t)1 << 31) || Di != 128) return CSA2_ERR_INVALID_ARG;
  if (n_rows == 0) return CSA2_OK;
  if (!codes || !sf || !w_bf16 || !k_idx || !k_scale) return CSA2_ERR_INVALID_ARG;
  const void *ptrs[] = {codes, sf, rows, w_bf16, k_idx, k_scale};
  for (const void *p : ptrs)
    if (!aligned16(p)) return CSA2_ERR_INVALID_ARG;
  if (int r = check_device()) return r;
  if (!index_keys_supported()) return CSA2_ERR_UNSUPPORTED;
  return cuda_status(launch_index_keys(codes, sf, n_rows, rows, w_bf16, k_idx, k_scale,
                                       static_cast<cudaStream_t>(stream)));
}

// ---- the local sliding-window branch ------------------------------------------------------

int csa2_swa_kv_quant_fp8(const void *x_bf16, int64_t n_rows, int d, const int64_t *out_rows,
                          uint8_t *swa_kv, void *stream) {
  if (n_rows < 0 || d < 16 || d > 4096 || d % 16 != 0) return CSA2_ERR_INVALID_ARG;
  if (n_rows == 0) return CSA2_OK;
  if (!x_bf16 || !swa_kv) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(swa_kv) || !aligned16(out_rows))
    return CSA2_ERR_INVALID_ARG;
  if (int r = check_device()) return r;
  return cuda_status(launch_fp8_quant(x_bf16, n_rows, d, out_rows, swa_kv,
                                      static_cast<cudaStream_t>(stream)));
}

// The window's extra checks: 0 <= n_win <= ring, a ring buffer when there is a window, and the
// tensor-core kernels (H <= 64).
static int swa_args_ok(int H, const uint8_t *swa_kv, int ring, int n_win) {
  if (n_win < 0 || n_win > 8192 || ring < 1 || n_win > ring) return CSA2_ERR_INVALID_ARG;
  if (n_win > 0 && (!swa_kv || !aligned16(swa_kv))) return CSA2_ERR_INVALID_ARG;
  if (H > 64) return CSA2_ERR_UNSUPPORTED;
  return CSA2_OK;
}

size_t csa2_sparse_swa_attn_decode_workspace_size(int B, int H, int topk, int n_win) {
  if (B < 0 || H < 1 || topk < 1 || n_win < 0) return 0;
  return align_up(attn_mma_workspace_bytes(B, H, topk, n_win));
}

int csa2_sparse_swa_attn_decode(const void *q_bf16, int B, int H, const uint8_t *codes,
                                const uint8_t *sf, const int64_t *cu_ctx, const int32_t *idx,
                                int topk, const uint8_t *swa_kv, int ring, int n_win,
                                float softmax_scale, void *out_bf16, float *lse, void *workspace,
                                size_t ws_bytes, void *stream) {
  if (int r = attn_args_ok(B, H, codes, sf, cu_ctx, idx, topk, softmax_scale, q_bf16, out_bf16,
                           lse, workspace))
    return r;
  if (int r = swa_args_ok(H, swa_kv, ring, n_win)) return r;
  if (B == 0) return CSA2_OK;
  if (!attn_mma_supported(H, topk, n_win)) return CSA2_ERR_UNSUPPORTED;
  const size_t need = csa2_sparse_swa_attn_decode_workspace_size(B, H, topk, n_win);
  if (ws_bytes < need || (need && !workspace)) return CSA2_ERR_WORKSPACE;
  if (int r = check_device()) return r;
  return cuda_status(launch_attn_mma(q_bf16, B, H, codes, sf, cu_ctx, idx, topk, softmax_scale,
                                     out_bf16, lse, workspace, static_cast<cudaStream_t>(stream),
                                     swa_kv, ring, n_win));
}

size_t csa2_sparse_swa_attn_prefill_workspace_size(int T, int H, int topk, int n_win) {
  (void)T, (void)H, (void)topk, (void)n_win;
  return 0;  // the tensor-core kernel keeps everything on chip
}

int csa2_sparse_swa_attn_prefill(const void *q_bf16, int T, int H, const int32_t *q_seq,
                                 const int32_t *q_vis, const uint8_t *codes, const uint8_t *sf,
                                 const int64_t *cu_ctx, int B, const int32_t *idx, int topk,
                                 const uint8_t *swa_kv, int ring, int n_win, float softmax_scale,
                                 void *out_bf16, float *lse, void *workspace, size_t ws_bytes,
                                 void *stream) {
  (void)ws_bytes;
  if (int r = attn_args_ok(T, H, codes, sf, cu_ctx, idx, topk, softmax_scale, q_bf16, out_bf16,
                           lse, workspace))
    return r;
  if (int r = swa_args_ok(H, swa_kv, ring, n_win)) return r;
  if (B < 1) return CSA2_ERR_INVALID_ARG;
  if (T == 0) return CSA2_OK;
  if (!q_seq || !aligned16(q_seq) || !q_vis || !aligned16(q_vis)) return CSA2_ERR_INVALID_ARG;
  if (!attn_prefill_supported(H)) return CSA2_ERR_UNSUPPORTED;
  if (int r = check_device()) return r;
  return cuda_status(launch_attn_prefill(q_bf16, T, H, q_seq, codes, sf, cu_ctx, idx, topk,
                                         softmax_scale, out_bf16, lse,
                                         static_cast<cudaStream_t>(stream), q_vis, swa_kv, ring,
                                         n_win));
}

int csa2_device_status(int *status, int reset, void *stream) {
  if (!status) return CSA2_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_csa2_status, sizeof(int), 0, cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return CSA2_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return CSA2_ERR_CUDA;
  *status = v;
  if (reset) {
    const int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_csa2_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                                st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return CSA2_ERR_CUDA;
  }
  return CSA2_OK;
}

uint64_t csa2_kernel_launches(void) {
  return g_kernel_launches.load(std::memory_order_relaxed);
}

}  // extern "C"

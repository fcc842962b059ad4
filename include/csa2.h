/*
 * csa2.h -- C ABI of the CSA2 hot path on one NVIDIA B300 (sm_103a).
 *
 * The operations follow the description of DeepSeek-V4.1-Flash's Compressed Sparse Attention 2
 * on two public pages:
 *   [MC]   "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (model card),
 *          Introduction, paragraph "Compressed Sparse Attention 2 (CSA2)".
 *   [WIKI] "DeepSeek V4.1-Flash" (aiwiki.ai), sections "Compressed Sparse Attention 2" and
 *          "KV-cache formats and bounded replay".
 * The pages give prose only (no formula); the exact definitions used here (rounding rules, score
 * formula, tie rule, softmax) are stated beside each entry point.
 *
 * Conventions shared by every entry point
 *   - Every data pointer is caller-owned DEVICE memory on the current CUDA device, aligned to 16
 *     bytes.  The library never allocates; scratch comes in through (workspace, ws_bytes), sized
 *     by the matching *_workspace_size() query (host-only, no GPU call).  Workspace must be
 *     256-byte aligned.  Its contents need not be initialised and are garbage afterwards.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).  Every call only
 *     enqueues work: it returns before the GPU has run it and never synchronises.
 *   - Return value: CSA2_OK (0) or a negative CSA2_ERR_* code.  Invalid arguments are detected on
 *     the host before anything is enqueued, and then nothing is enqueued.  No call aborts, exits
 *     or prints.  csa2_error_string() names a code.
 *   - Calls are thread-safe: they mutate no host state.  Two calls whose outputs or workspaces
 *     overlap must be ordered by the caller (same stream or events).
 *   - Positions ("idx") are sequence-local token numbers: row cu_ctx[b] + t of the cache holds
 *     position t of sequence b.  -1 marks an empty slot.
 *   - A device that is not sm_103 makes every call return CSA2_ERR_UNSUPPORTED.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CSA2_OK 0
#define CSA2_ERR_INVALID_ARG (-1) /* null required pointer, bad size, misalignment, bad dtype */
#define CSA2_ERR_UNSUPPORTED (-2) /* device is not sm_103 */
#define CSA2_ERR_CUDA (-3)        /* a CUDA runtime call or a kernel launch failed */
#define CSA2_ERR_WORKSPACE (-4)   /* ws_bytes is smaller than the *_workspace_size() result */
#define CSA2_ERR_TIMEOUT (-5)     /* a bounded device-side wait expired (csa2_device_status) */

/* Element types of index queries / index keys. */
#define CSA2_BF16 0 /* bfloat16, 2 bytes */
#define CSA2_E4M3 1 /* OCP FP8 E4M3 ("fn": no inf, max 448), 1 byte */

/* Latent width of one main-KV row and the sizes derived from it. */
#define CSA2_D 512
#define CSA2_ROW_CODE_BYTES (CSA2_D / 2)  /* 256: two E2M1 codes per byte */
#define CSA2_ROW_SF_BYTES (CSA2_D / 16)   /* 32: one E4M3 scale per 16 channels */

/* Human-readable name of a CSA2_* status code (static storage, never NULL). */
const char *csa2_error_string(int status);

/* ------------------------------------------------------------------------------------------ */
/* 1. FP4 main-KV quantisation                                                                  */
/* ------------------------------------------------------------------------------------------ */
/*
 * [MC] Introduction, CSA2 paragraph: the main KV cache holds E2M1 (FP4) values, and every group
 * of 16 channels shares one E4M3 scale; [WIKI] "KV-cache formats and bounded replay" likewise
 * keeps the main global KV in FP4.  The scale-selection and rounding rules are not given there; this library defines,
 * for each row and each group g of 16 consecutive channels:
 *     amax   = max |x_i| over the group              (x is bf16; bf16 -> fp32 is exact)
 *     scode  = E4M3(amax / 6)                         (fp32 division, round-to-nearest-even,
 *                                                      saturating at 448)
 *     s      = value(scode)
 *     code_i = 0 if s == 0, else E2M1(x_i / s)        (fp32 division, round-to-nearest-even,
 *                                                      saturating at 6, sign bit kept, so a
 *                                                      negative value that rounds to 0 is 0x8)
 *
 * x_bf16   [n_rows, d] bf16, row-major.
 * n_rows   number of rows (>= 0; 0 enqueues nothing).
 * d        channels per row: a multiple of 32, 32 <= d <= 4096 (the cache uses CSA2_D).
 * out_rows NULL, or [n_rows] int64: input row i is written to output row out_rows[i] (appending
 *          one new token per sequence into a ragged cache).  NULL means output row i.
 * codes    [*, d/2] uint8: byte j of a row = channel 2j (low nibble) | channel 2j+1 (high nibble).
 * sf       [*, d/16] uint8: byte g = E4M3 scale of channels 16g..16g+15.
 * Output codes and scales are bit-exact functions of the input (no accumulation order).  An
 * infinite x saturates like any large value (its group's scale is 448, its code 0x7 or 0xF);
 * NaN inputs are outside the definition and give unspecified codes.
 */
int csa2_kv_quant_fp4(const void *x_bf16, int64_t n_rows, int d, const int64_t *out_rows,
                      uint8_t *codes, uint8_t *sf, void *stream);

/* ------------------------------------------------------------------------------------------ */
/* 2. Indexer score + Top-K (Full and Reindex modes)                                            */
/* ------------------------------------------------------------------------------------------ */
/*
 * [WIKI] "Compressed Sparse Attention 2": Full mode computes index keys and queries and a fresh
 * top-k selection; Reindex mode reuses the index keys of an earlier layer but computes a new
 * query and a new selection; in the decoder's hierarchical indexer the first Full layer scores
 * all causally visible positions and later Reindex layers search only the candidate pool.  The
 * score formula is not given on the pages; this library defines, for query n with sequence
 * b = q_seq[n] and visible length V = q_vis[n]:
 *     score(t) = sum_h w[n,h] * max(0, kscale_t * sum_c q_idx[n,h,c] * k_idx[cu_ctx[b]+t, c])
 * for candidate positions t < V (kscale_t = k_scale[cu_ctx[b]+t], or 1 if k_scale is NULL).
 * Selection: the min(topk, #candidates) candidates with the largest score; equal scores
 * (+0 == -0) go to the lower position.  Output: selected positions in ascending order, then -1.
 * Scores are accumulated in fp32 on tensor cores; the selection is the exact Top-K of those
 * fp32 scores.
 *
 * q_idx     [nq, Hi, Di] of q_dtype.            w [nq, Hi] fp32.
 * q_dtype / k_dtype  must be equal: CSA2_BF16 (then Di == 64) or CSA2_E4M3 (then Di == 128);
 *           so every index-key row is 128 bytes.  1 <= Hi <= 16.
 * k_idx     [k_rows, Di] of k_dtype, sequence b occupying rows [cu_ctx[b], cu_ctx[b+1]).
 * k_rows    number of rows of k_idx (>= cu_ctx[B]); bounds every key-tile load.
 * k_scale   NULL or [k_rows] fp32 per-key scale (> 0).
 * cu_ctx    [B+1] int64, non-decreasing, cu_ctx[0] == 0.
 * q_seq     [nq] int32 in [0, B).   q_vis [nq] int32, 0 <= q_vis[n] <= rows of its sequence and
 *           q_vis[n] <= max_vis.  (Decode: q_vis = L_b; chunked prefill: q_vis = P0 + i + 1.)
 * max_vis   host-side upper bound of q_vis (sizes grids and workspace).
 * cand_blocks  NULL for Full mode (all t < V are candidates).  Reindex mode: [nq, n_cand_blocks]
 *           int32 block ids; candidates are t = block_size*id + i (0 <= i < block_size), t < V,
 *           for every id >= 0; valid ids must be distinct and in ascending order (as
 *           csa2_hier_candidate_pool writes them); -1 entries are ignored.  block_size = 8.
 * topk      1 <= topk <= 4096.
 * out_idx   [nq, topk] int32.
 * out_block_max  Full mode only: NULL, or [nq, ceil(max_vis/8)] fp32 receiving the block maxima
 *           bm[n,b] = max score over positions [8b, 8b+8) ∩ [0, V) (entries b >= ceil(V/8) are
 *           left undefined); this is the input of csa2_hier_candidate_pool.
 */
size_t csa2_index_score_topk_workspace_size(int nq, int64_t max_vis, int n_cand_blocks,
                                            int topk);
int csa2_index_score_topk(const void *q_idx, int q_dtype, const float *w, int nq, int Hi, int Di,
                          const void *k_idx, int k_dtype, int64_t k_rows, const float *k_scale,
                          const int64_t *cu_ctx, int B, const int32_t *q_seq,
                          const int32_t *q_vis, int64_t max_vis, const int32_t *cand_blocks,
                          int n_cand_blocks, int topk, int32_t *out_idx, float *out_block_max,
                          void *workspace, size_t ws_bytes, void *stream);

/*
 * csa2_index_score_topk_reindex_noalloc -- Reindex mode of csa2_index_score_topk that takes no
 * workspace.  The pages have no counterpart to this entry point; it exists for callers that
 * cannot allocate device memory when they call the library: for example a plugin running inside
 * another engine that hands it only input and output buffers, or a process that has reserved
 * all device memory up front, where a cudaMalloc would fail or stall the device.
 *
 * Arguments and results are exactly those of csa2_index_score_topk with cand_blocks non-NULL
 * (Reindex mode) and no out_block_max, workspace or ws_bytes.  The scratch it needs -- one fp32
 * score per candidate slot -- lives in a fixed array of 1,048,576 floats (4 MiB) inside the
 * library, which every GPU that loads the library holds until the process exits.  Requests with
 * nq * n_cand_blocks * 8 > 1,048,576 (e.g. more than 64 queries over a 2,048-block pool) return
 * CSA2_ERR_WORKSPACE and enqueue nothing.  The call allocates nothing (no cudaMalloc, no
 * cudaFree, no allocating library routine).
 *
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.  Every call shares the
 * one array: two calls whose work overlaps on the GPU (different streams without ordering, or
 * different host threads on the same device) race on it and give undefined results.  Nothing in
 * the array needs clearing between calls: each call writes every slot it reads.
 */
int csa2_index_score_topk_reindex_noalloc(const void *q_idx, int q_dtype, const float *w, int nq,
                                          int Hi, int Di, const void *k_idx, int k_dtype,
                                          int64_t k_rows, const float *k_scale,
                                          const int64_t *cu_ctx, int B, const int32_t *q_seq,
                                          const int32_t *q_vis, int64_t max_vis,
                                          const int32_t *cand_blocks, int n_cand_blocks, int topk,
                                          int32_t *out_idx, void *stream);

/*
 * csa2_index_block_max -- the Full-mode scan alone: block maxima of the index score over every
 * causally visible position, without a selection.  [WIKI] "Compressed Sparse Attention 2": the
 * first Full layer of the hierarchical indexer ranks blocks of eight positions by the largest
 * index score they contain; these maxima are what csa2_hier_candidate_pool ranks.
 * Arguments as csa2_index_score_topk in Full mode (no topk, cand_blocks or workspace);
 * out_block_max [nq, ceil(max_vis/8)] fp32 is required and receives exactly the values
 * csa2_index_score_topk writes there (entries b >= ceil(q_vis[n]/8) are left undefined).
 * One kernel launch; no scratch memory.
 */
int csa2_index_block_max(const void *q_idx, int q_dtype, const float *w, int nq, int Hi, int Di,
                         const void *k_idx, int k_dtype, int64_t k_rows, const float *k_scale,
                         const int64_t *cu_ctx, int B, const int32_t *q_seq, const int32_t *q_vis,
                         int64_t max_vis, float *out_block_max, void *stream);

/* ------------------------------------------------------------------------------------------ */
/* 3. Hierarchical candidate pool                                                               */
/* ------------------------------------------------------------------------------------------ */
/*
 * [MC] Introduction: in the hierarchical indexer, the first Full-mode layer builds a candidate
 * pool and the later indexing layers search only inside it; [WIKI] "Compressed Sparse Attention
 * 2": that layer ranks blocks by the largest index score they contain, and the released pool is
 * 2,048 blocks of eight positions (16,384 positions), whatever the context length.
 * For query n the pool is the min(n_pool_blocks, ceil(q_vis[n]/block_size)) blocks with the
 * largest block_max[n, b] (ties to the lower block id), block ids in ascending order, -1 padded.
 *
 * block_max       [nq, max_blocks] fp32 (row stride max_blocks), from csa2_index_score_topk.
 * q_vis           [nq] int32, ceil(q_vis[n]/block_size) <= max_blocks.
 * block_size      must be 8.     n_pool_blocks  1 <= n_pool_blocks <= 4096 (2048 on the pages).
 * out_pool_blocks [nq, n_pool_blocks] int32; pass it as cand_blocks to Reindex layers.
 * workspace / ws_bytes  at least csa2_hier_candidate_pool_workspace_size(nq, max_blocks,
 *           n_pool_blocks) bytes (0 when few blocks or many queries: one CTA per query then).
 */
size_t csa2_hier_candidate_pool_workspace_size(int nq, int64_t max_blocks, int n_pool_blocks);
int csa2_hier_candidate_pool(const float *block_max, int nq, const int32_t *q_vis,
                             int64_t max_blocks, int block_size, int n_pool_blocks,
                             int32_t *out_pool_blocks, void *workspace, size_t ws_bytes,
                             void *stream);

/*
 * csa2_index_score_topk_pool -- the first Full layer of the hierarchical decoder in one call:
 * the Full-mode selection of csa2_index_score_topk (cand_blocks NULL) and the candidate pool of
 * csa2_hier_candidate_pool over the same block maxima ([MC] Introduction: the first Full-mode
 * layer is the one that builds the pool).  out_idx, out_block_max (optional here too) and
 * out_pool_blocks are exactly what csa2_index_score_topk followed by csa2_hier_candidate_pool
 * would write.  Both selections take the top blocks by block maximum, so when n_pool_blocks >=
 * min(topk, ceil(max_vis/8)) the pool is also the block list the Full selection draws its
 * positions from, and one block selection serves both.
 *
 * Arguments as csa2_index_score_topk (Full mode) plus block_size (must be 8), n_pool_blocks
 * (1..4096) and out_pool_blocks ([nq, n_pool_blocks] int32); workspace / ws_bytes at least
 * csa2_index_score_topk_pool_workspace_size(nq, max_vis, topk, n_pool_blocks) bytes.
 * pool_event  NULL, or a cudaEvent_t created by the caller: it is recorded on `stream` as soon
 *             as out_pool_blocks is complete (before the position selection that fills out_idx),
 *             so work that needs only the pool (the Reindex layers) can wait on it and start
 *             early.  The call neither creates nor destroys it.
 */
size_t csa2_index_score_topk_pool_workspace_size(int nq, int64_t max_vis, int topk,
                                                 int n_pool_blocks);
int csa2_index_score_topk_pool(const void *q_idx, int q_dtype, const float *w, int nq, int Hi,
                               int Di, const void *k_idx, int k_dtype, int64_t k_rows,
                               const float *k_scale, const int64_t *cu_ctx, int B,
                               const int32_t *q_seq, const int32_t *q_vis, int64_t max_vis,
                               int topk, int32_t *out_idx, float *out_block_max,
                               int block_size, int n_pool_blocks, int32_t *out_pool_blocks,
                               void *workspace, size_t ws_bytes, void *stream, void *pool_event);

/* ------------------------------------------------------------------------------------------ */
/* 4. Sparse attention, decode                                                                  */
/* ------------------------------------------------------------------------------------------ */
/*
 * [MC] Introduction: layers may share one Top-K index set for their sparse attention, which
 * reads only the selected rows of the FP4 main KV.  Definition used here, per sequence b and head h:
 *     khat_j = dequant(codes[cu_ctx[b]+idx[b,j]], sf[...])   (value(code) * value(scale), exact)
 *     s_j    = softmax_scale * <q[b,h,:], khat_j>             over slots with idx[b,j] >= 0
 *     out    = sum_j softmax(s)_j * khat_j                     (K = V = the latent row)
 *     lse    = log(sum_j exp(s_j))     (natural log; -inf and out = 0 when no slot is valid)
 * Reuse mode ([WIKI] CSA2: a Reuse layer takes the latest compatible Top-K result instead of
 * selecting again) is this call with the idx buffer of an earlier layer.
 *
 * q_bf16  [B, H, 512] bf16.   1 <= H <= 128.   codes [rows, 256] / sf [rows, 32] (the cache).
 * cu_ctx  [B+1] int64.        idx [B, topk] int32, each >= 0 entry < cu_ctx[b+1]-cu_ctx[b].
 * topk    1 <= topk <= 16384. softmax_scale > 0 (1/sqrt(512) in the tests).
 * out_bf16 [B, H, 512] bf16.  lse NULL or [B, H] fp32.
 */
size_t csa2_sparse_attn_decode_workspace_size(int B, int H, int topk);
int csa2_sparse_attn_decode(const void *q_bf16, int B, int H, const uint8_t *codes,
                            const uint8_t *sf, const int64_t *cu_ctx, const int32_t *idx, int topk,
                            float softmax_scale, void *out_bf16, float *lse, void *workspace,
                            size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------------------------ */
/* 5. Sparse attention, chunked prefill                                                         */
/* ------------------------------------------------------------------------------------------ */
/*
 * As csa2_sparse_attn_decode, for T query tokens each with its own idx row (causality is carried
 * by the indexer's q_vis).  The query-key contraction is a block-scaled FP4 product: the query is
 * first quantised per (token, head) row with exactly the csa2_kv_quant_fp4 rule (16-channel E4M3
 * scales, E2M1 values), and the definition above then uses that dequantised query.  (The kernel
 * computes that product on the exactly dequantised fp16 values with fp32 accumulation.)  The
 * probability-value product uses fp16 probabilities and the exactly dequantised rows.
 *
 * q_bf16  [T, H, 512] bf16.    q_seq [T] int32 in [0, B).   idx [T, topk] int32.
 * out_bf16 [T, H, 512] bf16.   lse [T, H] fp32 or NULL.
 */
size_t csa2_sparse_attn_prefill_workspace_size(int T, int H, int topk);
int csa2_sparse_attn_prefill(const void *q_bf16, int T, int H, const int32_t *q_seq,
                             const uint8_t *codes, const uint8_t *sf, const int64_t *cu_ctx,
                             int B, const int32_t *idx, int topk, float softmax_scale,
                             void *out_bf16, float *lse, void *workspace, size_t ws_bytes,
                             void *stream);

/*
 * csa2_sparse_attn_prefill_fp4pv -- the full-FP4 variant of csa2_sparse_attn_prefill: the
 * workload asks for both prefill products, QK^T and PV, as block-scaled FP4 contractions.  The
 * probability-value product then needs P and V in FP4 with their scales along the contraction
 * axis (the slots), which the cache's per-channel scales are not.  Definition (per token and
 * head; slots j of idx[t] in blocks of 16 consecutive slots, empty slots are zero rows):
 *     s_j  = softmax_scale * <qhat_h, khat_j>      (qhat: the FP4-quantised query, as prefill)
 *     p_j  = exp(s_j - max_j s_j)
 *     Pt_j = FP4(p_j) in its block:   sc = E4M3(max p / 6),  Pt = E2M1(p / sc) * sc
 *     Vt_j = FP4(khat_j) per channel in its block, the same rule
 *     out  = sum_j Pt_j Vt_j / sum_j Pt_j,   lse = max_j s_j + log(sum_j Pt_j)
 * (fp32 divisions, round to nearest even, saturating; no valid slot: out 0, lse -inf).  Arguments
 * as csa2_sparse_attn_prefill without a workspace; H <= 64.  The numerators come from the
 * special-function unit's 2^x, so a numerator code can differ from an exactly computed one where
 * p / sc lies within a few ulps of an E2M1 rounding boundary.
 */
int csa2_sparse_attn_prefill_fp4pv(const void *q_bf16, int T, int H, const int32_t *q_seq,
                                   const uint8_t *codes, const uint8_t *sf, const int64_t *cu_ctx,
                                   int B, const int32_t *idx, int topk, float softmax_scale,
                                   void *out_bf16, float *lse, void *stream);

/* ------------------------------------------------------------------------------------------ */
/* 5b. Index keys derived from main-KV rows                                                     */
/* ------------------------------------------------------------------------------------------ */
/*
 * [WIKI] "Compressed Sparse Attention 2": CSA2 derives index keys from main KV entries rather
 * than through a separate hidden-state compression path.  The pages give no formula; this
 * library defines, for each listed cache row t (x = its dequantised FP4 row, 512 channels) and
 * the layer's index-key projection W [Di, 512] bf16:
 *     y_i   = sum_c W[i,c] x[c]                   (fp32 accumulation on the tensor cores)
 *     s     = max_i |y_i| / 448                   (fp32 division; 1 when every y_i is 0)
 *     key_i = E4M3(y_i / s)                       (round to nearest even, saturating)
 * and writes key row t of k_idx [*, Di] (E4M3) and k_scale[t] = s: exactly the k_idx / k_scale
 * inputs of csa2_index_score_topk (score uses s * <q_h, key>).
 * codes / sf: the FP4 cache.  rows: NULL (rows 0..n_rows-1) or [n_rows] int64 cache rows (e.g. the
 * new tokens of a step).  Di must be 128.  y accumulates in fp32 in the tensor core's order and
 * y_i / s is taken as y_i times the fp32 reciprocal of s, so a key can differ from a correctly
 * rounded evaluation by one code where y_i / s lies within a few fp32 ulps of an E4M3 rounding
 * boundary.
 */
int csa2_index_keys_from_kv(const uint8_t *codes, const uint8_t *sf, int64_t n_rows,
                            const int64_t *rows, const void *w_bf16, int Di, uint8_t *k_idx,
                            float *k_scale, void *stream);

/* ------------------------------------------------------------------------------------------ */
/* 6. The local sliding-window branch                                                           */
/* ------------------------------------------------------------------------------------------ */
/*
 * [WIKI] "Compressed Sparse Attention 2": every CSA2 layer creates, besides its query, its own
 * local sliding-window keys and values; [WIKI] "KV-cache formats and bounded replay": the local
 * sliding-window KV is stored in FP8 (the main global KV in FP4).  The pages give neither the
 * window length nor how the two attentions combine; this library defines:
 *   - local row: one 512-channel row per token and layer, each element E4M3 ("fn", round to
 *     nearest even, saturating at +-448, sign kept), no scale.  K = V = the local row.
 *   - ring buffer: sequence b's local rows occupy rows [b*ring, (b+1)*ring) of swa_kv; position t
 *     is row b*ring + t % ring (so only the last `ring` positions are kept).
 *   - window: a query that sees V positions attends to the local rows of its last
 *     min(n_win, V) positions (its own included), n_win <= ring.
 *   - one softmax over the union: s = softmax_scale * <q_h, row> over the selected FP4 rows
 *     (as csa2_sparse_attn_decode / _prefill) and the window's local rows together; out and lse
 *     are over the union (equivalently the two partial attentions merged by their lse).
 */

/* bf16 rows -> E4M3 local rows.  x_bf16 [n_rows, d] (d a multiple of 16, <= 4096); out_rows
 * NULL (row i) or [n_rows] int64 destination rows of swa_kv [*, d] uint8.  Bit-exact. */
int csa2_swa_kv_quant_fp8(const void *x_bf16, int64_t n_rows, int d, const int64_t *out_rows,
                          uint8_t *swa_kv, void *stream);

/* Decode: csa2_sparse_attn_decode plus the window of each sequence's last min(n_win, L_b)
 * positions (L_b = cu_ctx[b+1] - cu_ctx[b]; the cache already holds the current token).
 * swa_kv [B*ring, 512] uint8; 1 <= ring; 0 <= n_win <= ring (0: no window); H <= 64 (else
 * CSA2_ERR_UNSUPPORTED); ceil(topk/32) + ceil(n_win/32) <= 256.  Workspace: see the size query. */
size_t csa2_sparse_swa_attn_decode_workspace_size(int B, int H, int topk, int n_win);
int csa2_sparse_swa_attn_decode(const void *q_bf16, int B, int H, const uint8_t *codes,
                                const uint8_t *sf, const int64_t *cu_ctx, const int32_t *idx,
                                int topk, const uint8_t *swa_kv, int ring, int n_win,
                                float softmax_scale, void *out_bf16, float *lse, void *workspace,
                                size_t ws_bytes, void *stream);

/* Chunked prefill: csa2_sparse_attn_prefill plus, for token i, the window of the last
 * min(n_win, q_vis[i]) positions of its sequence q_seq[i] (q_vis [T] int32 as given to the
 * indexer: token i sees positions [0, q_vis[i])).  swa_kv [B*ring, 512] uint8 must already hold
 * the local rows of every window position, the chunk's own tokens included, so ring >= n_win +
 * T - 1 for a chunk of T tokens of one sequence.  H <= 64.  Needs no workspace (size 0). */
size_t csa2_sparse_swa_attn_prefill_workspace_size(int T, int H, int topk, int n_win);
int csa2_sparse_swa_attn_prefill(const void *q_bf16, int T, int H, const int32_t *q_seq,
                                 const int32_t *q_vis, const uint8_t *codes, const uint8_t *sf,
                                 const int64_t *cu_ctx, int B, const int32_t *idx, int topk,
                                 const uint8_t *swa_kv, int ring, int n_win, float softmax_scale,
                                 void *out_bf16, float *lse, void *workspace, size_t ws_bytes,
                                 void *stream);

/* ------------------------------------------------------------------------------------------ */
/* Device status                                                                                */
/* ------------------------------------------------------------------------------------------ */
/*
 * Every device-side wait in this library is bounded.  A wait that runs out records
 * CSA2_ERR_TIMEOUT in a per-device status word, and the kernel returns without further writes.
 * csa2_device_status() synchronises `stream`, copies that word into *status and, if reset != 0,
 * clears it.  Returns CSA2_OK or CSA2_ERR_CUDA.
 */
int csa2_device_status(int *status, int reset, void *stream);

/*
 * Number of kernels this library has enqueued in this process since it was loaded (all devices
 * and streams; calls that only validate or enqueue nothing add 0).  For launch accounting.
 */
uint64_t csa2_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H */

// index_score.cu -- indexer scores on CUDA cores (used for bf16 keys and as the general path).
//
// score(t) = sum_h w_h * max(0, kscale_t * <q_h, k_t>)   ("DeepSeek V4.1-Flash", aiwiki.ai,
// section "Compressed Sparse Attention 2": Full layers compute index keys and queries and score
// all causally visible positions; the formula itself is this library's definition).
//
// Two kernels share one per-key routine, so a position scored by the Full-mode scan and again by
// candidate scoring gets the identical fp32 value:
//   * score_scan:  every visible position of every query -> block maxima over 8 positions
//                  (the Full layer ranks blocks by the largest score inside them);
//   * score_cand:  the positions of a list of blocks (Reindex over the candidate pool, and the
//                  second stage of Full-mode Top-K).
#include "common.cuh"

namespace csa2 {

constexpr int kMaxHi = 16;
constexpr int kRowBytes = 128;  // Di * element size: 64 bf16 or 128 E4M3

// fp32 score of one 128-byte key row against the query held in shared memory as floats.
template <int DT>
__device__ __forceinline__ float score_key(const uint8_t *__restrict__ krow,
                                           const float *__restrict__ qs,
                                           const float *__restrict__ ws, int Hi, int Di,
                                           float kscale) {
  float acc[kMaxHi];
#pragma unroll
  for (int h = 0; h < kMaxHi; ++h) acc[h] = 0.0f;
  const uint4 *src = reinterpret_cast<const uint4 *>(krow);
#pragma unroll 1
  for (int chunk = 0; chunk < kRowBytes / 16; ++chunk) {
    const uint4 raw = __ldg(src + chunk);
    const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
    float kv[16];
    int ne;
    if (DT == CSA2_BF16) {
      ne = 8;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        kv[2 * i] = bf16_lo(wds[i]);
        kv[2 * i + 1] = bf16_hi(wds[i]);
      }
    } else {
      ne = 16;
#pragma unroll
      for (int i = 0; i < 16; ++i) kv[i] = e4m3_to_float((wds[i >> 2] >> (8 * (i & 3))) & 0xFFu);
    }
    const int c0 = chunk * ne;
#pragma unroll
    for (int h = 0; h < kMaxHi; ++h) {
      if (h < Hi) {
        const float *qh = qs + h * Di + c0;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < ne) acc[h] = fmaf(qh[i], kv[i], acc[h]);
      }
    }
  }
  float score = 0.0f;
#pragma unroll
  for (int h = 0; h < kMaxHi; ++h)
    if (h < Hi) score = fmaf(ws[h], fmaxf(acc[h] * kscale, 0.0f), score);
  return score;
}

template <int DT>
__device__ __forceinline__ void load_query(const void *q_idx, const float *w, int n, int Hi,
                                           int Di, float *qs, float *ws) {
  const int ne = Hi * Di;
  if (DT == CSA2_BF16) {
    const uint16_t *q = static_cast<const uint16_t *>(q_idx) + (int64_t)n * ne;
    for (int i = threadIdx.x; i < ne; i += blockDim.x) qs[i] = __uint_as_float((uint32_t)q[i] << 16);
  } else {
    const uint8_t *q = static_cast<const uint8_t *>(q_idx) + (int64_t)n * ne;
    for (int i = threadIdx.x; i < ne; i += blockDim.x) qs[i] = e4m3_to_float(q[i]);
  }
  for (int i = threadIdx.x; i < Hi; i += blockDim.x) ws[i] = w[(int64_t)n * Hi + i];
}

template <int DT>
__global__ void __launch_bounds__(256) score_scan_kernel(
    const void *__restrict__ q_idx, const float *__restrict__ w, int Hi, int Di,
    const uint8_t *__restrict__ k_idx, const float *__restrict__ k_scale,
    const int64_t *__restrict__ cu_ctx, const int32_t *__restrict__ q_seq,
    const int32_t *__restrict__ q_vis, float *__restrict__ bm, int64_t bm_stride) {
  pdl_wait();
  pdl_trigger();
  __shared__ float qs[kMaxHi * 128];
  __shared__ float ws[kMaxHi];
  const int n = blockIdx.y;
  const int64_t V = q_vis[n];
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x;
  if (t0 >= V) return;  // uniform over the CTA
  load_query<DT>(q_idx, w, n, Hi, Di, qs, ws);
  __syncthreads();
  const int64_t base = cu_ctx[q_seq[n]];
  const int64_t t = t0 + threadIdx.x;
  float s = -INFINITY;
  if (t < V) {
    const float ks = k_scale ? k_scale[base + t] : 1.0f;
    s = score_key<DT>(k_idx + (base + t) * kRowBytes, qs, ws, Hi, Di, ks);
  }
  // block max over 8 consecutive positions = 8 consecutive lanes
  s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, 1));
  s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, 2));
  s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, 4));
  if ((threadIdx.x & 7) == 0 && t < V) bm[(int64_t)n * bm_stride + (t >> 3)] = s;
}

template <int DT>
__global__ void __launch_bounds__(256) score_cand_kernel(
    const void *__restrict__ q_idx, const float *__restrict__ w, int Hi, int Di,
    const uint8_t *__restrict__ k_idx, const float *__restrict__ k_scale,
    const int64_t *__restrict__ cu_ctx, const int32_t *__restrict__ q_seq,
    const int32_t *__restrict__ q_vis, const int32_t *__restrict__ cand_blocks,
    int n_cand_blocks, float *__restrict__ scores) {
  pdl_wait();
  pdl_trigger();
  __shared__ float qs[kMaxHi * 128];
  __shared__ float ws[kMaxHi];
  const int n = blockIdx.y;
  load_query<DT>(q_idx, w, n, Hi, Di, qs, ws);
  __syncthreads();
  const int64_t n_slots = (int64_t)n_cand_blocks * kBlock;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_slots) return;
  const int64_t V = q_vis[n];
  const int blk = cand_blocks[(int64_t)n * n_cand_blocks + (i >> 3)];
  const int64_t t = (int64_t)blk * kBlock + (i & 7);
  float s = 0.0f;
  if (blk >= 0 && t < V) {
    const int64_t base = cu_ctx[q_seq[n]];
    const float ks = k_scale ? k_scale[base + t] : 1.0f;
    s = score_key<DT>(k_idx + (base + t) * kRowBytes, qs, ws, Hi, Di, ks);
  }
  scores[(int64_t)n * n_slots + i] = s;
}

cudaError_t launch_score_scan(const void *q_idx, int dtype, const float *w, int nq, int Hi,
                              int Di, const void *k_idx, const float *k_scale,
                              const int64_t *cu_ctx, const int32_t *q_seq, const int32_t *q_vis,
                              int64_t max_vis, float *bm, int64_t bm_stride, cudaStream_t st) {
  if (nq == 0 || max_vis == 0) return cudaSuccess;
  dim3 grid((unsigned)((max_vis + 255) / 256), (unsigned)nq);
  const uint8_t *k = static_cast<const uint8_t *>(k_idx);
  cudaError_t e;
  if (dtype == CSA2_BF16)
    e = launch_pdl(score_scan_kernel<CSA2_BF16>, grid, dim3(256), 0, st, q_idx, w, Hi, Di, k,
                   k_scale, cu_ctx, q_seq, q_vis, bm, bm_stride);
  else
    e = launch_pdl(score_scan_kernel<CSA2_E4M3>, grid, dim3(256), 0, st, q_idx, w, Hi, Di, k,
                   k_scale, cu_ctx, q_seq, q_vis, bm, bm_stride);
  note_launches(1);
  return e;
}

cudaError_t launch_score_cand(const void *q_idx, int dtype, const float *w, int nq, int Hi,
                              int Di, const void *k_idx, const float *k_scale,
                              const int64_t *cu_ctx, const int32_t *q_seq, const int32_t *q_vis,
                              const int32_t *cand_blocks, int n_cand_blocks, float *scores,
                              cudaStream_t st) {
  if (nq == 0 || n_cand_blocks == 0) return cudaSuccess;
  const int64_t n_slots = (int64_t)n_cand_blocks * kBlock;
  dim3 grid((unsigned)((n_slots + 255) / 256), (unsigned)nq);
  const uint8_t *k = static_cast<const uint8_t *>(k_idx);
  cudaError_t e;
  if (dtype == CSA2_BF16)
    e = launch_pdl(score_cand_kernel<CSA2_BF16>, grid, dim3(256), 0, st, q_idx, w, Hi, Di, k,
                   k_scale, cu_ctx, q_seq, q_vis, cand_blocks, n_cand_blocks, scores);
  else
    e = launch_pdl(score_cand_kernel<CSA2_E4M3>, grid, dim3(256), 0, st, q_idx, w, Hi, Di, k,
                   k_scale, cu_ctx, q_seq, q_vis, cand_blocks, n_cand_blocks, scores);
  note_launches(1);
  return e;
}

}  // namespace csa2

// common.cuh -- shared device helpers of the CSA2 CUDA library (sm_103a only).
#pragma once

#include <atomic>
#include <mutex>

#include <algorithm>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa2.h"

namespace csa2 {

constexpr int kD = CSA2_D;              // latent width of a main-KV row
constexpr int kCodeBytes = kD / 2;      // 256 bytes of E2M1 codes per row
constexpr int kSfBytes = kD / 16;       // 32 E4M3 scales per row
constexpr int kBlock = 8;               // positions per indexer block (pool granularity)

// ------------------------------------------------------------------------------------------
// Number formats, device side.  Written independently of any CPU code: bit placement, not
// tables or search.
// ------------------------------------------------------------------------------------------

// E4M3 ("fn") byte -> float, exact.  Normal: sign | (e + 120) << 23 | m << 20; subnormal m * 2^-9.
__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
  uint32_t e = (b >> 3) & 15u, m = b & 7u;
  float mag = (e == 0) ? (float)m * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (m << 20));
  return (b & 0x80u) ? -mag : mag;
}

// E2M1 code (low nibble) -> float magnitude with sign, exact.
__device__ __forceinline__ float e2m1_to_float(uint32_t c) {
  // magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6} as exponent/mantissa placement:
  // e = (c>>1)&3, m = c&1; e == 0 -> 0.5*m; else (1 + m/2) * 2^(e-1)
  uint32_t e = (c >> 1) & 3u, m = c & 1u;
  float mag = (e == 0) ? 0.5f * (float)m : __uint_as_float(((e + 126u) << 23) | (m << 22));
  return (c & 8u) ? -mag : mag;
}

// float >= 0 -> E4M3 code, round to nearest even (subnormals included), saturating at 448 (0x7E),
// by the conversion instruction; +inf and NaN also give 0x7E.
__device__ __forceinline__ uint32_t float_to_e4m3_sat(float s) {
  if (!(s < 448.0f)) return 0x7Eu;
  uint16_t two;
  // the first source lands in the upper byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(two) : "f"(0.0f), "f"(s));
  return two & 0xFFu;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Order-preserving map of a finite float to uint32 (larger float -> larger key), with -0 == +0.
// Finite floats map to [0x00800000, 0xFF7FFFFF]; key 0 never comes from a finite float.
__device__ __forceinline__ uint32_t float_key(float v) {
  uint32_t u = (v == 0.0f) ? 0u : __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Programmatic dependent launch.  The library's kernels are enqueued with programmatic stream
// serialisation (launch_pdl), so the CTAs of a kernel may be scheduled while the kernel before
// it drains.  Every kernel calls pdl_wait() before its first global-memory access (read or
// write): it returns once the previous grid has completed and its writes are visible.  A kernel
// calls pdl_trigger() once it holds its own resources (after any TMEM allocation), which lets
// the next kernel's CTAs start their prologue; so every CTA of an earlier grid has allocated
// before any CTA of a later grid exists, and a later CTA only ever waits for TMEM that an
// earlier one frees.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Per-device status word written by bounded device-side waits that ran out.  The library is
// built as one translation unit (csa2_lib.cu), so this is its single definition.
__device__ int g_csa2_status = 0;

}  // namespace csa2

// ------------------------------------------------------------------------------------------
// Host-side launchers (defined in the kernel files, called from api.cu).  All return
// cudaError_t of the launch.
// ------------------------------------------------------------------------------------------
namespace csa2 {

// cudaFuncSetAttribute(kernel, attr, value) once per (kernel address, device) per process: the
// value never changes for a kernel, and repeating the call costs host time on every launch.
inline cudaError_t set_attr_once(const void *kernel, cudaFuncAttribute attr, int value) {
  struct Entry { const void *k; int attr; uint64_t devs; };
  static std::mutex mu;
  static Entry table[64];
  static int used = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  std::lock_guard<std::mutex> lock(mu);
  Entry *ent = nullptr;
  for (int i = 0; i < used; ++i)
    if (table[i].k == kernel && table[i].attr == (int)attr) ent = &table[i];
  if (ent && bit && (ent->devs & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, attr, value);
  if (e != cudaSuccess) return e;
  if (!ent && used < 64) ent = &table[used++], ent->k = kernel, ent->attr = (int)attr, ent->devs = 0;
  if (ent) ent->devs |= bit;
  return cudaSuccess;
}
template <class K>
inline cudaError_t set_smem_once(K *kernel, cudaFuncAttribute attr, int value) {
  return set_attr_once(reinterpret_cast<const void *>(kernel), attr, value);
}

// Enqueue `kern` on `st` with programmatic stream serialisation (see pdl_wait / pdl_trigger).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Process-wide count of kernels enqueued by the library (csa2_kernel_launches).
inline std::atomic<uint64_t> g_kernel_launches{0};
inline void note_launches(int n) { g_kernel_launches.fetch_add(n, std::memory_order_relaxed); }

cudaError_t launch_kv_quant(const void *x, int64_t n_rows, int d, const int64_t *out_rows,
                            uint8_t *codes, uint8_t *sf, cudaStream_t st);

// Full-mode scan: block maxima of the score for every visible position of every query.
cudaError_t launch_score_scan(const void *q_idx, int dtype, const float *w, int nq, int Hi,
                              int Di, const void *k_idx, const float *k_scale,
                              const int64_t *cu_ctx, const int32_t *q_seq, const int32_t *q_vis,
                              int64_t max_vis, float *bm, int64_t bm_stride, cudaStream_t st);

// Candidate scoring: scores of the positions of n_cand_blocks listed blocks per query.
cudaError_t launch_score_cand(const void *q_idx, int dtype, const float *w, int nq, int Hi,
                              int Di, const void *k_idx, const float *k_scale,
                              const int64_t *cu_ctx, const int32_t *q_seq, const int32_t *q_vis,
                              const int32_t *cand_blocks, int n_cand_blocks, float *scores,
                              cudaStream_t st);

// Top-K selection.  Element i of query n lives at vals[n*stride + i], i < n_elems.
//   map == nullptr: element i is block/position i, valid iff i < ceil(q_vis[n] / unit)
//                   (unit = 8 for block maxima, 1 for positions);
//   map != nullptr: element i is position map[n*map_stride + i/8]*8 + i%8, valid iff the block
//                   id is >= 0 and the position is < q_vis[n].
//   pos_vals != nullptr: the value of an element is pos_vals[n*pos_stride + position] instead.
//   ws: workspace of topk_workspace_bytes(nq, n_elems) bytes (may be null when that is 0 or to
//       force the one-CTA-per-query path).
cudaError_t launch_topk(const float *vals, int64_t stride, int64_t n_elems, const int32_t *map,
                        int64_t map_stride, int unit, const int32_t *q_vis, int nq, int topk,
                        int32_t *out, cudaStream_t st, const float *pos_vals = nullptr,
                        int64_t pos_stride = 0, void *ws = nullptr);
size_t topk_workspace_bytes(int nq, int64_t n_elems);

// Tensor-core indexer (index_mma.cu, index_multi.cu).
bool index_mma_supported(int nq);   // single-query scan (nq <= 1024)
bool cand_mma_supported();          // candidate scoring, any nq
bool index_multi_supported(int nq, int Hi, int B);  // 32-query scan over one sequence
cudaError_t launch_score_scan_multi(const void *q_idx, int dtype, const float *w, int nq,
                                    const void *k_idx, int64_t k_rows, const float *k_scale,
                                    const int32_t *q_vis, int64_t max_vis, float *bm,
                                    int64_t bm_stride, float *scores, int64_t sc_stride,
                                    cudaStream_t st);
cudaError_t launch_score_scan_mma(const void *q_idx, int dtype, const float *w, int nq, int Hi,
                                  const void *k_idx, int64_t k_rows, const float *k_scale,
                                  const int64_t *cu_ctx, const int32_t *q_seq,
                                  const int32_t *q_vis, int64_t max_vis, float *bm,
                                  int64_t bm_stride, float *scores, int64_t sc_stride,
                                  cudaStream_t st);
cudaError_t launch_score_cand_mma(const void *q_idx, int dtype, const float *w, int nq, int Hi,
                                  const void *k_idx, int64_t k_rows, const float *k_scale,
                                  const int64_t *cu_ctx, const int32_t *q_seq,
                                  const int32_t *q_vis, const int32_t *cand, int n_cand,
                                  float *scores, cudaStream_t st);

cudaError_t launch_attn(const void *q_bf16, const uint8_t *q_codes, const uint8_t *q_sf, int nq,
                        int H, const int32_t *q_seq, const uint8_t *codes, const uint8_t *sf,
                        const int64_t *cu_ctx, const int32_t *idx, int topk, float scale,
                        void *out_bf16, float *lse, void *workspace, cudaStream_t st);
size_t attn_workspace_bytes(int nq, int H, int topk);

// Tensor-core prefill attention (attn_prefill.cu): one CTA per query token, H <= 64; the query
// is FP4-quantised inside the kernel.  With n_win > 0 the last n_win of the q_vis[i] positions
// token i sees add their local rows (swa_kv, ring) to the same softmax.
bool attn_prefill_supported(int H);
cudaError_t launch_attn_prefill(const void *q_bf16, int T, int H, const int32_t *q_seq,
                                const uint8_t *codes, const uint8_t *sf, const int64_t *cu_ctx,
                                const int32_t *idx, int topk, float scale, void *out_bf16,
                                float *lse, cudaStream_t st, const int32_t *q_vis = nullptr,
                                const uint8_t *swa_kv = nullptr, int ring = 1, int n_win = 0);

// The full-FP4 PV variant of prefill attention (attn_fp4pv.cu): H <= 64, no workspace.
cudaError_t launch_attn_fp4pv(const void *q_bf16, int T, int H, const int32_t *q_seq,
                              const uint8_t *codes, const uint8_t *sf, const int64_t *cu_ctx,
                              const int32_t *idx, int topk, float scale, void *out_bf16,
                              float *lse, cudaStream_t st);

// Tensor-core decode attention (attn_mma.cu): H <= 64, tiles of 128 selected rows, partial
// results merged by a combine kernel; with n_win > 0 (swa_kv, ring) the window's local rows join
// the same softmax.  Few tiles in all go to the small-tile kernel of attn_small.cu instead.
bool attn_mma_supported(int H, int topk, int n_win = 0);
size_t attn_mma_workspace_bytes(int nq, int H, int topk, int n_win = 0);
cudaError_t launch_attn_mma(const void *q_bf16, int nq, int H, const uint8_t *codes,
                            const uint8_t *sf, const int64_t *cu_ctx, const int32_t *idx,
                            int topk, float scale, void *out_bf16, float *lse, void *workspace,
                            cudaStream_t st, const uint8_t *swa_kv = nullptr, int ring = 1,
                            int n_win = 0);

// The decode attention for few tiles (attn_small.cu): tiles of 32 rows x 32 heads, chosen by
// launch_attn_mma when they fit in about one wave; the same arguments and result.
bool attn_small_preferred(int nq, int H, int topk, int n_win);
size_t attn_small_workspace_bytes(int nq, int H, int topk, int n_win);
cudaError_t launch_attn_small(const void *q_bf16, int nq, int H, const uint8_t *codes,
                              const uint8_t *sf, const int64_t *cu_ctx, const int32_t *idx,
                              int topk, float scale, void *out_bf16, float *lse, void *workspace,
                              cudaStream_t st, const uint8_t *swa_kv, int ring, int n_win);

// Index keys derived from main-KV rows (index_keys.cu): keys [*, 128] E4M3 and k_scale of the
// given cache rows (rows NULL: rows 0..n_rows-1), projection W [128, 512] bf16.
bool index_keys_supported();
cudaError_t launch_index_keys(const uint8_t *codes, const uint8_t *sf, int64_t n_rows,
                              const int64_t *rows, const void *w_bf16, uint8_t *keys,
                              float *k_scale, cudaStream_t st);

// FP8 (E4M3) local sliding-window rows: bf16 -> E4M3, round to nearest even, saturating.
cudaError_t launch_fp8_quant(const void *x, int64_t n_rows, int d, const int64_t *out_rows,
                             uint8_t *out, cudaStream_t st);

}  // namespace csa2

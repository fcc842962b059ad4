// topk.cu -- exact Top-K selection with the lower-position tie rule, one CTA per query.
//
// Order: larger score first, equal scores (+0 == -0) -> lower position first.  Output: the
// selected positions in ascending order, then -1.  Used for Full-mode selection, the candidate
// pool ("selects blocks by their maximum index score", "DeepSeek V4.1-Flash", aiwiki.ai, section
// "Compressed Sparse Attention 2") and Reindex selection.
//
// Algorithm: radix select on order-preserving 32-bit keys, most significant digit first
// (11 + 11 + 10 bits), each digit found from a shared-memory histogram and a block-wide suffix
// scan, stopping early once a whole bin is taken.  That yields a threshold key T and the number
// need_eq of elements equal to T that are taken (the lowest positions among them).  A final
// ordered pass compacts the selected elements in index order with block-wide prefix sums, which
// gives ascending output without a sort.
#include "common.cuh"

namespace csa2 {

constexpr int kTopkThreads = 1024;
constexpr int kWarps = kTopkThreads / 32;

struct ElemView {
  const float *vals;
  const float *pos_vals;  // non-null: the value of an element is pos_vals[its position]
  const int32_t *map;  // nullptr: identity
  int64_t n_elems;
  int64_t limit;       // identity: valid iff i < limit; map: valid iff pos < limit
  __device__ __forceinline__ bool get(int64_t i, uint32_t &key, int64_t &pos) const {
    if (map) {
      const int blk = map[i >> 3];
      pos = (int64_t)blk * kBlock + (i & 7);
      if (blk < 0 || pos >= limit) return false;
    } else {
      pos = i;
      if (i >= limit) return false;
    }
    key = float_key(pos_vals ? pos_vals[pos] : vals[i]);
    return true;
  }
};

// Block-wide exclusive scan of one uint32 per thread; returns the exclusive prefix and writes
// the block total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *warp_tot,
                                                         uint32_t &total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_tot[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    uint32_t t = warp_tot[lane];
    uint32_t ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += y;
    }
    warp_tot[lane] = ti - t;  // exclusive warp offsets
    if (lane == 31) warp_tot[32] = ti;
  }
  __syncthreads();
  const uint32_t res = warp_tot[wid] + inc - v;
  total = warp_tot[32];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(
    const float *__restrict__ vals, int64_t stride, const float *__restrict__ pos_vals,
    int64_t pos_stride, int64_t n_elems,
    const int32_t *__restrict__ map, int64_t map_stride, int unit,
    const int32_t *__restrict__ q_vis, int topk, int32_t *__restrict__ out) {
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t warp_tot[33];
  __shared__ uint32_t s_digit, s_above, s_nvalid;

  const int n = blockIdx.x;
  const int64_t V = q_vis[n];
  ElemView ev;
  ev.vals = vals ? vals + (int64_t)n * stride : nullptr;
  ev.pos_vals = pos_vals ? pos_vals + (int64_t)n * pos_stride : nullptr;
  ev.map = map ? map + (int64_t)n * map_stride : nullptr;
  ev.n_elems = n_elems;
  ev.limit = map ? V : (V + unit - 1) / unit;
  int32_t *o = out + (int64_t)n * topk;

  uint32_t prefix = 0;      // digits fixed so far
  int pshift = 32;          // keys with (key >> pshift) == prefix are still in play
  uint32_t rem = 0;         // how many still to take among them
  uint32_t T = 0, need_eq = 0;
  bool done = false;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};

  if (threadIdx.x == 0) s_nvalid = 0;
  for (int pass = 0; pass < 3 && !done; ++pass) {
    const int shift = shifts[pass], nb = 1 << widths[pass];
    for (int i = threadIdx.x; i < nb; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    uint32_t local_valid = 0;
    for (int64_t i = threadIdx.x; i < n_elems; i += kTopkThreads) {
      uint32_t key;
      int64_t pos;
      if (!ev.get(i, key, pos)) continue;
      ++local_valid;
      if (pshift == 32 || (key >> pshift) == prefix)
        atomicAdd(&hist[(key >> shift) & (nb - 1)], 1u);
    }
    if (pass == 0) {
      local_valid = __reduce_add_sync(0xffffffffu, local_valid);
      if ((threadIdx.x & 31) == 0) atomicAdd(&s_nvalid, local_valid);
    }
    __syncthreads();
    if (pass == 0) {
      rem = min((uint32_t)topk, s_nvalid);
      if (rem == 0) break;
    }
    // suffix scan: thread i owns bins nb-1-2i and nb-2-2i (descending digit order)
    uint32_t c0 = 0, c1 = 0;
    const int b0 = nb - 1 - 2 * threadIdx.x, b1 = b0 - 1;
    if (b0 >= 0) c0 = hist[b0];
    if (b1 >= 0) c1 = hist[b1];
    uint32_t tot;
    const uint32_t before = block_exclusive_scan(c0 + c1, warp_tot, tot);
    // the digit where the count from the top first reaches rem
    if (b0 >= 0 && before < rem && before + c0 >= rem) {
      s_digit = b0; s_above = before;
    } else if (b1 >= 0 && before + c0 < rem && before + c0 + c1 >= rem) {
      s_digit = b1; s_above = before + c0;
    }
    __syncthreads();
    const uint32_t digit = s_digit;
    const uint32_t cnt = hist[digit];
    rem -= s_above;
    prefix = (pshift == 32) ? digit : ((prefix << widths[pass]) | digit);
    pshift = shift;
    if (cnt == rem || pass == 2) {
      if (cnt == rem) {  // every key of this bin is taken: select key >= prefix << shift
        T = (prefix << shift) - 1u;  // prefix << shift >= 0x00800000 for finite values
        need_eq = 0;
      } else {
        T = prefix;
        need_eq = rem;
      }
      done = true;
    }
    __syncthreads();
  }

  if (!done) {  // no valid element
    for (int i = threadIdx.x; i < topk; i += kTopkThreads) o[i] = -1;
    return;
  }
  const uint32_t k_eff = min((uint32_t)topk, s_nvalid);

  // ordered compaction: chunks of 4 consecutive elements per thread
  uint32_t gt_base = 0, eq_base = 0;
  for (int64_t c0 = 0; c0 < n_elems; c0 += 4 * kTopkThreads) {
    uint32_t keys[4];
    int64_t poss[4];
    bool valid[4];
    uint32_t ngt = 0, neq = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t i = c0 + 4 * threadIdx.x + j;
      valid[j] = (i < n_elems) && ev.get(i, keys[j], poss[j]);
      if (valid[j]) {
        ngt += keys[j] > T;
        neq += keys[j] == T;
      }
    }
    uint32_t tot;
    const uint32_t ex = block_exclusive_scan(ngt | (neq << 16), warp_tot, tot);
    uint32_t gt_r = gt_base + (ex & 0xFFFFu), eq_r = eq_base + (ex >> 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (!valid[j]) continue;
      const bool gt = keys[j] > T, eq = keys[j] == T;
      if (gt || (eq && eq_r < need_eq)) {
        const uint32_t slot = gt_r + min(eq_r, need_eq);
        o[slot] = (int32_t)poss[j];
      }
      gt_r += gt;
      eq_r += eq;
    }
    gt_base += tot & 0xFFFFu;
    eq_base += tot >> 16;
  }
  for (int i = k_eff + threadIdx.x; i < topk; i += kTopkThreads) o[i] = -1;
}

cudaError_t launch_topk(const float *vals, int64_t stride, int64_t n_elems, const int32_t *map,
                        int64_t map_stride, int unit, const int32_t *q_vis, int nq, int topk,
                        int32_t *out, cudaStream_t st, const float *pos_vals,
                        int64_t pos_stride) {
  if (nq == 0) return cudaSuccess;
  topk_kernel<<<nq, kTopkThreads, 0, st>>>(vals, stride, pos_vals, pos_stride, n_elems, map,
                                           map_stride, unit, q_vis, topk, out);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace csa2

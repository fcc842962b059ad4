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
// ordered pass writes the selected elements in index order: every warp owns one contiguous
// segment, counts its selections with ballots, one block-wide scan gives each warp its output
// offset, and a second sweep emits positions in order -- ascending output without a sort.
// The scores live in L2; each pass keeps 16 independent loads in flight per thread.
#include "common.cuh"

namespace csa2 {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kUnroll = 16;

struct ElemView {
  const float *vals;
  const float *pos_vals;  // non-null: the value of an element is pos_vals[its position]
  const int32_t *map;     // nullptr: identity
  int64_t n_elems;
  int64_t limit;          // identity: valid iff i < limit; map: valid iff pos < limit
  __device__ __forceinline__ bool get(int64_t i, uint32_t &key, int32_t &pos) const {
    if (i >= n_elems) return false;
    int64_t p;
    if (map) {
      const int blk = __ldg(map + (i >> 3));
      p = (int64_t)blk * kBlock + (i & 7);
      if (blk < 0 || p >= limit) return false;
    } else {
      p = i;
      if (i >= limit) return false;
    }
    pos = (int32_t)p;
    key = float_key(pos_vals ? pos_vals[p] : vals[i]);
    return true;
  }
};

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// Block-wide exclusive scan of one uint32 per thread; also returns the block total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *warp_tot,
                                                         uint32_t &total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint32_t inc = warp_incl_scan(v);
  if (lane == 31) warp_tot[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    const uint32_t t = warp_tot[lane];
    const uint32_t ti = warp_incl_scan(t);
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
    int64_t pos_stride, int64_t n_elems, const int32_t *__restrict__ map, int64_t map_stride,
    int unit, const int32_t *__restrict__ q_vis, int topk, int32_t *__restrict__ out) {
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t warp_tot[33];
  __shared__ uint32_t seg_gt[kTopkWarps], seg_eq[kTopkWarps];
  __shared__ uint32_t s_digit, s_above, s_nvalid;

  const int n = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int64_t V = q_vis[n];
  ElemView ev;
  ev.vals = vals ? vals + (int64_t)n * stride : nullptr;
  ev.pos_vals = pos_vals ? pos_vals + (int64_t)n * pos_stride : nullptr;
  ev.map = map ? map + (int64_t)n * map_stride : nullptr;
  ev.n_elems = n_elems;
  ev.limit = map ? V : (V + unit - 1) / unit;
  int32_t *o = out + (int64_t)n * topk;

  uint32_t prefix = 0;  // digits fixed so far
  int pshift = 32;      // keys with (key >> pshift) == prefix are still in play
  uint32_t rem = 0;     // how many still to take among them
  uint32_t T = 0, need_eq = 0;
  bool done = false;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};

  if (tid == 0) s_nvalid = 0;
  for (int pass = 0; pass < 3 && !done; ++pass) {
    const int shift = shifts[pass], nb = 1 << widths[pass];
    for (int i = tid; i < nb; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    uint32_t local_valid = 0;
    for (int64_t base = 0; base < n_elems; base += (int64_t)kTopkThreads * kUnroll) {
      uint32_t keys[kUnroll];
      bool ok[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        int32_t pos;
        ok[u] = ev.get(base + (int64_t)u * kTopkThreads + tid, keys[u], pos);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (!ok[u]) continue;
        ++local_valid;
        if (pshift == 32 || (keys[u] >> pshift) == prefix)
          atomicAdd(&hist[(keys[u] >> shift) & (nb - 1)], 1u);
      }
    }
    if (pass == 0) {
      local_valid = __reduce_add_sync(0xffffffffu, local_valid);
      if (lane == 0) atomicAdd(&s_nvalid, local_valid);
    }
    __syncthreads();
    if (pass == 0) {
      rem = min((uint32_t)topk, s_nvalid);
      if (rem == 0) break;
    }
    // suffix scan: thread i owns bins nb-1-2i and nb-2-2i (descending digit order)
    uint32_t c0 = 0, c1 = 0;
    const int b0 = nb - 1 - 2 * tid, b1 = b0 - 1;
    if (b0 >= 0) c0 = hist[b0];
    if (b1 >= 0) c1 = hist[b1];
    uint32_t tot;
    const uint32_t before = block_exclusive_scan(c0 + c1, warp_tot, tot);
    // the digit where the count from the top first reaches rem
    if (b0 >= 0 && before < rem && before + c0 >= rem) {
      s_digit = b0;
      s_above = before;
    } else if (b1 >= 0 && before + c0 < rem && before + c0 + c1 >= rem) {
      s_digit = b1;
      s_above = before + c0;
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
    for (int i = tid; i < topk; i += kTopkThreads) o[i] = -1;
    return;
  }
  const uint32_t k_eff = min((uint32_t)topk, s_nvalid);

  // ordered emission: warp w owns elements [w*seg, (w+1)*seg)
  const int64_t seg = ((n_elems + kTopkWarps - 1) / kTopkWarps + 31) / 32 * 32;
  const int64_t w0 = (int64_t)wid * seg, w1 = min(n_elems, w0 + seg);
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint32_t ngt = 0, neq = 0;
  for (int64_t b = w0; b < w1; b += 32 * kUnroll) {
    uint32_t keys[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = b + 32 * u + lane;
      int32_t pos;
      ok[u] = i < w1 && ev.get(i, keys[u], pos);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      ngt += __popc(__ballot_sync(0xffffffffu, ok[u] && keys[u] > T));
      neq += __popc(__ballot_sync(0xffffffffu, ok[u] && keys[u] == T));
    }
  }
  if (lane == 0) {
    seg_gt[wid] = ngt;
    seg_eq[wid] = neq;
  }
  __syncthreads();
  if (wid == 0) {
    const uint32_t g = seg_gt[lane], e = seg_eq[lane];
    const uint32_t gi = warp_incl_scan(g), ei = warp_incl_scan(e);
    seg_gt[lane] = gi - g;
    seg_eq[lane] = ei - e;
  }
  __syncthreads();
  uint32_t gt_r = seg_gt[wid], eq_r = seg_eq[wid];
  for (int64_t b = w0; b < w1; b += 32 * kUnroll) {
    uint32_t keys[kUnroll];
    int32_t poss[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = b + 32 * u + lane;
      ok[u] = i < w1 && ev.get(i, keys[u], poss[u]);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const bool gt = ok[u] && keys[u] > T, eq = ok[u] && keys[u] == T;
      const uint32_t bgt = __ballot_sync(0xffffffffu, gt), beq = __ballot_sync(0xffffffffu, eq);
      const uint32_t my_gt = gt_r + __popc(bgt & lt_mask), my_eq = eq_r + __popc(beq & lt_mask);
      if (gt || (eq && my_eq < need_eq)) o[my_gt + min(my_eq, need_eq)] = poss[u];
      gt_r += __popc(bgt);
      eq_r += __popc(beq);
    }
  }
  for (int i = k_eff + tid; i < topk; i += kTopkThreads) o[i] = -1;
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

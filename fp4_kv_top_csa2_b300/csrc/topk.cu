// topk.cu -- exact Top-K selection with the lower-position tie rule, one CTA per query.
//
// Order: larger score first, equal scores (+0 == -0) -> lower position first.  Output: the
// selected positions in ascending order, then -1.  Used for Full-mode selection, the candidate
// pool (blocks ranked by the largest index score inside them, "DeepSeek V4.1-Flash", aiwiki.ai,
// section "Compressed Sparse Attention 2") and Reindex selection.
//
// Keys are order-preserving 32-bit images of the scores (key 0 = not a candidate).  Every kernel
// finds the k-th largest key T, takes every key > T and the need_eq = k - #(keys > T) keys equal
// to T with the lowest positions, and emits in index order: each warp owns a contiguous
// segment, counts its selections with ballots, one scan gives each warp its offset, and a
// second sweep writes positions (no sort).  T comes from radix11_kth: 11-bit digits, a shared
// histogram per digit and a block scan, finished by a single warp ranking the keys once no more
// than 32 remain in play.
//
// Kernels, by size (launch_topk picks one):
//   * topk_reg_kernel -- n <= 16,384 elements, any number of queries, one 1024-thread CTA per
//     query.  The elements stay in registers (16 per thread).  A threshold from the exact rank
//     of 128 sampled keys keeps a little over k candidates, which are compacted in index order
//     into shared memory; the selection runs on them.
//   * topk_filter_kernel + topk_select_kernel -- larger n, at most 64 queries (the decoder's
//     131,072 block maxima): one filter CTA per 4,096-element chunk keeps the (key, position)
//     pairs at or above a threshold from the exact rank of 256 strided samples (the same in
//     every CTA); one select CTA per query gathers the kept lists and selects.
//   * topk_kernel -- larger n with many queries (chunked prefill): one CTA per query; up to
//     16,384 elements staged in shared memory, else a strided sample of 8,192 keys gives an
//     estimate T_est (kth_radix, 8-bit digits) and the keys >= T_est are staged instead.
// A sampled threshold that keeps fewer than k elements (or more than the staging room) falls
// back to selecting over all elements, so every path is exact.  The three ways an element can
// be addressed (block maxima by index; candidate slots through a block list with slot-indexed
// or position-indexed scores) are separate kernel instances, so every global load is
// straight-line code with clamped indices and validity as a mask.
#include "common.cuh"

namespace csa2 {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kUnroll = 8;       // loads in flight per thread (key + position)
constexpr int kSmemCap = 16384;  // elements held in shared memory
constexpr int kWarpCap = kSmemCap / kTopkWarps;  // per-warp staging slots (512)
constexpr int kSample = 8192;
constexpr size_t kTopkSmem = (size_t)kSmemCap * 8;

enum TopkMode { kById = 0, kMapSlot = 1, kMapPos = 2 };

template <int MODE>
struct ElemView {  // elements in global memory
  const float *vals;   // kById / kMapSlot: value of element i; kMapPos: value of position p
  const int32_t *map;  // kMapSlot / kMapPos: element i -> position map[i/8]*8 + i%8
  int64_t n_elems;     // >= 1
  int64_t limit;       // kById: valid iff i < limit; mapped: valid iff position < limit
  int64_t val_len;     // readable length of vals (>= 1)
  __device__ __forceinline__ uint32_t get(int64_t i, int32_t &pos) const {
    const bool in = i < n_elems;
    const int64_t ic = in ? i : n_elems - 1;
    int64_t p, vi;
    bool ok;
    if (MODE == kById) {
      p = ic;
      vi = ic;
      ok = in && ic < limit;
    } else {
      const int blk = __ldg(map + (ic >> 3));
      p = (int64_t)(blk < 0 ? 0 : blk) * kBlock + (ic & 7);
      ok = in && blk >= 0 && p < limit;
      vi = MODE == kMapSlot ? ic : (p < val_len ? p : val_len - 1);
    }
    const float v = __ldg(vals + vi);
    pos = (int32_t)p;
    return ok ? float_key(v) : 0u;
  }
  // position of element i (i < n_elems, a candidate)
  __device__ __forceinline__ int32_t pos_of(int64_t i) const {
    if (MODE == kById) return (int32_t)i;
    return __ldg(map + (i >> 3)) * kBlock + (int32_t)(i & 7);
  }
};

struct SmemView {  // elements in shared memory; key 0 marks a non-candidate
  const uint32_t *key;
  const int32_t *pos;
  int64_t n_elems;
  __device__ __forceinline__ uint32_t get(int64_t i, int32_t &p) const {
    const bool in = i < n_elems;
    p = pos[in ? i : 0];
    return in ? key[i] : 0u;
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

struct TopkShared {
  uint32_t red[2][8][kTopkWarps];
  uint32_t seg_a[kTopkWarps], seg_b[kTopkWarps];
  uint32_t s_a, s_b;
  uint32_t hist[8][256];
  uint32_t bcast[2];
  __align__(16) uint32_t hist11[2][2048];  // radix11_kth (zero between uses)
  uint32_t tab[512];
  uint32_t rsc[68];  // radix11_kth scratch
};

constexpr int kClBits = 11;  // radix digit width of the register and shared-memory selections
constexpr int kClBins = 1 << kClBits;

// Inclusive scan over the 1024 threads of the block (ends with a barrier, so wsum is free).
__device__ __forceinline__ uint32_t block_incl_scan_1024(uint32_t v, uint32_t *wsum) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t inc = warp_incl_scan(v);
  if (lane == 31) wsum[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    const uint32_t t = wsum[lane];
    wsum[lane] = warp_incl_scan(t) - t;
  }
  __syncthreads();
  inc += wsum[wid];
  __syncthreads();
  return inc;
}

// Exclusive prefix of tab[0 .. count) in place (count <= 32 * MAXPER), by warp 0 alone; the sum
// goes to *total.  Callers put a barrier before (table complete) and after (results visible).
template <int MAXPER>
__device__ __forceinline__ void warp0_excl_scan_table(uint32_t *tab, int count, uint32_t *total) {
  const int lane = threadIdx.x & 31;
  const int per = (count + 31) / 32;
  uint32_t v[MAXPER], sum = 0u;
#pragma unroll
  for (int i = 0; i < MAXPER; ++i) {
    const int idx = lane * per + i;
    v[i] = (i < per && idx < count) ? tab[idx] : 0u;
    sum += v[i];
  }
  const uint32_t inc = warp_incl_scan(sum);
  uint32_t run = inc - sum;
#pragma unroll
  for (int i = 0; i < MAXPER; ++i) {
    const int idx = lane * per + i;
    if (i < per && idx < count) {
      tab[idx] = run;
      run += v[i];
    }
  }
  if (lane == 31 && total) *total = inc;
}

// k-th largest (1 <= k <= number of candidates) of the keys this block visits: visit(f) calls
// f(key) for each of the calling thread's keys (0 = not a candidate); all candidates lie in
// [lo, hi].  11-bit digits below the leading bits lo and hi share: a shared histogram per digit
// (atomics), a block-wide scan of its 2,048 bins from the top.  Once at most 32 keys remain in
// play, one warp ranks them directly instead of further digits.  hist[0] is zero on entry and
// both buffers are zero on return; sc is scratch for 2 * 32 + 4 words.  need = k - #(keys > T).
// Block size 1024.
template <class Visit>
__device__ uint32_t radix11_kth(Visit visit, uint32_t k, uint32_t lo, uint32_t hi,
                                uint32_t (*hist)[kClBins], uint32_t *sc, uint32_t &need) {
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t *wsum = sc, *small = sc + 32, *bc = sc + 64;
  int b = (lo == hi) ? 0 : 32 - __clz(lo ^ hi);
  uint32_t T = b >= 32 ? 0u : (hi & ~((1u << b) - 1u));
  uint32_t rem = k;
  uint32_t in_play = 0xFFFFFFFFu;  // keys in play before the digit (unknown at first)
  int pb = 0;
  while (b > 0) {
    const int hs = b;  // keys in play share T's bits at and above hs
    if (in_play <= 32u) {
      // gather the (at most 32) keys in play, rank them in one warp
      if (tid == 0) bc[3] = 0u;
      __syncthreads();
      const uint32_t Tc = T;
      visit([&](uint32_t key) {
        if (key != 0u && (hs >= 32 || (key >> hs) == (Tc >> hs))) small[atomicAdd(&bc[3], 1u)] = key;
      });
      __syncthreads();
      if (tid < 32) {
        const uint32_t cnt = bc[3];
        const uint32_t mine = (uint32_t)lane < cnt ? small[lane] : 0u;
        uint32_t g = 0u, e = 0u;
        for (uint32_t j = 0; j < cnt; ++j) {
          const uint32_t x = small[j];
          g += x > mine;
          e += x == mine;
        }
        // the key with g < rem <= g + e (equal keys agree)
        if ((uint32_t)lane < cnt && g < rem && rem <= g + e) {
          bc[0] = mine;
          bc[1] = g;
        }
      }
      __syncthreads();
      T = bc[0];
      rem -= bc[1];
      break;
    }
    const int w = b >= kClBits ? kClBits : b;
    b -= w;
    const int s = b;
    uint32_t *h = hist[pb];
    const uint32_t Tc = T;
    visit([&](uint32_t key) {
      if (key != 0u && (hs >= 32 || (key >> hs) == (Tc >> hs)))
        atomicAdd(&h[(key >> s) & ((1u << w) - 1u)], 1u);
    });
    __syncthreads();
    const int hb0 = kClBins - 1 - 2 * tid, hb1 = hb0 - 1;
    const uint32_t c0 = h[hb0], c1 = h[hb1];
    const uint32_t inc = block_incl_scan_1024(c0 + c1, wsum), exc = inc - c0 - c1;
    h[hb0] = 0u;  // every read of this buffer happened before the scan's barriers
    h[hb1] = 0u;
    if (exc < rem && inc >= rem) {  // exactly one thread: the keys in play number >= rem
      const bool first = exc + c0 >= rem;
      bc[0] = (uint32_t)(first ? hb0 : hb1);
      bc[1] = first ? exc : exc + c0;
      bc[2] = first ? c0 : c1;
    }
    __syncthreads();
    T |= bc[0] << s;
    rem -= bc[1];
    in_play = bc[2];
    __syncthreads();  // bc is rewritten by the next digit
    pb ^= 1;
  }
  need = rem;
  return T;
}

// Counts of candidates with key >= cand[j] (j < NT) over the view, block-wide.
template <int NT, class View>
__device__ void count_ge_n(const View &ev, int64_t n_elems, const uint32_t (&cand)[NT],
                           uint32_t (&cnt)[NT], TopkShared &sh, int &parity) {
  uint32_t c[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) c[j] = 0;
  for (int64_t base = 0; base < n_elems; base += (int64_t)kTopkThreads * kUnroll) {
    uint32_t keys[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      int32_t pos;
      keys[u] = ev.get(base + (int64_t)u * kTopkThreads + threadIdx.x, pos);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int j = 0; j < NT; ++j) c[j] += keys[u] >= cand[j];
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    c[j] = __reduce_add_sync(0xffffffffu, c[j]);
    if (lane == 0) sh.red[parity][j][wid] = c[j];
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < NT; ++j) cnt[j] = __reduce_add_sync(0xffffffffu, sh.red[parity][j][lane]);
  parity ^= 1;
}

// Shared-memory specialization: only the keys are read, only the n stored elements are visited.
template <int NT>
__device__ void count_ge_n(const SmemView &sv, int64_t n_elems, const uint32_t (&cand)[NT],
                           uint32_t (&cnt)[NT], TopkShared &sh, int &parity) {
  uint32_t c[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) c[j] = 0;
  const int n = (int)n_elems;
  for (int i0 = threadIdx.x; i0 < n; i0 += 4 * kTopkThreads) {
    uint32_t keys[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * kTopkThreads;
      keys[u] = i < n ? sv.key[i] : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int j = 0; j < NT; ++j) c[j] += keys[u] >= cand[j];
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    c[j] = __reduce_add_sync(0xffffffffu, c[j]);
    if (lane == 0) sh.red[parity][j][wid] = c[j];
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < NT; ++j) cnt[j] = __reduce_add_sync(0xffffffffu, sh.red[parity][j][lane]);
  parity ^= 1;
}

// Smallest and largest candidate key of the shared-memory set (block-wide).
__device__ __forceinline__ void key_range(const SmemView &sv, int64_t n_elems, TopkShared &sh,
                                          int &parity, uint32_t &kmin, uint32_t &kmax) {
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int i = threadIdx.x; i < (int)n_elems; i += kTopkThreads) {
    const uint32_t k = sv.key[i];
    if (k != 0u) {
      lo = min(lo, k);
      hi = max(hi, k);
    }
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  if (lane == 0) {
    sh.red[parity][0][wid] = lo;
    sh.red[parity][1][wid] = hi;
  }
  __syncthreads();
  kmin = __reduce_min_sync(0xffffffffu, sh.red[parity][0][lane]);
  kmax = __reduce_max_sync(0xffffffffu, sh.red[parity][1][lane]);
  parity ^= 1;
}

// The k-th largest key (1 <= k <= number of candidates), three bits per round.
template <class View>
__device__ uint32_t kth_largest(const View &ev, int64_t n_elems, uint32_t k, TopkShared &sh,
                                int &parity, uint32_t prefix = 0u, int b = 32) {
  // the answer is known to start with the top (32 - b) bits of `prefix`
  uint32_t T = b >= 32 ? 0u : (prefix & ~((1u << b) - 1u));
  while (b > 0) {
    const int w = b >= 3 ? 3 : b;
    b -= w;
    uint32_t cand[7], cnt[7];
#pragma unroll
    for (int j = 0; j < 7; ++j)  // candidates beyond this round's width never qualify
      cand[j] = (j + 1 < (1 << w)) ? (T | ((uint32_t)(j + 1) << b)) : 0xFFFFFFFFu;
    count_ge_n<7>(ev, n_elems, cand, cnt, sh, parity);
    uint32_t best = 0;
#pragma unroll
    for (int j = 0; j < 7; ++j)
      if (j + 1 < (1 << w) && cnt[j] >= k) best = j + 1;
    T |= best << b;
  }
  return T;
}

// Ordered emission of the elements with key > T, plus the first need_eq with key == T.
template <class View>
__device__ void ordered_emit(const View &ev, int64_t n_elems, uint32_t T, uint32_t need_eq,
                             TopkShared &sh, int32_t *o) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int64_t seg = ((n_elems + kTopkWarps - 1) / kTopkWarps + 31) / 32 * 32;
  const int64_t w0 = (int64_t)wid * seg, w1 = min(n_elems, w0 + seg);
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint32_t ngt = 0, neq = 0;
  for (int64_t b = w0; b < w1; b += 32 * kUnroll) {
    uint32_t keys[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = b + 32 * u + lane;
      int32_t pos;
      keys[u] = ev.get(i, pos);
      if (i >= w1) keys[u] = 0u;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      ngt += __popc(__ballot_sync(0xffffffffu, keys[u] != 0u && keys[u] > T));
      neq += __popc(__ballot_sync(0xffffffffu, keys[u] != 0u && keys[u] == T));
    }
  }
  if (lane == 0) {
    sh.seg_a[wid] = ngt;
    sh.seg_b[wid] = neq;
  }
  __syncthreads();
  if (wid == 0) {
    const uint32_t g = sh.seg_a[lane], e = sh.seg_b[lane];
    const uint32_t gi = warp_incl_scan(g), ei = warp_incl_scan(e);
    sh.seg_a[lane] = gi - g;
    sh.seg_b[lane] = ei - e;
  }
  __syncthreads();
  uint32_t gt_r = sh.seg_a[wid], eq_r = sh.seg_b[wid];
  for (int64_t b = w0; b < w1; b += 32 * kUnroll) {
    uint32_t keys[kUnroll];
    int32_t poss[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = b + 32 * u + lane;
      keys[u] = ev.get(i, poss[u]);
      if (i >= w1) keys[u] = 0u;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const bool gt = keys[u] != 0u && keys[u] > T, eq = keys[u] != 0u && keys[u] == T;
      const uint32_t bgt = __ballot_sync(0xffffffffu, gt), beq = __ballot_sync(0xffffffffu, eq);
      const uint32_t my_gt = gt_r + __popc(bgt & lt_mask), my_eq = eq_r + __popc(beq & lt_mask);
      if (gt || (eq && my_eq < need_eq)) o[my_gt + min(my_eq, need_eq)] = poss[u];
      gt_r += __popc(bgt);
      eq_r += __popc(beq);
    }
  }
}

// k-th largest of n keys held in shared memory (key 0 = not a candidate), by radix select over
// the low b bits (the candidates all share the bits of `prefix` above them): 8-bit digits,
// histograms privatised per warp group (8 sub-histograms of 256 bins, summed per bin), a warp
// scan over the 256 bins from the top.  Returns T; *need_eq = how many keys equal to T are in
// the Top-k (k - #keys > T).  Works for any block size that is a multiple of 32 (<= 1024).
__device__ uint32_t kth_radix(const uint32_t *keys, int n, uint32_t k, uint32_t prefix, int b,
                              uint32_t (*hist)[256], uint32_t *bcast, uint32_t *need_eq) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int nthr = blockDim.x, nwarp = nthr >> 5;
  const int sub = wid & 7;
  uint32_t T = b >= 32 ? 0u : (prefix & ~((1u << b) - 1u));
  uint32_t rem = k;
  while (b > 0) {
    const int w = b >= 8 ? 8 : b;
    b -= w;
    const int shift = b;
    const int hi_shift = shift + w;  // keys still in play share T's bits at and above hi_shift
    for (int i = tid; i < 8 * 256; i += nthr) (&hist[0][0])[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += nthr) {
      const uint32_t key = keys[i];
      const bool in = key != 0u && (hi_shift >= 32 || (key >> hi_shift) == (T >> hi_shift));
      if (in) atomicAdd(&hist[sub][(key >> shift) & ((1u << w) - 1u)], 1u);
    }
    __syncthreads();
    if (wid == 0) {  // lane l owns bins 255-8l .. 248-8l (descending digit order)
      uint32_t c[8], s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int bin = 255 - 8 * lane - j;
        uint32_t t = 0;
#pragma unroll
        for (int g = 0; g < 8; ++g) t += hist[g][bin];
        c[j] = t;
        s += t;
      }
      const uint32_t inc = warp_incl_scan(s), before = inc - s;
      // the lane whose bins cross rem (at most one)
      if (before < rem && inc >= rem) {
        uint32_t acc = before;
        int j = 0;
        for (; j < 8; ++j) {
          if (acc + c[j] >= rem) break;
          acc += c[j];
        }
        bcast[0] = (uint32_t)(255 - 8 * lane - j);
        bcast[1] = acc;
      }
    }
    __syncthreads();
    T |= bcast[0] << shift;
    rem -= bcast[1];
    __syncthreads();
    (void)nwarp;
  }
  *need_eq = rem;
  return T;
}

template <class View>
__device__ __forceinline__ void start_bits(const View &, int64_t, TopkShared &, int &,
                                           uint32_t &prefix, int &b) {
  prefix = 0u;
  b = 32;
}
__device__ __forceinline__ void start_bits(const SmemView &sv, int64_t n, TopkShared &sh,
                                           int &parity, uint32_t &prefix, int &b) {
  uint32_t kmin, kmax;
  key_range(sv, n, sh, parity, kmin, kmax);
  prefix = kmax;
  b = (kmin == kmax) ? 0 : 32 - __clz(kmin ^ kmax);  // bits below the shared leading ones
}

// Shared-memory set (at most 16,384 elements in index order, 1024 threads; sh.hist11 zero on
// entry and on return): count and range, the k-th largest key by radix11_kth, then the ordered
// emission -- per (round, warp) counts of the keys > T and == T, one block scan, and every
// selected element's output slot from its ballots.
__device__ void select_and_emit(const SmemView &sv, int64_t n_elems, int topk, TopkShared &sh,
                                int &parity, int32_t *o) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int m = (int)n_elems;
  uint32_t lo = 0xFFFFFFFFu, hi = 0u, cnt = 0u;
  for (int i = tid; i < m; i += kTopkThreads) {
    const uint32_t k = sv.key[i];
    if (k != 0u) {
      lo = min(lo, k);
      hi = max(hi, k);
      ++cnt;
    }
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  if (lane == 0) {
    sh.red[parity][0][wid] = lo;
    sh.red[parity][1][wid] = hi;
    sh.red[parity][2][wid] = cnt;
  }
  __syncthreads();
  lo = __reduce_min_sync(0xffffffffu, sh.red[parity][0][lane]);
  hi = __reduce_max_sync(0xffffffffu, sh.red[parity][1][lane]);
  cnt = __reduce_add_sync(0xffffffffu, sh.red[parity][2][lane]);
  parity ^= 1;
  const uint32_t k_eff = min((uint32_t)topk, cnt);
  uint32_t T = 0u, need = 0u;  // k_eff == cnt: every candidate
  if (k_eff < cnt)
    T = radix11_kth(
        [&](auto f) {
          for (int i = tid; i < m; i += kTopkThreads) f(sv.key[i]);
        },
        k_eff, lo, hi, sh.hist11, sh.rsc, need);
  const int rounds = (m + kTopkThreads - 1) / kTopkThreads;  // <= 16
  for (int rr = 0; rr < rounds; ++rr) {
    const int i = rr * kTopkThreads + tid;
    const uint32_t kk = i < m ? sv.key[i] : 0u;
    const uint32_t a = __popc(__ballot_sync(0xffffffffu, kk > T));
    const uint32_t e = __popc(__ballot_sync(0xffffffffu, kk == T && kk != 0u));
    if (lane == 0) sh.tab[rr * 32 + wid] = a | (e << 16);
  }
  __syncthreads();
  if (wid == 0) warp0_excl_scan_table<16>(sh.tab, rounds * 32, nullptr);
  __syncthreads();
  const uint32_t lt = (1u << lane) - 1u;
  for (int rr = 0; rr < rounds; ++rr) {
    const int i = rr * kTopkThreads + tid;
    const uint32_t kk = i < m ? sv.key[i] : 0u;
    const bool gt = kk > T, eq = kk == T && kk != 0u;
    const uint32_t bgt = __ballot_sync(0xffffffffu, gt), beq = __ballot_sync(0xffffffffu, eq);
    const uint32_t t = sh.tab[rr * 32 + wid];
    const uint32_t my_gt = (t & 0xFFFFu) + __popc(bgt & lt);
    const uint32_t my_eq = (t >> 16) + __popc(beq & lt);
    if (gt || (eq && my_eq < need)) o[my_gt + min(my_eq, need)] = sv.pos[i];
  }
  for (int i = (int)k_eff + tid; i < topk; i += kTopkThreads) o[i] = -1;
}

template <class View>
__device__ void select_and_emit(const View &ev, int64_t n_elems, int topk, TopkShared &sh,
                                int &parity, int32_t *o) {
  uint32_t cand1[1] = {1u}, nv[1];
  count_ge_n<1>(ev, n_elems, cand1, nv, sh, parity);
  const uint32_t k_eff = min((uint32_t)topk, nv[0]);
  if (k_eff > 0) {
    uint32_t prefix;
    int b0;
    start_bits(ev, n_elems, sh, parity, prefix, b0);
    const uint32_t T = kth_largest(ev, n_elems, k_eff, sh, parity, prefix, b0);
    uint32_t n_gt = 0;
    if (T != 0xFFFFFFFFu) {
      uint32_t c[1] = {T + 1u}, r[1];
      count_ge_n<1>(ev, n_elems, c, r, sh, parity);
      n_gt = r[0];
    }
    ordered_emit(ev, n_elems, T, k_eff - n_gt, sh, o);
  }
  for (int i = (int)k_eff + threadIdx.x; i < topk; i += kTopkThreads) o[i] = -1;
}

template <int MODE>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(
    const float *__restrict__ vals, int64_t stride, int64_t n_elems,
    const int32_t *__restrict__ map, int64_t map_stride, int unit,
    const int32_t *__restrict__ q_vis, int topk, int32_t *__restrict__ out) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t topk_smem[];
  uint32_t *skey = reinterpret_cast<uint32_t *>(topk_smem);
  int32_t *spos = reinterpret_cast<int32_t *>(topk_smem + (size_t)kSmemCap * 4);
  __shared__ TopkShared sh;
  int parity = 0;

  const int n = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  for (int i = tid; i < 2 * 2048; i += kTopkThreads) (&sh.hist11[0][0])[i] = 0u;
  int32_t *o = out + (int64_t)n * topk;
  if (n_elems <= 0) {
    for (int i = tid; i < topk; i += kTopkThreads) o[i] = -1;
    return;
  }
  const int64_t V = q_vis[n];
  ElemView<MODE> ev;
  ev.vals = vals + (int64_t)n * stride;
  ev.val_len = stride > 0 ? stride : 1;
  ev.map = map ? map + (int64_t)n * map_stride : nullptr;
  ev.n_elems = n_elems;
  ev.limit = MODE == kById ? (V + unit - 1) / unit : V;

  if (n_elems <= kSmemCap) {
    // ---- small: copy everything (non-candidates -> key 0), keep index order
    for (int64_t base = 0; base < n_elems; base += (int64_t)kTopkThreads * kUnroll) {
      uint32_t k[kUnroll];
      int32_t p[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) k[u] = ev.get(base + (int64_t)u * kTopkThreads + tid, p[u]);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = base + (int64_t)u * kTopkThreads + tid;
        if (i < n_elems) {
          skey[i] = k[u];
          spos[i] = p[u];
        }
      }
    }
    __syncthreads();
    SmemView sv{skey, spos, n_elems};
    select_and_emit(sv, n_elems, topk, sh, parity, o);
    return;
  }

  // ---- large: sample -> threshold estimate
  const int64_t step = n_elems / kSample;  // >= 2
  {
    uint32_t k[kSample / kTopkThreads];
#pragma unroll
    for (int u = 0; u < kSample / kTopkThreads; ++u) {
      int32_t p;
      k[u] = ev.get((int64_t)(u * kTopkThreads + tid) * step, p);
    }
#pragma unroll
    for (int u = 0; u < kSample / kTopkThreads; ++u) {
      skey[u * kTopkThreads + tid] = k[u];
      spos[u * kTopkThreads + tid] = 0;
    }
  }
  __syncthreads();
  SmemView smp{skey, spos, kSample};
  const int64_t r_want = (int64_t)topk * kSample * 8 / (n_elems * 5) + 16;  // ~1.6 K kept
  const uint32_t r = (uint32_t)(r_want < kSample ? r_want : kSample);
  uint32_t t_est = 1u;  // every candidate key is >= 1
  {
    uint32_t c1[1] = {1u}, nvs[1];
    count_ge_n<1>(smp, kSample, c1, nvs, sh, parity);
    if (nvs[0] >= r) {
      uint32_t kmin, kmax, need_eq;
      key_range(smp, kSample, sh, parity, kmin, kmax);
      const int b = (kmin == kmax) ? 0 : 32 - __clz(kmin ^ kmax);
      t_est = kth_radix(skey, kSample, r, kmax, b, sh.hist, sh.bcast, &need_eq);
    }
  }
  __syncthreads();  // the sample is no longer needed

  // ---- one sweep: each warp appends its candidates >= t_est (index order) to its slots
  const int64_t seg = ((n_elems + kTopkWarps - 1) / kTopkWarps + 31) / 32 * 32;
  const int64_t w0 = (int64_t)wid * seg, w1 = min(n_elems, w0 + seg);
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint32_t nval = 0, wr = 0;
  for (int64_t b = w0; b < w1; b += 32 * kUnroll) {
    uint32_t keys[kUnroll];
    int32_t poss[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = b + 32 * u + lane;
      keys[u] = ev.get(i, poss[u]);
      if (i >= w1) keys[u] = 0u;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      nval += keys[u] != 0u;
      const bool take = keys[u] >= t_est;  // t_est >= 1 excludes non-candidates
      const uint32_t bt = __ballot_sync(0xffffffffu, take);
      const uint32_t slot = wr + __popc(bt & lt_mask);
      if (take && slot < (uint32_t)kWarpCap) {
        skey[wid * kWarpCap + slot] = keys[u];
        spos[wid * kWarpCap + slot] = poss[u];
      }
      wr += __popc(bt);
    }
  }
  nval = __reduce_add_sync(0xffffffffu, nval);
  if (lane == 0) {
    sh.seg_a[wid] = nval;
    sh.seg_b[wid] = wr;
  }
  __syncthreads();
  if (wid == 0) {
    const uint32_t a = sh.seg_a[lane], b = sh.seg_b[lane];
    const uint32_t ai = warp_incl_scan(a), bi = warp_incl_scan(b);
    const uint32_t over = __ballot_sync(0xffffffffu, b > (uint32_t)kWarpCap);
    sh.seg_b[lane] = bi - b;  // exclusive offsets of each warp's kept run
    if (lane == 31) {
      sh.s_a = ai;                              // candidates
      sh.s_b = over ? (bi | 0x80000000u) : bi;  // kept (+ overflow flag)
    }
  }
  __syncthreads();
  const uint32_t total_valid = sh.s_a, kept = sh.s_b & 0x7FFFFFFFu;
  const bool overflow = (sh.s_b & 0x80000000u) != 0u;
  const uint32_t k_eff = min((uint32_t)topk, total_valid);
  if (overflow || kept < k_eff) {  // the estimate missed: select over global memory
    select_and_emit(ev, n_elems, topk, sh, parity, o);
    return;
  }
  // compact the warp runs into one index-ordered array (read everything, then write)
  {
    const uint32_t my_cnt = wr, my_off = sh.seg_b[wid];
    uint32_t kk[kWarpCap / 32];
    int32_t pp[kWarpCap / 32];
#pragma unroll
    for (int e = 0; e < kWarpCap / 32; ++e) {
      const uint32_t s = e * 32 + lane;
      kk[e] = s < my_cnt ? skey[wid * kWarpCap + s] : 0u;
      pp[e] = s < my_cnt ? spos[wid * kWarpCap + s] : 0;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < kWarpCap / 32; ++e) {
      const uint32_t s = e * 32 + lane;
      if (s < my_cnt) {
        skey[my_off + s] = kk[e];
        spos[my_off + s] = pp[e];
      }
    }
  }
  __syncthreads();
  SmemView sv{skey, spos, (int64_t)kept};
  select_and_emit(sv, kept, topk, sh, parity, o);
}

// ------------------------------------------------------------------------------------------
// Few queries over many elements: spread the sweep over many SMs.
//   topk_filter_kernel  grid (chunks of 4096 elements, queries): every CTA derives the same
//                       threshold T_est from the same strided sample of 1024 keys, then writes
//                       its chunk's candidates with key >= T_est, in index order, to the
//                       chunk's workspace slots, with the chunk's kept and candidate counts.
//   topk_select_kernel  one CTA per query: gathers the kept elements of all chunks (index order)
//                       into shared memory and selects there; if the estimate kept fewer than
//                       K, or more than fit, it selects over global memory instead.
// ------------------------------------------------------------------------------------------
constexpr int kTkChunk = 4096;
constexpr int kFilterThreads = 256;
constexpr int kFilterSample = kFilterThreads;  // one sampled key per thread

struct ChunkWs {  // per query: [n_chunks][kTkChunk] keys, positions, then [n_chunks] counts
  uint32_t *keys;
  int32_t *pos;
  uint32_t *kept;
  uint32_t *valid;
};

__device__ __forceinline__ ChunkWs chunk_ws(void *ws, int n, int n_chunks) {
  const size_t per_q = (size_t)n_chunks * kTkChunk * 8 + (size_t)n_chunks * 8;
  char *b = static_cast<char *>(ws) + (size_t)n * per_q;
  ChunkWs c;
  c.keys = reinterpret_cast<uint32_t *>(b);
  c.pos = reinterpret_cast<int32_t *>(b + (size_t)n_chunks * kTkChunk * 4);
  c.kept = reinterpret_cast<uint32_t *>(b + (size_t)n_chunks * kTkChunk * 8);
  c.valid = c.kept + n_chunks;
  return c;
}

template <int MODE>
__global__ void __launch_bounds__(kFilterThreads) topk_filter_kernel(
    const float *__restrict__ vals, int64_t stride, int64_t n_elems,
    const int32_t *__restrict__ map, int64_t map_stride, int unit,
    const int32_t *__restrict__ q_vis, int topk, void *ws) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t ks[kFilterSample];
  __shared__ uint32_t red[8][kFilterThreads / 32];
  __shared__ uint32_t wcnt[kFilterThreads / 32];
  __shared__ uint32_t t_sh;
  const int c = blockIdx.x, n = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int n_chunks = gridDim.x;
  const int64_t V = q_vis[n];
  ElemView<MODE> ev;
  ev.vals = vals + (int64_t)n * stride;
  ev.val_len = stride > 0 ? stride : 1;
  ev.map = map ? map + (int64_t)n * map_stride : nullptr;
  ev.n_elems = n_elems;
  ev.limit = MODE == kById ? (V + unit - 1) / unit : V;
  // the shared threshold estimate: the r-th largest of a strided sample of the whole array,
  // found by the exact rank of every sampled key (same sample and result in every CTA);
  // r = the expected number of sampled keys in the Top-K + 2.5 standard deviations + 3
  const int64_t step = n_elems / kFilterSample;  // >= 2 (n_elems > 2 * kFilterSample)
  {
    int32_t p;
    ks[tid] = ev.get((int64_t)tid * step, p);
  }
  if (tid == 0) t_sh = 1u;  // every candidate, unless a sampled key qualifies below
  const uint32_t sv = __syncthreads_count(ks[tid] != 0u);
  const float mu = fminf((float)sv, (float)topk * (float)kFilterSample / (float)n_elems);
  const uint32_t r = (uint32_t)ceilf(mu + 2.5f * sqrtf(mu) + 3.0f);
  if (r <= sv) {
    const uint32_t mine = ks[tid];
    uint32_t g = 0u, e = 0u;
#pragma unroll 16
    for (int j = 0; j < kFilterSample; ++j) {
      const uint32_t x = ks[j];
      g += x > mine;
      e += x == mine;
    }
    if (mine != 0u && g < r && r <= g + e) t_sh = mine;  // equal keys write the same value
  }
  __syncthreads();
  const uint32_t t_est = t_sh;
  // this chunk: warp w owns elements [w*512, w*512+512) of it, 16 per lane, all loads in flight
  const int64_t c0 = (int64_t)c * kTkChunk + (int64_t)wid * (kTkChunk / 8);
  constexpr int kPer = kTkChunk / kFilterThreads;  // 16
  uint32_t keys[kPer];
  int32_t poss[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) keys[u] = ev.get(c0 + 32 * u + lane, poss[u]);
  uint32_t nval = 0, nkeep = 0;
  uint32_t take_mask[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    nval += keys[u] != 0u;
    take_mask[u] = __ballot_sync(0xffffffffu, keys[u] >= t_est);
    nkeep += __popc(take_mask[u]);
  }
  nval = __reduce_add_sync(0xffffffffu, nval);
  if (lane == 0) {
    wcnt[wid] = nkeep;
    red[0][wid] = nval;
  }
  __syncthreads();
  uint32_t off = 0, tot_keep = 0, tot_val = 0;
#pragma unroll
  for (int w = 0; w < kFilterThreads / 32; ++w) {
    off += (w < wid) ? wcnt[w] : 0u;
    tot_keep += wcnt[w];
    tot_val += red[0][w];
  }
  ChunkWs cw = chunk_ws(ws, n, n_chunks);
  uint32_t *okeys = cw.keys + (size_t)c * kTkChunk;
  int32_t *opos = cw.pos + (size_t)c * kTkChunk;
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    if (keys[u] >= t_est) {
      const uint32_t slot = off + __popc(take_mask[u] & lt_mask);
      okeys[slot] = keys[u];
      opos[slot] = poss[u];
    }
    off += __popc(take_mask[u]);
  }
  if (tid == 0) {
    cw.kept[c] = tot_keep;
    cw.valid[c] = tot_val;
  }
}

template <int MODE>
__global__ void __launch_bounds__(kTopkThreads) topk_select_kernel(
    const float *__restrict__ vals, int64_t stride, int64_t n_elems,
    const int32_t *__restrict__ map, int64_t map_stride, int unit,
    const int32_t *__restrict__ q_vis, int topk, int32_t *__restrict__ out, const void *ws,
    int n_chunks) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t topk_smem[];
  uint32_t *skey = reinterpret_cast<uint32_t *>(topk_smem);
  int32_t *spos = reinterpret_cast<int32_t *>(topk_smem + (size_t)kSmemCap * 4);
  __shared__ TopkShared sh;
  __shared__ uint32_t coff[1025];
  int parity = 0;
  const int n = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  for (int i = tid; i < 2 * 2048; i += kTopkThreads) (&sh.hist11[0][0])[i] = 0u;
  int32_t *o = out + (int64_t)n * topk;
  ChunkWs cw = chunk_ws(const_cast<void *>(ws), n, n_chunks);
  // chunk offsets (n_chunks <= 1024): block-wide exclusive scan of the kept counts
  const uint32_t kc = tid < n_chunks ? cw.kept[tid] : 0u;
  const uint32_t vc = tid < n_chunks ? cw.valid[tid] : 0u;
  const uint32_t inc = warp_incl_scan(kc);
  const uint32_t vtot_w = __reduce_add_sync(0xffffffffu, vc);
  if (lane == 31) sh.seg_a[wid] = inc;
  if (lane == 0) sh.seg_b[wid] = vtot_w;
  __syncthreads();
  if (wid == 0) {
    const uint32_t a = sh.seg_a[lane];
    const uint32_t ai = warp_incl_scan(a);
    const uint32_t vt = __reduce_add_sync(0xffffffffu, sh.seg_b[lane]);
    sh.seg_a[lane] = ai - a;
    if (lane == 31) {
      sh.s_a = ai;  // kept
      sh.s_b = vt;  // candidates
    }
  }
  __syncthreads();
  if (tid < n_chunks) coff[tid] = sh.seg_a[wid] + inc - kc;
  const uint32_t kept = sh.s_a, total_valid = sh.s_b;
  const uint32_t k_eff = min((uint32_t)topk, total_valid);
  __syncthreads();
  if (kept >= k_eff && kept <= (uint32_t)kSmemCap) {
    if (tid == 0) coff[n_chunks] = kept;
    __syncthreads();
    // warp w copies chunks w, w + 32, ... to their offsets (index order is chunk order)
    for (int c = wid; c < n_chunks; c += kTopkWarps) {
      const int cnt = (int)(coff[c + 1] - coff[c]), dst = (int)coff[c];
      const uint32_t *ck = cw.keys + (size_t)c * kTkChunk;
      const int32_t *cp = cw.pos + (size_t)c * kTkChunk;
      for (int j0 = 0; j0 < cnt; j0 += 32 * 4) {
        uint32_t kk[4];
        int32_t pp[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + u * 32 + lane;
          const int jc = j < cnt ? j : 0;
          kk[u] = ck[jc];
          pp[u] = cp[jc];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + u * 32 + lane;
          if (j < cnt) {
            skey[dst + j] = kk[u];
            spos[dst + j] = pp[u];
          }
        }
      }
    }
    __syncthreads();
    SmemView sv{skey, spos, (int64_t)kept};
    select_and_emit(sv, kept, topk, sh, parity, o);
    return;
  }
  const int64_t V = q_vis[n];  // the estimate missed: select over global memory
  ElemView<MODE> ev;
  ev.vals = vals + (int64_t)n * stride;
  ev.val_len = stride > 0 ? stride : 1;
  ev.map = map ? map + (int64_t)n * map_stride : nullptr;
  ev.n_elems = n_elems;
  ev.limit = MODE == kById ? (V + unit - 1) / unit : V;
  select_and_emit(ev, n_elems, topk, sh, parity, o);
}

// ------------------------------------------------------------------------------------------
// Register path: one CTA per query over at most 16,384 elements.  Thread tid holds, in round v
// (v < 4), the four consecutive elements 4096 v + 4 tid + j (j < 4): one 16-byte value load and
// one block-list load per round (scalar loads only at a ragged end or an unaligned row).
//   1. candidate count, smallest and largest key (block reduction);
//   2. threshold estimate t_lo: the r-th largest of 128 keys sampled across the elements (exact
//      rank of every sample: 1024 threads x 16 comparisons), r = the expected number of sampled
//      keys in the Top-K plus 2.5 standard deviations plus 3, so that at least K keys are >= t_lo
//      with high probability;
//   3. the keys >= t_lo and their positions are compacted in index order into shared memory
//      (per-round warp scans, one block scan); if they are fewer than K (the estimate was too
//      high) or more than the shared-memory capacity, step 4 runs over all keys in registers;
//   4. radix select of the k-th largest key T, 11-bit digits, one shared histogram per digit;
//   5. ordered emission of the keys > T and the first need = K - #(> T) keys == T.
constexpr int kRgThreads = 1024;
constexpr int kRgRounds = 4;
constexpr int kRgSpan = kRgThreads * 4 * kRgRounds;  // 16,384
constexpr int kRgSample = 128;
constexpr int kRgKeepCap = 8192;
static_assert(kRgKeepCap / kRgThreads >= kRgRounds, "round table");

struct RgShared {
  __align__(16) uint32_t hist[2][kClBins];
  uint32_t tab[(kRgKeepCap / kRgThreads) * 32];  // per (round, warp); 8 rounds of the compacted set
  uint32_t rsc[68];  // radix11_kth scratch
  uint32_t red[3][32];
  uint32_t samp[kRgSample];
  uint32_t sg[kRgSample], se[kRgSample];
  uint32_t bc[8];
  uint32_t kkey[kRgKeepCap];
  int32_t kpos[kRgKeepCap];
};
constexpr size_t kRgSmem = sizeof(RgShared);

// Keys (0 = not a candidate) and positions of elements e0 .. e0+3 (e0 = 4096 v + 4 tid).
template <int MODE>
__device__ __forceinline__ void load4(const ElemView<MODE> &ev, int e0, bool vec,
                                      uint32_t (&k)[4], int32_t (&pos)[4]) {
  const int n = (int)ev.n_elems;
  int blk = 0;
  if (MODE != kById) blk = e0 < n ? __ldg(ev.map + (e0 >> 3)) : -1;
  int64_t vbase;  // value index of element e0
  if (MODE == kMapPos) vbase = (int64_t)(blk < 0 ? 0 : blk) * kBlock + (e0 & 7);
  else vbase = e0;
  const bool full = e0 + 3 < n;
  float v[4];
  if (vec && full && (MODE != kMapPos || vbase + 3 < ev.val_len)) {
    const float4 f = __ldg(reinterpret_cast<const float4 *>(ev.vals + vbase));
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int64_t vi = vbase + j;
      const int64_t hi = MODE == kMapPos ? ev.val_len - 1 : (int64_t)n - 1;
      vi = vi < hi ? vi : hi;
      v[j] = __ldg(ev.vals + vi);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = e0 + j;
    int64_t p;
    bool ok;
    if (MODE == kById) {
      p = e;
      ok = e < n && p < ev.limit;
    } else {
      p = (int64_t)blk * kBlock + (e & 7);
      ok = e < n && blk >= 0 && p < ev.limit;
    }
    pos[j] = (int32_t)p;
    k[j] = ok ? float_key(v[j]) : 0u;
  }
}

// Exclusive offsets, in index order, of this thread's flagged elements of round v: the warp
// scan of per-thread counts plus the block-wide prefix in tab (filled by the caller).
__device__ __forceinline__ uint32_t warp_excl_scan(uint32_t c) {
  return warp_incl_scan(c) - c;
}

template <int MODE>
__global__ void __launch_bounds__(kRgThreads, 1) topk_reg_kernel(
    const float *__restrict__ vals, int64_t stride, int64_t n_elems,
    const int32_t *__restrict__ map, int64_t map_stride, int unit,
    const int32_t *__restrict__ q_vis, int topk, int32_t *__restrict__ out) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t rg_smem[];
  RgShared &sh = *reinterpret_cast<RgShared *>(rg_smem);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int n = blockIdx.x;
  const int64_t V = q_vis[n];
  ElemView<MODE> ev;
  ev.vals = vals + (int64_t)n * stride;
  ev.val_len = stride > 0 ? stride : 1;
  ev.map = map ? map + (int64_t)n * map_stride : nullptr;
  ev.n_elems = n_elems;
  ev.limit = MODE == kById ? (V + unit - 1) / unit : V;
  const bool vec = (reinterpret_cast<uintptr_t>(ev.vals) & 15u) == 0;
  uint32_t key[kRgRounds][4];
  {
    int32_t pdummy[kRgRounds][4];
#pragma unroll
    for (int v = 0; v < kRgRounds; ++v) load4(ev, 4096 * v + 4 * tid, vec, key[v], pdummy[v]);
  }
  sh.hist[0][tid] = 0u;
  sh.hist[0][tid + kRgThreads] = 0u;
  sh.hist[1][tid] = 0u;
  sh.hist[1][tid + kRgThreads] = 0u;
  if (tid < kRgSample) {
    sh.sg[tid] = 0u;
    sh.se[tid] = 0u;
  }
  // ---- 1. count and range
  uint32_t gmin, gmax, gcnt;
  {
    uint32_t lo = 0xFFFFFFFFu, hi = 0u, cnt = 0u;
#pragma unroll
    for (int v = 0; v < kRgRounds; ++v)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (key[v][j] != 0u) {
          lo = min(lo, key[v][j]);
          hi = max(hi, key[v][j]);
          ++cnt;
        }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    if (lane == 0) {
      sh.red[0][wid] = lo;
      sh.red[1][wid] = hi;
      sh.red[2][wid] = cnt;
    }
    // sample s (tid = 8 s): element 4096 ((s >> 2) & 3) + 4 tid + (s & 3)
    if ((tid & 7) == 0) {
      const int sidx = tid >> 3, vs = (sidx >> 2) & 3, js = sidx & 3;
      uint32_t x = 0u;
#pragma unroll
      for (int v = 0; v < kRgRounds; ++v)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (v == vs && j == js) x = key[v][j];
      sh.samp[sidx] = x;
    }
    __syncthreads();
    gmin = __reduce_min_sync(0xffffffffu, sh.red[0][lane]);
    gmax = __reduce_max_sync(0xffffffffu, sh.red[1][lane]);
    gcnt = __reduce_add_sync(0xffffffffu, sh.red[2][lane]);
  }
  const uint32_t k_eff = min((uint32_t)topk, gcnt);
  uint32_t T = 0u, need = 0u;  // k_eff == gcnt: every candidate (key > 0), none as "equal"
  int m = -1;                  // compacted count (-1: select straight from registers)
  if (k_eff < gcnt) {
    // ---- 2. threshold estimate from the sample
    {
      const int j = tid & (kRgSample - 1), q = tid / kRgSample;  // 8 slices of 16 samples
      const uint32_t sj = sh.samp[j];
      uint32_t g = 0u, e = 0u;
#pragma unroll
      for (int i = 0; i < kRgSample / 8; ++i) {
        const uint32_t x = sh.samp[q * (kRgSample / 8) + i];
        g += x > sj;
        e += x == sj;
      }
      atomicAdd(&sh.sg[j], g);
      atomicAdd(&sh.se[j], e);
    }
    const uint32_t sv = __syncthreads_count(tid < kRgSample && sh.samp[tid] != 0u);
    const float mu = (float)sv * (float)k_eff / (float)gcnt;
    const uint32_t r = (uint32_t)ceilf(mu + 2.5f * sqrtf(mu) + 3.0f);
    if (tid == 0) sh.bc[4] = 1u;  // keep every candidate unless a sample qualifies below
    __syncthreads();
    if (tid < kRgSample && r <= sv) {
      const uint32_t sj = sh.samp[tid], g = sh.sg[tid], e = sh.se[tid];
      if (sj != 0u && g < r && r <= g + e) sh.bc[4] = sj;  // the r-th largest sample
    }
    __syncthreads();
    const uint32_t t_lo = sh.bc[4];
    // ---- 3. compaction of the keys >= t_lo (index order)
    uint32_t cnt_v[kRgRounds];
#pragma unroll
    for (int v = 0; v < kRgRounds; ++v) {
      uint32_t c = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) c += key[v][j] >= t_lo && key[v][j] != 0u;
      cnt_v[v] = c;
      const uint32_t wt = __reduce_add_sync(0xffffffffu, c);
      if (lane == 0) sh.tab[v * 32 + wid] = wt;
    }
    __syncthreads();
    if (wid == 0) warp0_excl_scan_table<8>(sh.tab, kRgRounds * 32, &sh.bc[5]);
    __syncthreads();
    const uint32_t kept = sh.bc[5];
    if (kept >= k_eff && kept <= (uint32_t)kRgKeepCap) {
      uint32_t klo = 0xFFFFFFFFu;
#pragma unroll
      for (int v = 0; v < kRgRounds; ++v) {
        uint32_t slot = sh.tab[v * 32 + wid] + warp_excl_scan(cnt_v[v]);
        if (cnt_v[v]) {
          uint32_t kq[4];
          int32_t pq[4];
          // positions of the four elements (the block list is re-read from L1)
          {
            const int e0 = 4096 * v + 4 * tid;
            int blk = 0;
            if (MODE != kById) blk = __ldg(ev.map + (e0 >> 3));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              kq[j] = key[v][j];
              pq[j] = MODE == kById ? e0 + j : blk * kBlock + ((e0 + j) & 7);
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (kq[j] >= t_lo && kq[j] != 0u) {
              sh.kkey[slot] = kq[j];
              sh.kpos[slot] = pq[j];
              ++slot;
              klo = min(klo, kq[j]);
            }
        }
      }
      klo = __reduce_min_sync(0xffffffffu, klo);
      if (lane == 0) sh.red[0][wid] = klo;
      __syncthreads();
      klo = __reduce_min_sync(0xffffffffu, sh.red[0][lane]);
      m = (int)kept;
      // ---- 4. exact k-th largest over the compacted keys
      T = radix11_kth(
          [&](auto f) {
            for (int i = tid; i < m; i += kRgThreads) f(sh.kkey[i]);
          },
          k_eff, klo, gmax, sh.hist, sh.rsc, need);
    } else {
      T = radix11_kth(
          [&](auto f) {
#pragma unroll
            for (int v = 0; v < kRgRounds; ++v)
#pragma unroll
              for (int j = 0; j < 4; ++j) f(key[v][j]);
          },
          k_eff, gmin, gmax, sh.hist, sh.rsc, need);
    }
  }
  // ---- 5. ordered emission
  int32_t *o = out + (int64_t)n * topk;
  const uint32_t lt = (1u << lane) - 1u;
  if (m >= 0) {  // the compacted set, element i = rr * 1024 + tid (index order)
    const int rounds = (m + kRgThreads - 1) / kRgThreads;  // <= 8
    for (int rr = 0; rr < rounds; ++rr) {
      const int i = rr * kRgThreads + tid;
      const uint32_t kk = i < m ? sh.kkey[i] : 0u;
      const uint32_t a = __popc(__ballot_sync(0xffffffffu, kk > T));
      const uint32_t e = __popc(__ballot_sync(0xffffffffu, kk == T && kk != 0u));
      if (lane == 0) sh.tab[rr * 32 + wid] = a | (e << 16);
    }
    __syncthreads();
    if (wid == 0) warp0_excl_scan_table<8>(sh.tab, rounds * 32, nullptr);
    __syncthreads();
    for (int rr = 0; rr < rounds; ++rr) {
      const int i = rr * kRgThreads + tid;
      const uint32_t kk = i < m ? sh.kkey[i] : 0u;
      const bool gt = kk > T, eq = kk == T && kk != 0u;
      const uint32_t bgt = __ballot_sync(0xffffffffu, gt), beq = __ballot_sync(0xffffffffu, eq);
      const uint32_t t = sh.tab[rr * 32 + wid];
      const uint32_t my_gt = (t & 0xFFFFu) + __popc(bgt & lt);
      const uint32_t my_eq = (t >> 16) + __popc(beq & lt);
      if (gt || (eq && my_eq < need)) o[my_gt + min(my_eq, need)] = sh.kpos[i];
    }
  } else {  // straight from registers: per-round warp scans of (keys > T, keys == T) counts
    uint32_t c_v[kRgRounds];
#pragma unroll
    for (int v = 0; v < kRgRounds; ++v) {
      uint32_t a = 0u, e = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        a += key[v][j] > T;
        e += key[v][j] == T && key[v][j] != 0u;
      }
      c_v[v] = a | (e << 16);
      const uint32_t wt = __reduce_add_sync(0xffffffffu, c_v[v]);
      if (lane == 0) sh.tab[v * 32 + wid] = wt;
    }
    __syncthreads();
    if (wid == 0) warp0_excl_scan_table<8>(sh.tab, kRgRounds * 32, nullptr);
    __syncthreads();
#pragma unroll
    for (int v = 0; v < kRgRounds; ++v) {
      const uint32_t base = sh.tab[v * 32 + wid] + warp_excl_scan(c_v[v]);
      uint32_t my_gt = base & 0xFFFFu, my_eq = base >> 16;
      const int e0 = 4096 * v + 4 * tid;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t kk = key[v][j];
        const bool gt = kk > T, eq = kk == T && kk != 0u;
        if (gt || (eq && my_eq < need)) o[my_gt + min(my_eq, need)] = ev.pos_of(e0 + j);
        my_gt += gt;
        my_eq += eq;
      }
    }
  }
  for (int i = (int)k_eff + tid; i < topk; i += kRgThreads) o[i] = -1;
}

template <int MODE>
static cudaError_t launch_topk_reg(const float *vals, int64_t stride, int64_t n_elems,
                                   const int32_t *map, int64_t map_stride, int unit,
                                   const int32_t *q_vis, int nq, int topk, int32_t *out,
                                   cudaStream_t st) {
  cudaError_t e = set_smem_once(topk_reg_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kRgSmem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(topk_reg_kernel<MODE>, dim3(nq), dim3(kRgThreads), kRgSmem, st, vals, stride,
                 n_elems, map, map_stride, unit, q_vis, topk, out);
  note_launches(1);
  return e;
}

static bool topk_use_reg(int nq, int64_t n_elems) {
  (void)nq;  // one CTA per query, any number of queries
  return n_elems >= 1 && n_elems <= kRgSpan;
}

// The chunked two-kernel path serves few queries over many elements.
static bool topk_use_chunks(int nq, int64_t n_elems) {
  return !topk_use_reg(nq, n_elems) && nq <= 64 && n_elems > 2 * kFilterSample &&
         (n_elems + kTkChunk - 1) / kTkChunk <= 1024;
}

size_t topk_workspace_bytes(int nq, int64_t n_elems) {
  if (!topk_use_chunks(nq, n_elems)) return 0;
  const size_t n_chunks = (size_t)((n_elems + kTkChunk - 1) / kTkChunk);
  return (size_t)nq * (n_chunks * kTkChunk * 8 + n_chunks * 8);
}

template <int MODE>
static cudaError_t launch_topk_chunked(const float *vals, int64_t stride, int64_t n_elems,
                                       const int32_t *map, int64_t map_stride, int unit,
                                       const int32_t *q_vis, int nq, int topk, int32_t *out,
                                       void *ws, cudaStream_t st) {
  const int n_chunks = (int)((n_elems + kTkChunk - 1) / kTkChunk);
  cudaError_t e = launch_pdl(topk_filter_kernel<MODE>, dim3(n_chunks, nq), dim3(kFilterThreads),
                             0, st, vals, stride, n_elems, map, map_stride, unit, q_vis, topk,
                             ws);
  note_launches(1);
  if (e != cudaSuccess) return e;
  e = set_smem_once(topk_select_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                    (int)kTopkSmem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(topk_select_kernel<MODE>, dim3(nq), dim3(kTopkThreads), kTopkSmem, st, vals,
                 stride, n_elems, map, map_stride, unit, q_vis, topk, out, (const void *)ws,
                 n_chunks);
  note_launches(1);
  return e;
}

cudaError_t launch_topk(const float *vals, int64_t stride, int64_t n_elems, const int32_t *map,
                        int64_t map_stride, int unit, const int32_t *q_vis, int nq, int topk,
                        int32_t *out, cudaStream_t st, const float *pos_vals,
                        int64_t pos_stride, void *ws) {
  if (nq == 0) return cudaSuccess;
  if (topk_use_reg(nq, n_elems)) {
    if (!map)
      return launch_topk_reg<kById>(vals, stride, n_elems, nullptr, 0, unit, q_vis, nq, topk, out,
                                    st);
    if (pos_vals)
      return launch_topk_reg<kMapPos>(pos_vals, pos_stride, n_elems, map, map_stride, unit, q_vis,
                                      nq, topk, out, st);
    return launch_topk_reg<kMapSlot>(vals, stride, n_elems, map, map_stride, unit, q_vis, nq, topk,
                                     out, st);
  }
  if (ws && topk_use_chunks(nq, n_elems)) {
    if (!map)
      return launch_topk_chunked<kById>(vals, stride, n_elems, nullptr, 0, unit, q_vis, nq, topk,
                                        out, ws, st);
    if (pos_vals)
      return launch_topk_chunked<kMapPos>(pos_vals, pos_stride, n_elems, map, map_stride, unit,
                                          q_vis, nq, topk, out, ws, st);
    return launch_topk_chunked<kMapSlot>(vals, stride, n_elems, map, map_stride, unit, q_vis, nq,
                                         topk, out, ws, st);
  }
  cudaError_t e;
  if (!map) {
    e = set_smem_once(topk_kernel<kById>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                      (int)kTopkSmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(topk_kernel<kById>, dim3(nq), dim3(kTopkThreads), kTopkSmem, st, vals,
                   stride, n_elems, (const int32_t *)nullptr, (int64_t)0, unit, q_vis, topk, out);
  } else if (pos_vals) {
    e = set_smem_once(topk_kernel<kMapPos>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                      (int)kTopkSmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(topk_kernel<kMapPos>, dim3(nq), dim3(kTopkThreads), kTopkSmem, st,
                   pos_vals, pos_stride, n_elems, map, map_stride, unit, q_vis, topk, out);
  } else {
    e = set_smem_once(topk_kernel<kMapSlot>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                      (int)kTopkSmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(topk_kernel<kMapSlot>, dim3(nq), dim3(kTopkThreads), kTopkSmem, st, vals,
                   stride, n_elems, map, map_stride, unit, q_vis, topk, out);
  }
  note_launches(1);
  return e;
}

}  // namespace csa2

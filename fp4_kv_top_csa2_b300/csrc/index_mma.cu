// index_mma.cu -- indexer scores on the 5th-generation tensor cores (tcgen05), TMA-fed.
//
// score(t) = sum_h w_h * max(0, kscale_t * <q_h, k_t>)  ("DeepSeek V4.1-Flash", aiwiki.ai, section
// "Compressed Sparse Attention 2": Full layers score every causally visible position with index
// keys and queries; Reindex layers rescore the candidate pool with their own query; the
// formula is this library's definition).
//
// One MMA per 128 keys x 16 query rows x 32 bytes of K (swap-AB: the keys are the M=128 side so
// a single query's 8 heads fill N=16 with padding), four K-steps per 128-byte key row:
//   E4M3 keys, Di=128: kind::f8f6f4, K=32 per MMA;   bf16 keys, Di=64: kind::f16, K=16 per MMA.
// Accumulators live in TMEM (4 buffers x 16 columns); the epilogue applies ReLU, the head
// weights and the head sum in fp32, then either
//   SCAN: per-position scores (optional) and block maxima over 8 positions, or
//   CAND: scores of the positions of listed blocks (each 8-row block one TMA box).
// Both modes run the same MMA sequence and epilogue, so a position gets the same fp32 score.
//
// Warp roles (320 threads): warp 0 = TMA producer, warp 1 = TMEM allocator + MMA issuer,
// warps 2..9 = two epilogue groups of four (warp w reads TMEM lanes 32*(w%4)..+31); group g
// drains the accumulators of the tiles with an even (g = 0) or odd (g = 1) running index, so
// two tiles' epilogues are in flight at once.  Work = chunks of up to CT
// consecutive 128-key tiles of one query, dealt round-robin to a persistent grid.
#include "sm100.cuh"

namespace csa2 {

constexpr int kTileKeys = 128;
constexpr int kKeyRowBytes = 128;
constexpr int kTileBytes = kTileKeys * kKeyRowBytes;  // 16 KB
constexpr int kStages = 6;
constexpr int kAccBufs = 4;
constexpr int kAccCols = 16;                          // N
constexpr int kTmemCols = kAccBufs * kAccCols;        // 64
constexpr int kQRows = 16;
constexpr int kQBytes = kQRows * kKeyRowBytes;        // 2 KB
constexpr int kIdxEpiGroups = 2;                   // epilogue groups, alternate accumulators
constexpr int kIdxThreads = 64 + kIdxEpiGroups * 128;
constexpr int kMaxScanQueries = 1024;

struct IdxSmem {
  uint8_t keys[kStages][kTileBytes];  // 1024-byte aligned (base is aligned by the kernel)
  uint8_t q[2][kQBytes];
  uint64_t full[kStages], empty[kStages];
  uint64_t qfull[2], qempty[2];
  uint64_t tfull[kAccBufs], tempty[kAccBufs];
  uint32_t tmem_base;
  volatile int abort;
  int prefix[kMaxScanQueries + 1];  // SCAN: chunk prefix sums over queries
};

enum IdxMode { kScan = 0, kCand = 1 };

struct IdxParams {
  const float *w;
  const float *k_scale;
  const int64_t *cu_ctx;
  const int32_t *q_seq;
  const int32_t *q_vis;
  const int32_t *cand;  // CAND: [nq, n_cand]
  float *bm;            // SCAN: [nq, bm_stride]
  float *scores;        // SCAN: [nq, sc_stride] per position (optional); CAND: [nq, n_cand*8]
  int64_t bm_stride, sc_stride;
  int nq, Hi, n_cand, ct;  // ct = tiles per chunk
};

struct Chunk {
  int n, t0, t1;  // query, tile range [t0, t1)
};

__device__ __forceinline__ int scan_total(const IdxSmem &sm, int nq) { return sm.prefix[nq]; }

__device__ __forceinline__ Chunk chunk_of(const IdxSmem &sm, const IdxParams &p, int mode, int j) {
  Chunk c;
  if (mode == kCand) {
    const int tiles = (p.n_cand * kBlock + kTileKeys - 1) / kTileKeys;
    const int per_q = (tiles + p.ct - 1) / p.ct;
    c.n = j / per_q;
    const int k = j - c.n * per_q;
    c.t0 = k * p.ct;
    c.t1 = min(tiles, c.t0 + p.ct);
  } else {
    int lo = 0, hi = p.nq;  // first n with prefix[n+1] > j
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (sm.prefix[mid + 1] > j) hi = mid; else lo = mid + 1;
    }
    c.n = lo;
    const int k = j - sm.prefix[lo];
    const int tiles = (p.q_vis[lo] + kTileKeys - 1) / kTileKeys;
    c.t0 = k * p.ct;
    c.t1 = min(tiles, c.t0 + p.ct);
  }
  return c;
}

template <int DT, int MODE>
__global__ void __launch_bounds__(kIdxThreads, 1) index_mma_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
    const IdxParams p) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_u32 = smem_u32(smem_raw);
  IdxSmem &sm = *reinterpret_cast<IdxSmem *>(smem_raw + ((1024 - (base_u32 & 1023)) & 1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- set-up: barriers, TMEM, work table
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(&sm.full[s], 1); mbar_init(&sm.empty[s], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&sm.qfull[s], 1); mbar_init(&sm.qempty[s], 1); }
    for (int a = 0; a < kAccBufs; ++a) {
      mbar_init(&sm.tfull[a], 1);
      mbar_init(&sm.tempty[a], 128);
    }
    sm.abort = 0;
    fence_barrier_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&qmap);
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  pdl_wait();
  int total;
  if (MODE == kScan) {
    if (warp == 0) {  // chunk prefix sums over queries, 32 at a time
      int run = 0;
      if (lane == 0) sm.prefix[0] = 0;
      for (int b = 0; b < p.nq; b += 32) {
        const int n = b + lane;
        int c = 0;
        if (n < p.nq) {
          const int tiles = (p.q_vis[n] + kTileKeys - 1) / kTileKeys;
          c = (tiles + p.ct - 1) / p.ct;
        }
        int inc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += y;
        }
        if (n < p.nq) sm.prefix[n + 1] = run + inc;
        run += __shfl_sync(0xffffffffu, inc, 31);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();
  if (MODE == kScan) {
    total = scan_total(sm, p.nq);
  } else {
    const int tiles = (p.n_cand * kBlock + kTileKeys - 1) / kTileKeys;
    total = p.nq * ((tiles + p.ct - 1) / p.ct);
  }
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0, qi = 0;
      for (int j = blockIdx.x; j < total && !sm.abort; j += gridDim.x) {
        const Chunk c = chunk_of(sm, p, MODE, j);
        const int64_t base = p.cu_ctx[p.q_seq[c.n]];
        const uint32_t qs = qi & 1;
        if (!mbar_wait(&sm.qempty[qs], ((qi >> 1) & 1) ^ 1)) { sm.abort = 1; break; }
        mbar_arrive_expect_tx(&sm.qfull[qs], kQBytes);
        tma_load_2d(sm.q[qs], &qmap, &sm.qfull[qs], 0, c.n * p.Hi);
        ++qi;
        for (int t = c.t0; t < c.t1; ++t, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1;
          if (!mbar_wait(&sm.empty[s], ph ^ 1)) { sm.abort = 1; break; }
          mbar_arrive_expect_tx(&sm.full[s], kTileBytes);
          if (MODE == kScan) {
            tma_load_2d(sm.keys[s], &kmap, &sm.full[s], 0, (int32_t)(base + (int64_t)t * kTileKeys));
          } else {
            // the tile's block ids first (independent loads, one latency), then its boxes
            const int32_t *cand = p.cand + (int64_t)c.n * p.n_cand;
            int blk[kTileKeys / kBlock];
#pragma unroll
            for (int b = 0; b < kTileKeys / kBlock; ++b) {
              const int cb = t * (kTileKeys / kBlock) + b;
              blk[b] = cb < p.n_cand ? __ldg(cand + cb) : -1;
            }
#pragma unroll
            for (int b = 0; b < kTileKeys / kBlock; ++b) {
              const int32_t row =
                  blk[b] >= 0 ? (int32_t)(base + (int64_t)blk[b] * kBlock) : -kBlock;
              tma_load_2d(sm.keys[s] + b * kBlock * kKeyRowBytes, &kmap, &sm.full[s], 0, row);
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = DT == CSA2_E4M3 ? idesc_f32acc(0, 0, 128, kAccCols)
                                                 : idesc_f32acc(1, 1, 128, kAccCols);
      uint32_t it = 0, qi = 0, acc = 0;
      for (int j = blockIdx.x; j < total && !sm.abort; j += gridDim.x) {
        const Chunk c = chunk_of(sm, p, MODE, j);
        const uint32_t qs = qi & 1;
        if (!mbar_wait(&sm.qfull[qs], (qi >> 1) & 1)) { sm.abort = 1; break; }
        ++qi;
        const uint32_t qaddr = smem_u32(sm.q[qs]);
        for (int t = c.t0; t < c.t1; ++t, ++it, ++acc) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1;
          const uint32_t a = acc % kAccBufs, aph = (acc / kAccBufs) & 1;
          if (!mbar_wait(&sm.full[s], ph)) { sm.abort = 1; break; }
          if (!mbar_wait(&sm.tempty[a], aph ^ 1)) { sm.abort = 1; break; }
          tc_fence_after();
          const uint32_t kaddr = smem_u32(sm.keys[s]);
          const uint32_t d = tmem + a * kAccCols;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = desc_k128_sw128(kaddr + 32 * k);
            const uint64_t bd = desc_k128_sw128(qaddr + 32 * k);
            if (DT == CSA2_E4M3) mma_f8f6f4(d, ad, bd, idesc, k > 0);
            else mma_f16(d, ad, bd, idesc, k > 0);
          }
          mma_commit(&sm.empty[s]);
          mma_commit(&sm.tfull[a]);
        }
        mma_commit(&sm.qempty[qs]);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int quarter = warp & 3, group = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    uint32_t acc = 0;
    for (int j = blockIdx.x; j < total; j += gridDim.x) {
      const Chunk c = chunk_of(sm, p, MODE, j);
      const int64_t base = p.cu_ctx[p.q_seq[c.n]];
      const int64_t V = p.q_vis[c.n];
      float wv[kAccCols];
#pragma unroll
      for (int h = 0; h < kAccCols; ++h) wv[h] = h < p.Hi ? p.w[(int64_t)c.n * p.Hi + h] : 0.0f;
      bool ok = true;
      // CAND: this row's block id for every tile of the chunk, loaded up front (ct <= 16)
      int blks[16];
      if (MODE == kCand) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int cb = (int)((((int64_t)(c.t0 + i)) * kTileKeys + row) >> 3);
          blks[i] = (c.t0 + i < c.t1 && cb < p.n_cand) ? p.cand[(int64_t)c.n * p.n_cand + cb] : -1;
        }
      }
      for (int t = c.t0; t < c.t1; ++t, ++acc) {
        if ((int)(acc % kIdxEpiGroups) != group) continue;  // the other group's tile
        const uint32_t a = acc % kAccBufs, aph = (acc / kAccBufs) & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.tfull[a], aph));
        if (!ok) break;
        tc_fence_after();
        uint32_t r[16];
        tmem_ld16(lane_addr + a * kAccCols, r);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&sm.tempty[a]);
        // position of this row
        int64_t pos;
        bool valid;
        int64_t slot = 0;
        if (MODE == kScan) {
          pos = (int64_t)t * kTileKeys + row;
          valid = pos < V;
        } else {
          slot = (int64_t)t * kTileKeys + row;
          int blk = -1;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (t - c.t0 == i) blk = blks[i];
          pos = (int64_t)blk * kBlock + (slot & 7);
          valid = blk >= 0 && pos < V;
        }
        const float ks = (valid && p.k_scale) ? p.k_scale[base + pos] : 1.0f;
        float sc = 0.0f;
#pragma unroll
        for (int h = 0; h < kAccCols; ++h)
          if (h < p.Hi) sc = fmaf(wv[h], fmaxf(__uint_as_float(r[h]) * ks, 0.0f), sc);
        if (MODE == kScan) {
          if (valid && p.scores) p.scores[(int64_t)c.n * p.sc_stride + pos] = sc;
          float m = valid ? sc : -INFINITY;
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
          if ((lane & 7) == 0 && valid) p.bm[(int64_t)c.n * p.bm_stride + (pos >> 3)] = m;
        } else {
          if (slot < (int64_t)p.n_cand * kBlock)
            p.scores[(int64_t)c.n * p.n_cand * kBlock + slot] = valid ? sc : 0.0f;
        }
      }
      if (!ok) { sm.abort = 1; break; }
    }
  }
  // ---- tear-down
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// Tensor map of `rows` rows of 128 bytes, box = box_rows x 128 bytes, 128-byte swizzle.
static bool make_rows128_map(CUtensorMap *m, const void *base, int64_t rows, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rows <= 0) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

static int sm_count() {
  static int n = [] {
    int dev = 0, v = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    return v;
  }();
  return n;
}

template <int DT, int MODE>
static cudaError_t launch_index_mma_t(const CUtensorMap &km, const CUtensorMap &qm,
                                      const IdxParams &p, int grid, cudaStream_t st) {
  const size_t smem = sizeof(IdxSmem) + 1024;
  cudaError_t e = set_smem_once(index_mma_kernel<DT, MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(index_mma_kernel<DT, MODE>, dim3(grid), dim3(kIdxThreads), smem, st, km, qm, p);
  note_launches(1);
  return e;
}

bool index_mma_supported(int nq) { return nq <= kMaxScanQueries && encode_fn() != nullptr; }
bool cand_mma_supported() { return encode_fn() != nullptr; }

// Full-mode scan on tensor cores.  scores may be null (block maxima only).
cudaError_t launch_score_scan_mma(const void *q_idx, int dtype, const float *w, int nq, int Hi,
                                  const void *k_idx, int64_t k_rows, const float *k_scale,
                                  const int64_t *cu_ctx, const int32_t *q_seq,
                                  const int32_t *q_vis, int64_t max_vis, float *bm,
                                  int64_t bm_stride, float *scores, int64_t sc_stride,
                                  cudaStream_t st) {
  if (nq == 0 || max_vis == 0) return cudaSuccess;
  CUtensorMap km, qm;
  if (!make_rows128_map(&km, k_idx, k_rows, kTileKeys) ||
      !make_rows128_map(&qm, q_idx, (int64_t)nq * Hi, kQRows))
    return cudaErrorInvalidValue;
  IdxParams p{};
  p.w = w; p.k_scale = k_scale; p.cu_ctx = cu_ctx; p.q_seq = q_seq; p.q_vis = q_vis;
  p.bm = bm; p.bm_stride = bm_stride; p.scores = scores; p.sc_stride = sc_stride;
  p.nq = nq; p.Hi = Hi;
  const int grid = 2 * sm_count();
  const int64_t max_tiles = (max_vis + kTileKeys - 1) / kTileKeys;
  p.ct = (int)std::max<int64_t>(1, std::min<int64_t>(16, (nq * max_tiles + 4 * grid - 1) / (4 * grid)));
  return dtype == CSA2_E4M3 ? launch_index_mma_t<CSA2_E4M3, kScan>(km, qm, p, grid, st)
                            : launch_index_mma_t<CSA2_BF16, kScan>(km, qm, p, grid, st);
}

// Candidate scoring on tensor cores: scores[n, i] for the 8*n_cand slots of each query.
cudaError_t launch_score_cand_mma(const void *q_idx, int dtype, const float *w, int nq, int Hi,
                                  const void *k_idx, int64_t k_rows, const float *k_scale,
                                  const int64_t *cu_ctx, const int32_t *q_seq,
                                  const int32_t *q_vis, const int32_t *cand, int n_cand,
                                  float *scores, cudaStream_t st) {
  if (nq == 0 || n_cand == 0) return cudaSuccess;
  CUtensorMap km, qm;
  if (!make_rows128_map(&km, k_idx, k_rows, kBlock) ||
      !make_rows128_map(&qm, q_idx, (int64_t)nq * Hi, kQRows))
    return cudaErrorInvalidValue;
  IdxParams p{};
  p.w = w; p.k_scale = k_scale; p.cu_ctx = cu_ctx; p.q_seq = q_seq; p.q_vis = q_vis;
  p.cand = cand; p.n_cand = n_cand; p.scores = scores;
  p.nq = nq; p.Hi = Hi;
  const int sms = 2 * sm_count();
  const int tiles = (n_cand * kBlock + kTileKeys - 1) / kTileKeys;
  const int64_t total_tiles = (int64_t)nq * tiles;
  p.ct = (int)std::max<int64_t>(1, std::min<int64_t>(16, (total_tiles + 2 * sms - 1) / (2 * sms)));
  const int64_t chunks = (int64_t)nq * ((tiles + p.ct - 1) / p.ct);
  const int grid = (int)std::min<int64_t>(chunks, sms);
  return dtype == CSA2_E4M3 ? launch_index_mma_t<CSA2_E4M3, kCand>(km, qm, p, grid, st)
                            : launch_index_mma_t<CSA2_BF16, kCand>(km, qm, p, grid, st);
}

}  // namespace csa2

// index_keys.cu -- index keys derived from main-KV rows ("DeepSeek V4.1-Flash", aiwiki.ai,
// section "Compressed Sparse Attention 2": CSA2 derives index keys from main KV entries rather
// than through a separate hidden-state compression path).
//
// For each cached row t: x = the dequantised FP4 row (512 channels, exact in bf16), W the layer's
// index-key projection [128, 512] bf16:
//   y_i = sum_c W[i,c] x[c]    (tcgen05 kind::f16, bf16 x bf16, fp32 accumulation in TMEM)
//   s   = max_i |y_i| / 448     (fp32 division; 1 if every y_i is 0)
//   key_i = E4M3(y_i / s)       (y_i times the fp32 reciprocal of s, round to nearest even,
//                                saturating)
// keys [rows, 128] and k_scale [rows] = s are the indexer's k_idx and k_scale.
//
// Persistent CTAs (one per SM): W stays in shared memory (eight 128B-swizzled chunks of 64
// channels, loaded once by TMA) as the K-major B operand, N = 128 key dimensions.  Per tile of
// 128 rows, warps 0..7 gather the FP4 rows (16-byte loads, the next tile's in flight) and dequantise
// them chunk by chunk into a 4-stage ring (the K-major A operand, M = 128 rows); warp 8 issues
// four M=128 x N=128 x K=16 MMAs per chunk into one of two TMEM accumulators; warps 9..16 drain
// the accumulator, two per lane quarter with 64 columns each (the row maximum is combined
// through shared memory, then the keys).
#include "sm100.cuh"

namespace csa2 {

constexpr int kIkRows = 128;                  // rows per tile (MMA M)
constexpr int kIkDi = 128;                    // key dimensions (MMA N)
constexpr int kIkStages = 4;                  // A-chunk ring
constexpr int kIkChunk = kIkRows * 128;       // one 64-channel chunk of rows or of W: 16 KB
constexpr int kIkWorkers = 256;               // warps 0..7
constexpr int kIkMmaWarp = 8;
constexpr int kIkEpiWarp0 = 9;                // warps 9..16: two per TMEM lane quarter
constexpr int kIkThreads = (kIkEpiWarp0 + 8) * 32;
constexpr int kIkOffW = 0;                                    // 8 x 16 KB
constexpr int kIkOffA = 8 * kIkChunk;                         // 4 x 16 KB
constexpr int kIkOffLut = kIkOffA + kIkStages * kIkChunk;     // 256 x u32
constexpr int kIkOffMisc = kIkOffLut + 1024;
constexpr int kIkSmem = kIkOffMisc + 128 + 1024 + 1024;  // misc, row maxima, alignment
static_assert(kIkSmem <= 232448, "shared memory per CTA");

struct IkMisc {
  uint64_t bar_w, full[kIkStages], empty[kIkStages], tfull[2], tempty[2];
  uint32_t tmem_base;
};
static_assert(sizeof(IkMisc) <= 128, "misc block");

__global__ void __launch_bounds__(kIkThreads, 1) index_keys_kernel(
    const __grid_constant__ CUtensorMap wmap, const uint8_t *__restrict__ codes,
    const uint8_t *__restrict__ sf, int64_t n_rows, const int64_t *__restrict__ rows,
    uint8_t *__restrict__ keys, float *__restrict__ k_scale) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  IkMisc &ms = *reinterpret_cast<IkMisc *>(sm + kIkOffMisc);
  uint32_t *lut = reinterpret_cast<uint32_t *>(sm + kIkOffLut);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t n_tiles = (n_rows + kIkRows - 1) / kIkRows;

  if (tid == 0) {
    mbar_init(&ms.bar_w, 1);
    for (int s = 0; s < kIkStages; ++s) {
      mbar_init(&ms.full[s], kIkWorkers);
      mbar_init(&ms.empty[s], 1);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(&ms.tfull[d], 1);
      mbar_init(&ms.tempty[d], 256);
    }
    fence_barrier_init();
    prefetch_tensormap(&wmap);
  }
  if (warp == kIkMmaWarp) {
    tmem_alloc(&ms.tmem_base, 256);
    tmem_relinquish();
  }
  if (tid < 256) lut[tid] = pack_bf16x2(e2m1_to_float(tid & 15), e2m1_to_float(tid >> 4));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;
  pdl_wait();
  pdl_trigger();
  bool ok = true;

  if (warp < 8) {
    // ------------------------------------------------------------------ producers (warps 0..7)
    // thread: row r = tid / 2 of the tile, channels 32*half .. +31 of every 64-channel chunk.
    // A tile's eight chunks (eight 16-byte code loads and eight scale pairs) are loaded one tile
    // ahead, so the HBM latency overlaps the previous tile's work.
    const int r = tid >> 1, half = tid & 1;
    uint4 cur[8], nxt[8];
    uint32_t scur[8], snxt[8];
    auto load_tile = [&](int64_t tile, uint4 (&c)[8], uint32_t (&sc)[8]) {
      const int64_t slot = tile * kIkRows + r;
      const int64_t row = (tile < n_tiles && slot < n_rows) ? (rows ? rows[slot] : slot) : -1;
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) {
        c[kc] = row >= 0 ? __ldg(reinterpret_cast<const uint4 *>(codes + row * kCodeBytes +
                                                                 32 * kc + 16 * half))
                         : make_uint4(0, 0, 0, 0);
        sc[kc] = row >= 0 ? (uint32_t)__ldg(reinterpret_cast<const uint16_t *>(
                                sf + row * kSfBytes + 4 * kc + 2 * half))
                          : 0u;
      }
    };
    uint32_t it = 0;
    load_tile(blockIdx.x, cur, scur);
    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
      load_tile(tile + gridDim.x, nxt, snxt);  // in flight while this tile is dequantised
#pragma unroll
      for (int kc = 0; kc < 8; ++kc, ++it) {
        const uint32_t st = it % kIkStages, ph = (it / kIkStages) & 1;
        ok = mbar_wait(&ms.empty[st], ph ^ 1) && ok;
        const float fa = e4m3_to_float(scur[kc] & 0xFF), fb = e4m3_to_float(scur[kc] >> 8);
        const uint32_t sa = pack_bf16x2(fa, fa), sb = pack_bf16x2(fb, fb);
        const uint32_t w[4] = {cur[kc].x, cur[kc].y, cur[kc].z, cur[kc].w};
        uint8_t *dst = sm + kIkOffA + st * kIkChunk + r * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {  // 8 channels per 16-byte unit; units 4*half .. +3
          const uint32_t scl = u < 2 ? sa : sb;
          uint4 v;
          v.x = bf16x2_mul(lut[w[u] & 0xFF], scl);
          v.y = bf16x2_mul(lut[(w[u] >> 8) & 0xFF], scl);
          v.z = bf16x2_mul(lut[(w[u] >> 16) & 0xFF], scl);
          v.w = bf16x2_mul(lut[w[u] >> 24], scl);
          *reinterpret_cast<uint4 *>(dst + (((4 * half + u) ^ (r & 7)) << 4)) = v;
        }
        fence_async_smem();
        mbar_arrive(&ms.full[st]);
      }
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) cur[kc] = nxt[kc], scur[kc] = snxt[kc];
    }
  } else if (warp == kIkMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      mbar_arrive_expect_tx(&ms.bar_w, 8 * kIkChunk);
      for (int kc = 0; kc < 8; ++kc)
        tma_load_2d(sm + kIkOffW + kc * kIkChunk, &wmap, &ms.bar_w, kc * 64, 0);
      ok = mbar_wait(&ms.bar_w, 0) && ok;
      constexpr uint32_t idesc = idesc_f32acc(1, 1, kIkRows, kIkDi);  // bf16 x bf16
      const uint32_t wa = smem_u32(sm + kIkOffW), aa = smem_u32(sm + kIkOffA);
      uint32_t it = 0, nt = 0;
      for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++nt) {
        const uint32_t d = nt & 1, dph = (nt >> 1) & 1;
        ok = mbar_wait(&ms.tempty[d], dph ^ 1) && ok;
        tc_fence_after();
        for (int kc = 0; kc < 8; ++kc, ++it) {
          const uint32_t st = it % kIkStages, ph = (it / kIkStages) & 1;
          ok = mbar_wait(&ms.full[st], ph) && ok;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_f16(tmem + d * kIkDi, desc_k128_sw128(aa + st * kIkChunk + 32 * ks),
                    desc_k128_sw128(wa + kc * kIkChunk + 32 * ks), idesc, (kc | ks) != 0);
          mma_commit(&ms.empty[st]);
        }
        mma_commit(&ms.tfull[d]);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue (warps 9..16)
    const int quarter = warp & 3, half = (warp - kIkEpiWarp0) >> 2, r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    float *pmax = reinterpret_cast<float *>(sm + kIkOffMisc + 128);  // [2][128] row maxima
    uint32_t nt = 0;
    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++nt) {
      const uint32_t d = nt & 1, dph = (nt >> 1) & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&ms.tfull[d], dph)) && ok;
      tc_fence_after();
      const uint32_t ta = tmem + d * kIkDi + 64 * half + lane_off;
      uint32_t v[64];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_ld16(ta + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&v[16 * c]));
      tmem_ld_wait();
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fabsf(__uint_as_float(v[i])));
      pmax[half * 128 + r] = amax;
      asm volatile("bar.sync 1, 256;" ::: "memory");  // the two halves' maxima
      amax = fmaxf(pmax[r], pmax[128 + r]);
      asm volatile("bar.sync 1, 256;" ::: "memory");  // read before the next tile writes
      const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
      const float inv = __frcp_rn(s);
      const int64_t slot = tile * kIkRows + r;
      const int64_t row = slot < n_rows ? (rows ? rows[slot] : slot) : -1;
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        uint16_t lo, hi;
        const float q0 = __uint_as_float(v[4 * k]) * inv, q1 = __uint_as_float(v[4 * k + 1]) * inv;
        const float q2 = __uint_as_float(v[4 * k + 2]) * inv, q3 = __uint_as_float(v[4 * k + 3]) * inv;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(q1), "f"(q0));
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(q3), "f"(q2));
        pk[k] = (uint32_t)lo | ((uint32_t)hi << 16);
      }
      if (row >= 0) {
        uint4 *dst = reinterpret_cast<uint4 *>(keys + row * kIkDi + 64 * half);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        if (half == 0) k_scale[row] = ok ? s : 0.0f;
      }
      tc_fence_before();
      mbar_arrive(&ms.tempty[d]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kIkMmaWarp) tmem_dealloc(tmem, 256);
}

bool index_keys_supported() { return encode_fn() != nullptr; }

cudaError_t launch_index_keys(const uint8_t *codes, const uint8_t *sf, int64_t n_rows,
                              const int64_t *rows, const void *w_bf16, uint8_t *keys,
                              float *k_scale, cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap wm;
  memset(&wm, 0, sizeof(wm));
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)kIkDi};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, kIkDi};
  cuuint32_t estr[2] = {1, 1};
  if (enc(&wm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(w_bf16), dims, strides,
          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_once(index_keys_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kIkSmem);
  if (e != cudaSuccess) return e;
  const int64_t n_tiles = (n_rows + kIkRows - 1) / kIkRows;
  const int grid = (int)std::min<int64_t>(n_tiles, sm_count());
  e = launch_pdl(index_keys_kernel, dim3(grid), dim3(kIkThreads), kIkSmem, st, wm, codes, sf,
                 n_rows, rows, keys, k_scale);
  note_launches(1);
  return e;
}

}  // namespace csa2

// index_multi.cu -- Full-mode indexer scan for many queries over one sequence (chunked prefill).
//
// Same score as index_mma.cu (score(t) = sum_h w_h * max(0, kscale_t * <q_h, k_t>)), but 32
// query tokens share every 128-key tile: one MMA is M=128 keys x N=256 (32 queries x 8 heads)
// x K=32 bytes, four K-steps per 128-byte key row, so the keys are read once per 32 queries and
// the tensor pipe does real work.  Causal visibility per query (query i sees positions
// t < q_vis[i], "DeepSeek V4.1-Flash", aiwiki.ai, section "Compressed Sparse Attention 2":
// the indexer scores the causally visible positions) is applied in the epilogue, which writes
// the block maxima over 8 positions for every query.
//
// Warp roles (576 threads): warp 0 = TMA producer, warp 1 = TMEM allocator + MMA issuer,
// warps 2..17 = epilogue; warp w reads TMEM lanes 32*(w%4)..+31 and the 64 accumulator columns
// of queries 8*((w-2)/4) .. +7.  TMEM: two 256-column accumulators.  Work = chunks of up to
// CT key tiles of one 32-query group, dealt round-robin to a persistent grid (one CTA per SM).
#include "sm100.cuh"

namespace csa2 {

constexpr int kMqQ = 32;                        // queries per group
constexpr int kMqN = 256;                       // MMA N = 32 queries x 8 heads
constexpr int kMqStages = 4;
constexpr int kMqEpiWarps = 16;                 // epilogue warps: 4 per TMEM lane quarter
constexpr int kMqQPW = kMqQ / (kMqEpiWarps / 4);  // queries per epilogue warp (8)
constexpr int kMqThreads = 64 + kMqEpiWarps * 32;
constexpr int kMqQBytes = kMqN * 128;           // 32 KB

struct MqSmem {
  uint8_t keys[kMqStages][128 * 128];           // 16 KB tiles, 1024-byte aligned
  uint8_t q[2][kMqQBytes];
  __align__(16) float wsm[kMqEpiWarps][kMqQPW * 8];  // per epilogue warp: its queries' head weights
  int vsm[kMqEpiWarps][kMqQPW];        // and their visible lengths
  uint64_t full[kMqStages], empty[kMqStages];
  uint64_t qfull[2], qempty[2];
  uint64_t tfull[2], tempty[2];
  uint32_t tmem_base;
  volatile int abort;
};

struct MqParams {
  const float *w;        // [nq, 8]
  const float *k_scale;  // [k_rows] or null
  const int32_t *q_vis;  // [nq]
  float *bm;             // [nq, bm_stride]
  int64_t bm_stride;
  float *scores;         // [nq, sc_stride] per position (optional)
  int64_t sc_stride;
  int64_t base;          // first key row of the (single) sequence
  int64_t max_vis;       // largest q_vis (positions beyond it are never read)
  int nq, n_tiles, ct;   // key tiles of 128, tiles per chunk
};

// KS: per-key scales present (without them the epilogue skips the multiply by 1).
template <int DT, bool KS>
__global__ void __launch_bounds__(kMqThreads, 1) index_multi_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
    const MqParams p) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  MqSmem &sm = *reinterpret_cast<MqSmem *>(smem_raw + ((1024 - (raw_u32 & 1023)) & 1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_groups = (p.nq + kMqQ - 1) / kMqQ;
  const int chunks_per_group = (p.n_tiles + p.ct - 1) / p.ct;
  const int total = n_groups * chunks_per_group;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMqStages; ++s) { mbar_init(&sm.full[s], 1); mbar_init(&sm.empty[s], 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.qfull[s], 1);
      mbar_init(&sm.qempty[s], 1);
      mbar_init(&sm.tfull[s], 1);
      mbar_init(&sm.tempty[s], kMqEpiWarps * 32);
    }
    sm.abort = 0;
    fence_barrier_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&qmap);
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------------------ TMA producer
      uint32_t it = 0, qi = 0;
      for (int j = blockIdx.x; j < total && !sm.abort; j += gridDim.x) {
        const int g = j / chunks_per_group, t0 = (j % chunks_per_group) * p.ct;
        const int t1 = min(p.n_tiles, t0 + p.ct);
        const uint32_t qs = qi & 1;
        if (!mbar_wait(&sm.qempty[qs], ((qi >> 1) & 1) ^ 1)) { sm.abort = 1; break; }
        mbar_arrive_expect_tx(&sm.qfull[qs], kMqQBytes);
        tma_load_2d(sm.q[qs], &qmap, &sm.qfull[qs], 0, g * kMqN);
        ++qi;
        for (int t = t0; t < t1; ++t, ++it) {
          const uint32_t s = it % kMqStages, ph = (it / kMqStages) & 1;
          if (!mbar_wait(&sm.empty[s], ph ^ 1)) { sm.abort = 1; break; }
          mbar_arrive_expect_tx(&sm.full[s], 128 * 128);
          tma_load_2d(sm.keys[s], &kmap, &sm.full[s], 0, (int32_t)(p.base + (int64_t)t * 128));
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = DT == CSA2_E4M3 ? idesc_f32acc(0, 0, 128, kMqN)
                                                 : idesc_f32acc(1, 1, 128, kMqN);
      uint32_t it = 0, qi = 0, acc = 0;
      for (int j = blockIdx.x; j < total && !sm.abort; j += gridDim.x) {
        const int t0 = (j % chunks_per_group) * p.ct;
        const int t1 = min(p.n_tiles, t0 + p.ct);
        const uint32_t qs = qi & 1;
        if (!mbar_wait(&sm.qfull[qs], (qi >> 1) & 1)) { sm.abort = 1; break; }
        ++qi;
        const uint32_t qaddr = smem_u32(sm.q[qs]);
        for (int t = t0; t < t1; ++t, ++it, ++acc) {
          const uint32_t s = it % kMqStages, ph = (it / kMqStages) & 1;
          const uint32_t a = acc & 1, aph = (acc >> 1) & 1;
          if (!mbar_wait(&sm.full[s], ph)) { sm.abort = 1; break; }
          if (!mbar_wait(&sm.tempty[a], aph ^ 1)) { sm.abort = 1; break; }
          tc_fence_after();
          const uint32_t kaddr = smem_u32(sm.keys[s]);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = desc_k128_sw128(kaddr + 32 * k);
            const uint64_t bd = desc_k128_sw128(qaddr + 32 * k);
            if (DT == CSA2_E4M3) mma_f8f6f4(tmem + a * kMqN, ad, bd, idesc, k > 0);
            else mma_f16(tmem + a * kMqN, ad, bd, idesc, k > 0);
          }
          mma_commit(&sm.empty[s]);
          mma_commit(&sm.tfull[a]);
        }
        mma_commit(&sm.qempty[qs]);
      }
    }
  } else {  // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;                 // 0 .. kMqEpiWarps-1
    const int quarter = warp & 3, qslot = ew >> 2;  // queries qslot*kMqQPW .. +kMqQPW-1
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    // After the transposed block-maximum reduction below, lane l holds the maximum of block
    // l/8 (of this warp's 32 rows) for query rq of the warp's eight.
    const int rq = ((lane & 1) << 2) | (lane & 2) | ((lane >> 2) & 1);
    uint32_t acc = 0;
    for (int j = blockIdx.x; j < total; j += gridDim.x) {
      const int g = j / chunks_per_group, t0 = (j % chunks_per_group) * p.ct;
      const int t1 = min(p.n_tiles, t0 + p.ct);
      const int q0 = g * kMqQ + qslot * kMqQPW;
      // this chunk's weights and visible lengths (this warp's queries; a query beyond nq sees
      // nothing, so every store below is masked by visibility alone)
      float *wq = sm.wsm[ew];
      int *vq = sm.vsm[ew];
      __syncwarp();
      for (int i = lane; i < kMqQPW * 8; i += 32) {
        const int q = q0 + i / 8;
        wq[i] = q < p.nq ? __ldg(p.w + (int64_t)q * 8 + (i & 7)) : 0.0f;
      }
      if (lane < kMqQPW) {
        const int q = q0 + lane;
        vq[lane] = q < p.nq ? p.q_vis[q] : 0;
      }
      __syncwarp();
      const int vmin = __reduce_min_sync(0xffffffffu, lane < kMqQPW ? vq[lane] : INT_MAX);
      const int my_vis = vq[rq];
      float *const bm_row = p.bm + (int64_t)(q0 + rq) * p.bm_stride;
      float *const sc_rows = p.scores ? p.scores + (int64_t)q0 * p.sc_stride : nullptr;
      bool ok = true;
      for (int t = t0; t < t1; ++t, ++acc) {
        const uint32_t a = acc & 1, aph = (acc >> 1) & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.tfull[a], aph));
        if (!ok) break;
        tc_fence_after();
        const int64_t pos = (int64_t)t * 128 + row;
        const float ks = (KS && pos < p.max_vis) ? p.k_scale[p.base + pos] : 1.0f;
        // every position of this tile is visible to all eight queries
        const bool all_vis = (int64_t)t * 128 + 128 <= vmin;
        float v[kMqQPW];
        {
          uint32_t r[4][16];
          const uint32_t col = lane_addr + a * kMqN + qslot * kMqQPW * 8;
#pragma unroll
          for (int l = 0; l < 4; ++l) tmem_ld16(col + 16 * l, r[l]);  // four loads, one wait
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&sm.tempty[a]);  // the accumulator is in registers: release it
          const float4 *w4 = reinterpret_cast<const float4 *>(wq);
#pragma unroll
          for (int qq = 0; qq < kMqQPW; ++qq) {
            const float4 wa = w4[2 * qq], wb = w4[2 * qq + 1];
            const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
            float sc = 0.0f;
#pragma unroll
            for (int h = 0; h < 8; ++h) {
              const float x = __uint_as_float(r[qq >> 1][8 * (qq & 1) + h]);
              sc = fmaf(wv[h], fmaxf(KS ? x * ks : x, 0.0f), sc);
            }
            v[qq] = sc;
          }
        }
        if (sc_rows) {
          float *sp = sc_rows + pos;
          if (all_vis) {
#pragma unroll
            for (int qq = 0; qq < kMqQPW; ++qq, sp += p.sc_stride) *sp = v[qq];
          } else {
#pragma unroll
            for (int qq = 0; qq < kMqQPW; ++qq, sp += p.sc_stride)
              if (pos < vq[qq]) *sp = v[qq];
          }
        }
        if (!all_vis) {
#pragma unroll
          for (int qq = 0; qq < kMqQPW; ++qq) v[qq] = pos < vq[qq] ? v[qq] : -INFINITY;
        }
        // Block maxima of eight queries over eight lanes in three exchange steps: at each
        // step a lane keeps half of its queries, sends the other half to its partner and takes
        // the maximum with what it receives.
        const bool b0 = lane & 1, b1 = lane & 2, b2 = lane & 4;
        float u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float keep = b0 ? v[i + 4] : v[i], send = b0 ? v[i] : v[i + 4];
          u[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 1));
        }
        float y[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float keep = b1 ? u[i + 2] : u[i], send = b1 ? u[i] : u[i + 2];
          y[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 2));
        }
        {
          const float keep = b2 ? y[1] : y[0], send = b2 ? y[0] : y[1];
          const float m = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 4));
          const int64_t first = (int64_t)t * 128 + quarter * 32 + (lane & ~7);
          if (first < my_vis) bm_row[first >> 3] = m;
        }
      }
      if (!ok) { sm.abort = 1; break; }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

bool index_multi_supported(int nq, int Hi, int B) {
  return B == 1 && Hi == 8 && nq > 1024 && encode_fn() != nullptr;
}

// Block maxima of every query over one sequence (all queries in sequence 0, rows from 0), and
// the score of every visible position when `scores` is not null.
cudaError_t launch_score_scan_multi(const void *q_idx, int dtype, const float *w, int nq,
                                    const void *k_idx, int64_t k_rows, const float *k_scale,
                                    const int32_t *q_vis, int64_t max_vis, float *bm,
                                    int64_t bm_stride, float *scores, int64_t sc_stride,
                                    cudaStream_t st) {
  if (nq == 0 || max_vis == 0) return cudaSuccess;
  CUtensorMap km, qm;
  if (!make_rows128_map(&km, k_idx, k_rows, 128) ||
      !make_rows128_map(&qm, q_idx, (int64_t)nq * 8, kMqN))
    return cudaErrorInvalidValue;
  MqParams p{};
  p.w = w; p.k_scale = k_scale; p.q_vis = q_vis; p.bm = bm; p.bm_stride = bm_stride;
  p.scores = scores; p.sc_stride = sc_stride;
  p.base = 0; p.max_vis = max_vis; p.nq = nq;
  p.n_tiles = (int)((max_vis + 127) / 128);
  const int grid = sm_count();
  const int64_t groups = (nq + kMqQ - 1) / kMqQ;
  p.ct = (int)std::max<int64_t>(1, std::min<int64_t>(16, groups * p.n_tiles / (grid * 8)));
  const size_t smem = sizeof(MqSmem) + 1024;
  auto go = [&](auto kern) {
    cudaError_t err = set_smem_once(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(grid), dim3(kMqThreads), smem, st, km, qm, p);
  };
  cudaError_t e;
  if (dtype == CSA2_E4M3)
    e = k_scale ? go(index_multi_kernel<CSA2_E4M3, true>) : go(index_multi_kernel<CSA2_E4M3, false>);
  else
    e = k_scale ? go(index_multi_kernel<CSA2_BF16, true>) : go(index_multi_kernel<CSA2_BF16, false>);
  note_launches(1);
  return e;
}

}  // namespace csa2

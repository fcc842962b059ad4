// attn_mma.cu -- sparse decode attention over gathered FP4 rows on the tensor cores (tcgen05).
//
// For sequence n, head h: softmax_j(scale * q_h . khat_j) over the selected rows j, applied to
// the same rows (K = V = the dequantised latent row; the model card's Introduction, CSA2
// paragraph: attention reuses "Top-K sparse-attention indices" into the FP4 main KV).
//
// One CTA = one query (sequence) x one tile of 64 selected rows, all heads (H <= 64, padded to
// the M=128 MMA shape).  Steps:
//   1. Q [H x 512] bf16 arrives by TMA as eight 128B-swizzled K-chunks of 64 channels; each
//      selected row arrives as two bulk copies (256 B of codes, 32 B of scales).
//   2. Every row is dequantised exactly (E2M1 x E4M3 has <= 6 significant bits) to bf16 and
//      stored once, as eight 128B-swizzled chunks [64 rows x 64 channels].
//   3. S = Q Khat^T: kind::f16, M=128 (heads) x N=64 (rows) x K=512, fp32 in TMEM.
//   4. Softmax rows (exp2 domain; four warps, two per 32-column half of S), P split into bf16
//      hi + lo parts (P ~ hi + lo to 2^-17).
//   5. O^T = Vhat^T (P_hi + P_lo)^T: kind::f16, the same dequantised chunks read as the
//      MN-major A operand (channels contiguous, M=128 channels = two chunks), P as the K-major
//      B operand (N=64 heads), fp32 in TMEM columns 0..255 (S lives in 256..319).
//   6. Channels on TMEM lanes make the epilogue coalesced: a warp stores 32 consecutive channels
//      of one head per instruction.  The unnormalised O rows and the per-head (max, sum) go to
//      workspace; a combine kernel merges the tiles of each query.
#include <cstring>

#include "sm100.cuh"

namespace csa2 {

constexpr int kAttTS = 64;          // selected rows per CTA
constexpr int kAttThreads = 256;
constexpr int kAttTmemCols = 512;
constexpr int kColS = 256;          // S [heads x rows]; O^T takes columns 0..255

// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;                         // 8 chunks x (64 rows x 128 B) = 64 KB
constexpr int kOffK = 64 * 1024;                 // 8 chunks x (64 rows x 128 B) = 64 KB
constexpr int kOffPhi = 128 * 1024;              // 64 rows x 128 B
constexpr int kOffPlo = 136 * 1024;              // 64 rows x 128 B
constexpr int kOffRawC = 144 * 1024;             // 64 rows x 256 B codes
constexpr int kOffRawS = kOffRawC + kAttTS * 256;  // 64 rows x 32 B scales
constexpr int kOffLut = kOffRawS + kAttTS * 32;    // 256 x u32
constexpr int kOffMisc = kOffLut + 1024;
constexpr int kAttSmem = kOffMisc + 1024 + 1024;  // + alignment slack
// The M=128 operand read of Q chunk 7 runs 8 KB past its 64 real rows, into K-chunk 0:
// readable, and it only feeds unused accumulator lanes.

struct AttMisc {
  uint64_t bar_q, bar_g, bar_s, bar_o;
  uint32_t tmem_base;
  int slot_ok[kAttTS];
  float m2[64];
  float mh[2][64], lh[2][64];  // per-half row max / sum of the softmax
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162 *>(&a);
  __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162 *>(&b);
  __nv_bfloat162 z = __hmul2(x, y);
  return *reinterpret_cast<uint32_t *>(&z);
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(sm100::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(sm100::smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <bool kQfp4>
__global__ void __launch_bounds__(kAttThreads, 1) attn_mma_kernel(
    const __grid_constant__ CUtensorMap qmap, const uint8_t *__restrict__ q_codes,
    const uint8_t *__restrict__ q_sf, int H, const int32_t *__restrict__ q_seq,
    const uint8_t *__restrict__ codes, const uint8_t *__restrict__ sf,
    const int64_t *__restrict__ cu_ctx, const int32_t *__restrict__ idx, int topk,
    float scale_log2e, int n_tiles, float *__restrict__ o_part, float *__restrict__ m_part,
    float *__restrict__ l_part) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t *sm = smem_raw + ((1024 - (raw_u32 & 1023)) & 1023);
  AttMisc &ms = *reinterpret_cast<AttMisc *>(sm + kOffMisc);
  uint32_t *lut = reinterpret_cast<uint32_t *>(sm + kOffLut);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, n = blockIdx.y;

  if (tid == 0) {
    mbar_init(&ms.bar_q, 1);
    mbar_init(&ms.bar_g, kAttTS);
    mbar_init(&ms.bar_s, 1);
    mbar_init(&ms.bar_o, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&ms.tmem_base, kAttTmemCols);
    tmem_relinquish();
  }
  // byte of two E2M1 codes -> bf16x2 of their values (exact)
  lut[tid] = pack_bf16x2(e2m1_to_float(tid & 15), e2m1_to_float(tid >> 4));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;
  pdl_wait();
  pdl_trigger();
  const int64_t base = cu_ctx[q_seq ? q_seq[n] : n];

  // ---- 1. loads
  if (!kQfp4 && tid == 0) {
    mbar_arrive_expect_tx(&ms.bar_q, 8 * 64 * 128);
    for (int kc = 0; kc < 8; ++kc) tma_load_2d(sm + kOffQ + kc * 8192, &qmap, &ms.bar_q, kc * 64, n * H);
  }
  if (tid < kAttTS) {
    const int slot = tile * kAttTS + tid;
    const int r = slot < topk ? idx[(int64_t)n * topk + slot] : -1;
    ms.slot_ok[tid] = r >= 0;
    if (r >= 0) {
      const int64_t row = base + r;
      mbar_arrive_expect_tx(&ms.bar_g, 288);
      bulk_g2s(sm + kOffRawC + tid * 256, codes + row * kCodeBytes, 256, &ms.bar_g);
      bulk_g2s(sm + kOffRawS + tid * 32, sf + row * kSfBytes, 32, &ms.bar_g);
    } else {  // empty slot: zero row (value 0, never NaN) and masked in the softmax
      uint4 z = make_uint4(0, 0, 0, 0);
      uint4 *c = reinterpret_cast<uint4 *>(sm + kOffRawC + tid * 256);
      for (int i = 0; i < 16; ++i) c[i] = z;
      uint4 *s = reinterpret_cast<uint4 *>(sm + kOffRawS + tid * 32);
      s[0] = z;
      s[1] = z;
      mbar_arrive(&ms.bar_g);
    }
  }
  if (kQfp4) {  // prefill: exactly dequantised FP4 query rows into the swizzled Q chunks
    for (int v = tid; v < 64 * 64; v += kAttThreads) {
      const int h = v >> 6, rest = v & 63, kc = rest >> 3, u = rest & 7;
      uint4 w = make_uint4(0, 0, 0, 0);
      if (h < H) {
        const int64_t qrow = (int64_t)n * H + h;
        const int c0 = kc * 64 + u * 8;
        const uint32_t cw = *reinterpret_cast<const uint32_t *>(q_codes + qrow * kCodeBytes + c0 / 2);
        const float sc = e4m3_to_float(q_sf[qrow * kSfBytes + c0 / 16]);
        const uint32_t s2 = pack_bf16x2(sc, sc);
        w.x = bf16x2_mul(lut[cw & 0xFF], s2);
        w.y = bf16x2_mul(lut[(cw >> 8) & 0xFF], s2);
        w.z = bf16x2_mul(lut[(cw >> 16) & 0xFF], s2);
        w.w = bf16x2_mul(lut[cw >> 24], s2);
      }
      *reinterpret_cast<uint4 *>(sm + kOffQ + kc * 8192 + h * 128 + ((u ^ (h & 7)) << 4)) = w;
    }
  }
  bool ok = mbar_wait(&ms.bar_g, 0);

  // ---- 2. dequantise the rows once: chunk kc holds channels 64kc..64kc+63 of all 64 rows
  for (int v = tid; v < kAttTS * 64; v += kAttThreads) {
    const int j = v >> 6, rest = v & 63, kc = rest >> 3, u = rest & 7;
    const int c0 = kc * 64 + u * 8;
    const uint32_t cw = *reinterpret_cast<const uint32_t *>(sm + kOffRawC + j * 256 + c0 / 2);
    const float sc = e4m3_to_float(sm[kOffRawS + j * 32 + c0 / 16]);
    const uint32_t s2 = pack_bf16x2(sc, sc);
    uint4 w;
    w.x = bf16x2_mul(lut[cw & 0xFF], s2);
    w.y = bf16x2_mul(lut[(cw >> 8) & 0xFF], s2);
    w.z = bf16x2_mul(lut[(cw >> 16) & 0xFF], s2);
    w.w = bf16x2_mul(lut[cw >> 24], s2);
    *reinterpret_cast<uint4 *>(sm + kOffK + kc * 8192 + j * 128 + ((u ^ (j & 7)) << 4)) = w;
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- 3. S = Q Khat^T
  if (tid == 0) {
    if (!kQfp4) ok = ok && mbar_wait(&ms.bar_q, 0);
    constexpr uint32_t idesc = idesc_f32acc(1, 1, 128, kAttTS);
    const uint32_t qa = smem_u32(sm + kOffQ), ka = smem_u32(sm + kOffK);
    for (int kc = 0; kc < 8; ++kc)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_f16(tmem + kColS, desc_k128_sw128(qa + kc * 8192 + 32 * ks),
                desc_k128_sw128(ka + kc * 8192 + 32 * ks), idesc, (kc | ks) != 0);
    mma_commit(&ms.bar_s);
  }

  // ---- 4. softmax: warps 0,1 and 4,5 read TMEM lanes 0..63 (= heads); warps 0,1 take the
  //         columns (rows) 0..31 of S, warps 4,5 the columns 32..63
  if ((warp & 3) < 2) {
    ok = __all_sync(0xffffffffu, mbar_wait(&ms.bar_s, 0)) && ok;
    tc_fence_after();
    const int h = (warp & 3) * 32 + lane;
    const int half = warp >> 2, j0 = half * 32;
    float s[32];
    {
      const uint32_t la = tmem + kColS + j0 + ((uint32_t)((warp & 3) * 32) << 16);
      uint32_t r[2][16];
      tmem_ld16(la, r[0]);
      tmem_ld16(la + 16, r[1]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i) s[16 * c + i] = __uint_as_float(r[c][i]) * scale_log2e;
    }
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (ms.slot_ok[j0 + j]) m = fmaxf(m, s[j]);
    ms.mh[half][h] = m;
    asm volatile("bar.sync 1, 128;" ::: "memory");  // the four softmax warps
    m = fmaxf(ms.mh[0][h], ms.mh[1][h]);
    float l = 0.0f;
    uint32_t hi[16], lo[16];
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float p0 = ms.slot_ok[j0 + j] ? exp2f(s[j] - m) : 0.0f;
      const float p1 = ms.slot_ok[j0 + j + 1] ? exp2f(s[j + 1] - m) : 0.0f;
      l += p0 + p1;
      const __nv_bfloat16 h0 = __float2bfloat16_rn(p0), h1 = __float2bfloat16_rn(p1);
      hi[j / 2] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
      lo[j / 2] = pack_bf16x2(p0 - __bfloat162float(h0), p1 - __bfloat162float(h1));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int off = h * 128 + (((4 * half + u) ^ (h & 7)) << 4);
      *reinterpret_cast<uint4 *>(sm + kOffPhi + off) =
          make_uint4(hi[4 * u], hi[4 * u + 1], hi[4 * u + 2], hi[4 * u + 3]);
      *reinterpret_cast<uint4 *>(sm + kOffPlo + off) =
          make_uint4(lo[4 * u], lo[4 * u + 1], lo[4 * u + 2], lo[4 * u + 3]);
    }
    if (half == 0) ms.m2[h] = m;
    ms.lh[half][h] = l;
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- 5. O^T = Vhat^T P^T: M=128 channels (two chunks), N=64 heads, K=16 rows per MMA
  if (tid == 0) {
    constexpr uint32_t idesc_pv = idesc_f32acc(1, 1, 128, 64) | (1u << 15);  // A MN-major
    const uint32_t ka = smem_u32(sm + kOffK);
    const uint32_t ph = smem_u32(sm + kOffPhi), pl = smem_u32(sm + kOffPlo);
    for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
      for (int ks = 0; ks < kAttTS / 16; ++ks) {
        const uint64_t ad = desc_mn_sw128_atoms(ka + (2 * mb) * 8192 + ks * 16 * 128, 8192);
        mma_f16(tmem + mb * 64, ad, desc_k128_sw128(ph + 32 * ks), idesc_pv, ks != 0);
        mma_f16(tmem + mb * 64, ad, desc_k128_sw128(pl + 32 * ks), idesc_pv, 1);
      }
    }
    mma_commit(&ms.bar_o);
  }

  // ---- 6. epilogue: warp w reads lanes 32(w%4).. (channels) and heads 32(w/4)..+31 of every
  //         M block; column 64*mb + h of O^T is channel 128*mb + lane
  ok = __all_sync(0xffffffffu, mbar_wait(&ms.bar_o, 0)) && ok;
  tc_fence_after();
  {
    const int q4 = warp & 3, hh = warp >> 2;
    const uint32_t la = tmem + ((uint32_t)(q4 * 32) << 16);
    float *obase = o_part + ((int64_t)n * n_tiles + tile) * H * kD;
#pragma unroll 1
    for (int mb = 0; mb < 4; ++mb) {
      uint32_t r0[16], r1[16];
      tmem_ld16(la + mb * 64 + hh * 32, r0);
      tmem_ld16(la + mb * 64 + hh * 32 + 16, r1);
      tmem_ld_wait();
      float *oc = obase + mb * 128 + q4 * 32 + lane;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int h0 = hh * 32 + i, h1 = h0 + 16;
        if (h0 < H) oc[(int64_t)h0 * kD] = __uint_as_float(r0[i]);
        if (h1 < H) oc[(int64_t)h1 * kD] = __uint_as_float(r1[i]);
      }
    }
    if (tid < H) {
      const int64_t pr = ((int64_t)n * n_tiles + tile) * H + tid;
      m_part[pr] = ok ? ms.m2[tid] : -INFINITY;
      l_part[pr] = ok ? ms.lh[0][tid] + ms.lh[1][tid] : 0.0f;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kAttTmemCols);
}

// Merge the tiles of each (query, head): out = sum_t O_t 2^(m_t - M) / sum_t l_t 2^(m_t - M);
// lse = (M + log2 L) * ln 2.  m is in the log2 domain (logits * scale * log2 e).
// Grid (kD / 128, H, nq), 128 threads: thread = one channel.  The channel's partials of up to
// 32 tiles are loaded at once (before the weights are known), then summed in tile order.
constexpr int kCombBatch = 32;
__global__ void __launch_bounds__(128) attn_mma_combine_kernel(
    int H, int n_tiles, const float *__restrict__ o_part, const float *__restrict__ m_part,
    const float *__restrict__ l_part, uint16_t *__restrict__ out, float *__restrict__ lse) {
  __shared__ float wgt[256];
  __shared__ float sM, sL;
  pdl_wait();
  pdl_trigger();
  const int h = blockIdx.y, n = blockIdx.z, tid = threadIdx.x, lane = tid & 31;
  const int c = blockIdx.x * 128 + tid;
  const int64_t tstride = (int64_t)H * kD;  // floats between consecutive tiles
  const float *op = o_part + ((int64_t)n * n_tiles * H + h) * kD + c;
  float o[kCombBatch];
#pragma unroll
  for (int u = 0; u < kCombBatch; ++u) o[u] = u < n_tiles ? op[u * tstride] : 0.0f;
  if (tid < 32) {  // per-tile weights (n_tiles <= 256)
    float mt[8], lt[8];
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int t = lane + 32 * k;
      mt[k] = -INFINITY;
      lt[k] = 0.0f;
      if (t < n_tiles) {
        const int64_t pr = ((int64_t)n * n_tiles + t) * H + h;
        lt[k] = l_part[pr];
        mt[k] = m_part[pr];
        if (lt[k] > 0.0f) M = fmaxf(M, mt[k]);
      }
    }
    M = warp_max(M);
    float Lp = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int t = lane + 32 * k;
      if (t < n_tiles) {
        const float wv = (lt[k] > 0.0f) ? exp2f(mt[k] - M) : 0.0f;
        wgt[t] = wv;
        Lp += lt[k] * wv;
      }
    }
    Lp = warp_sum(Lp);
    if (lane == 0) {
      sM = M;
      sL = Lp;
    }
  }
  __syncthreads();
  float acc = 0.0f;
#pragma unroll
  for (int u = 0; u < kCombBatch; ++u)
    if (u < n_tiles) acc = fmaf(o[u], wgt[u], acc);
  for (int t0 = kCombBatch; t0 < n_tiles; t0 += kCombBatch) {
#pragma unroll
    for (int u = 0; u < kCombBatch; ++u) o[u] = t0 + u < n_tiles ? op[(t0 + u) * tstride] : 0.0f;
#pragma unroll
    for (int u = 0; u < kCombBatch; ++u)
      if (t0 + u < n_tiles) acc = fmaf(o[u], wgt[t0 + u], acc);
  }
  const float L = sL, M = sM;
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  out[((int64_t)n * H + h) * kD + c] = __bfloat16_as_ushort(__float2bfloat16_rn(acc * inv));
  if (blockIdx.x == 0 && tid == 0 && lse)
    lse[(int64_t)n * H + h] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------
bool attn_mma_supported(int H, int topk) {
  return H <= 64 && (topk + kAttTS - 1) / kAttTS <= 256 && encode_fn() != nullptr;
}

size_t attn_mma_workspace_bytes(int nq, int H, int topk) {
  const size_t tiles = (size_t)(topk + kAttTS - 1) / kAttTS;
  const size_t rows = (size_t)nq * tiles * H;
  return rows * kD * sizeof(float) + 2 * rows * sizeof(float) + 1024;
}

static bool make_q_map(CUtensorMap *m, const void *q, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rows <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(q), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

cudaError_t launch_attn_mma(const void *q_bf16, const uint8_t *q_codes, const uint8_t *q_sf,
                            int nq, int H, const int32_t *q_seq, const uint8_t *codes,
                            const uint8_t *sf, const int64_t *cu_ctx, const int32_t *idx,
                            int topk, float scale, void *out_bf16, float *lse, void *workspace,
                            cudaStream_t st) {
  if (nq == 0) return cudaSuccess;
  const int n_tiles = (topk + kAttTS - 1) / kAttTS;
  const size_t rows = (size_t)nq * n_tiles * H;
  float *o_part = static_cast<float *>(workspace);
  float *m_part = o_part + rows * kD;
  float *l_part = m_part + rows;
  CUtensorMap qm;
  memset(&qm, 0, sizeof(qm));
  if (q_bf16 && !make_q_map(&qm, q_bf16, (int64_t)nq * H)) return cudaErrorInvalidValue;
  const float scale_log2e = scale * 1.4426950408889634f;
  dim3 grid(n_tiles, nq);
  cudaError_t e;
  if (q_bf16) {
    e = set_smem_once(attn_mma_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kAttSmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(attn_mma_kernel<false>, grid, dim3(kAttThreads), kAttSmem, st, qm,
                   (const uint8_t *)nullptr, (const uint8_t *)nullptr, H, q_seq, codes, sf, cu_ctx,
                   idx, topk, scale_log2e, n_tiles, o_part, m_part, l_part);
  } else {
    e = set_smem_once(attn_mma_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kAttSmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(attn_mma_kernel<true>, grid, dim3(kAttThreads), kAttSmem, st, qm, q_codes,
                   q_sf, H, q_seq, codes, sf, cu_ctx, idx, topk, scale_log2e, n_tiles, o_part,
                   m_part, l_part);
  }
  note_launches(1);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attn_mma_combine_kernel, dim3(kD / 128, H, nq), dim3(128), 0, st, H, n_tiles,
                 (const float *)o_part, (const float *)m_part, (const float *)l_part,
                 static_cast<uint16_t *>(out_bf16), lse);
  note_launches(1);
  return e;
}

}  // namespace csa2

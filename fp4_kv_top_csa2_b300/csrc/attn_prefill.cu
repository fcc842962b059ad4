// attn_prefill.cu -- sparse attention for chunked prefill on the tensor cores (tcgen05).
//
// Each query token has its own Top-K rows (the indexer's causal selection); the query is
// quantised to FP4 with the main-KV rule and used exactly dequantised (fp16-exact).  One CTA
// owns one query token (all heads, H <= 64) and walks its rows in tiles of 64 with an online
// softmax, so no partial results leave the CTA:
//   S   = Qhat Khat^T      kind::f16 (fp16), M=128 (heads, padded) x N=64 rows, fp32, TMEM cols 256..319
//   O^T = Vhat^T P^T       kind::f16, M=128 channels x N=64 heads x K=16 rows per MMA, four
//                          channel blocks -> TMEM cols 0..255 (channels on lanes, heads on
//                          columns), accumulated over all tiles.
// Vhat^T is the dequantised tile read as an MN-major A operand (two 64-channel atoms 8 KB
// apart), P^T the softmax numerators as a K-major B operand in fp16 hi + lo parts.  The FP4-dequantised
// query and rows are exact in fp16 (at most 6 significant bits, magnitudes 2^-10..2688), so
// both products run as f16 x f16 with fp32 accumulation.
// The softmax keeps, per head, a reference maximum m_ref; numerators are 2^(s - m_ref) and
// m_ref moves only when a tile's maximum exceeds it by more than 2^10 -- then that head's
// column of O^T (and its running sum) is rescaled in TMEM.  The output row is O / l in bf16,
// lse = (m_ref + log2 l) * ln 2.
#include "sm100.cuh"

namespace csa2 {

constexpr int kPfTS = 64;
constexpr int kPfWorkers = 256;                // warps 0..7: gather, dequantise, softmax, epilogue
constexpr int kPfMmaWarp = 8;                  // warp 8: TMEM allocation and every MMA issue
constexpr int kPfThreads = kPfWorkers + 32;
constexpr float kPfRescale = 10.0f;  // log2 headroom before the reference maximum moves

constexpr int kPfOffQ = 0;                     // 8 chunks x (64 rows x 128 B) = 64 KB (+8 KB overrun)
constexpr int kPfOffK = 64 * 1024;             // 8 chunks x (64 rows x 128 B) = 64 KB
constexpr int kPfOffPhi = 128 * 1024;          // 64 rows (heads) x 128 B (64 rows of the tile)
constexpr int kPfOffPlo = 136 * 1024;
constexpr int kPfOffRaw = 144 * 1024;          // 2 x (64 x 256 B codes + 64 x 32 B scales)
constexpr int kPfRawBytes = kPfTS * 288;       // 18 KB
constexpr int kPfOffMisc = kPfOffRaw + 2 * kPfRawBytes;
constexpr int kPfSmem = kPfOffMisc + 2048 + 1024;

struct PfMisc {
  uint64_t bar_dq[4], bar_pv[4], bar_s, bar_p;
  uint32_t tmem_base;
  int any_rescale[2];
  int rows[2][kPfTS];  // the row of each slot of the tiles held in the two raw buffers
  float factor[64];
  float mhalf[2][64];  // per-half tile maxima (then the second half's running sums)
};
static_assert(sizeof(PfMisc) <= 2048, "misc block");

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  return (uint32_t)__half_as_ushort(__float2half_rn(lo)) |
         ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
}
__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  __half2 x = *reinterpret_cast<__half2 *>(&a);
  __half2 y = *reinterpret_cast<__half2 *>(&b);
  __half2 z = __hmul2(x, y);
  return *reinterpret_cast<uint32_t *>(&z);
}

// Two E2M1 codes (one byte, channel 2j in the low nibble) -> f16x2 of their values (exact;
// the low nibble goes to the low half).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(r) : "r"(byte));
  return r;
}
// One E4M3 scale byte -> f16x2 holding it twice (exact: E4M3 values are fp16 normals).
__device__ __forceinline__ uint32_t e4m3_to_f16x2_dup(uint32_t byte) {
  uint32_t r;
  const uint16_t two = (uint16_t)(byte | (byte << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
  return r;
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// The 64 rows of one tile (sequence-local row numbers in rows[], -1 = empty slot) into a raw
// buffer: 64 x (256 B codes + 32 B scales) as 1,152 16-byte cp.async copies spread over the
// 256 worker threads (empty slots are zero-filled).  Completion: cp.async.wait_all by every
// worker, then a workers' barrier.
__device__ __forceinline__ void pf_gather_tile(uint8_t *raw, const int *rows, int tid, int64_t base,
                                               const uint8_t *codes, const uint8_t *sf) {
  for (int i = tid; i < kPfTS * 18; i += kPfWorkers) {
    const int j = i / 18, part = i - j * 18;
    const int r = rows[j];
    uint8_t *dst = part < 16 ? raw + j * 256 + part * 16 : raw + kPfTS * 256 + j * 32 + (part - 16) * 16;
    if (r >= 0) {
      const int64_t row = base + r;
      const uint8_t *src = part < 16 ? codes + row * kCodeBytes + part * 16
                                     : sf + row * kSfBytes + (part - 16) * 16;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm100::smem_u32(dst)),
                   "l"(reinterpret_cast<uint64_t>(src))
                   : "memory");
    } else {
      *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

__global__ void __launch_bounds__(kPfThreads, 1) attn_prefill_kernel(
    const uint8_t *__restrict__ q_codes, const uint8_t *__restrict__ q_sf, int H,
    const int32_t *__restrict__ q_seq, const uint8_t *__restrict__ codes,
    const uint8_t *__restrict__ sf, const int64_t *__restrict__ cu_ctx,
    const int32_t *__restrict__ idx, int topk, float scale_log2e, uint16_t *__restrict__ out,
    float *__restrict__ lse) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t *sm = smem_raw + ((1024 - (raw_u32 & 1023)) & 1023);
  PfMisc &ms = *reinterpret_cast<PfMisc *>(sm + kPfOffMisc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = blockIdx.x;
  const int32_t *idx_n = idx + (int64_t)n * topk;
  const int n_tiles = (topk + kPfTS - 1) / kPfTS;

  if (tid == 0) {
    for (int c = 0; c < 4; ++c) {
      mbar_init(&ms.bar_dq[c], kPfWorkers);
      mbar_init(&ms.bar_pv[c], 1);
    }
    mbar_init(&ms.bar_s, 1);
    mbar_init(&ms.bar_p, kPfWorkers);
    ms.any_rescale[0] = 0;
    ms.any_rescale[1] = 0;
    fence_barrier_init();
  }
  if (warp == kPfMmaWarp) {
    tmem_alloc(&ms.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;
  const uint32_t tS = tmem + 256;
  pdl_wait();
  pdl_trigger();
  bool ok = true;

  if (warp == kPfMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f32acc(0, 0, 128, kPfTS);              // f16 x f16
      constexpr uint32_t idesc_pv = idesc_f32acc(0, 0, 128, 64) | (1u << 15);    // A MN-major
      const uint32_t qa = smem_u32(sm + kPfOffQ), ka = smem_u32(sm + kPfOffK);
      const uint32_t ph = smem_u32(sm + kPfOffPhi), pl = smem_u32(sm + kPfOffPlo);
      for (int t = 0; t < n_tiles; ++t) {
        // S = Qhat Khat^T, two chunks at a time as the workers finish them
        for (int cp = 0; cp < 4; ++cp) {
          ok = mbar_wait(&ms.bar_dq[cp], t & 1) && ok;
          tc_fence_after();
          for (int kc = 2 * cp; kc < 2 * cp + 2; ++kc)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_f16(tS, desc_k128_sw128(qa + kc * 8192 + 32 * ks),
                      desc_k128_sw128(ka + kc * 8192 + 32 * ks), idesc_qk, (kc | ks) != 0);
        }
        mma_commit(&ms.bar_s);
        // O^T += Vhat^T (P_hi + P_lo)^T, one commit per 128-channel block so the next tile's
        // dequantisation can reuse chunks 2qb, 2qb+1 as soon as block qb is done
        ok = mbar_wait(&ms.bar_p, t & 1) && ok;
        tc_fence_after();
        for (int qb = 0; qb < 4; ++qb) {
#pragma unroll
          for (int ks = 0; ks < kPfTS / 16; ++ks) {
            const uint64_t ad = desc_mn_sw128_atoms(ka + (2 * qb) * 8192 + ks * 16 * 128, 8192);
            mma_f16(tmem + qb * 64, ad, desc_k128_sw128(ph + 32 * ks), idesc_pv,
                    (t > 0 || ks > 0) ? 1u : 0u);
            mma_f16(tmem + qb * 64, ad, desc_k128_sw128(pl + 32 * ks), idesc_pv, 1u);
          }
          mma_commit(&ms.bar_pv[qb]);
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ workers (warps 0..7)
    const int64_t base = cu_ctx[q_seq[n]];
    // the row indices of tile t sit in ms.rows[t & 1]; thread tid < 64 loads slot tid of the
    // tile two ahead into r_next
    int r_next = -1;
    if (tid < kPfTS) {
      ms.rows[0][tid] = tid < topk ? idx_n[tid] : -1;
      ms.rows[1][tid] = kPfTS + tid < topk ? idx_n[kPfTS + tid] : -1;
      r_next = 2 * kPfTS + tid < topk ? idx_n[2 * kPfTS + tid] : -1;
    }
    asm volatile("bar.sync 2, 256;" ::: "memory");
    pf_gather_tile(sm + kPfOffRaw, ms.rows[0], tid, base, codes, sf);
    // the FP4 query, exactly dequantised into the swizzled Q chunks
    for (int v = tid; v < 64 * 64; v += kPfWorkers) {
      const int h = v >> 6, rest = v & 63, kc = rest >> 3, u = rest & 7;
      uint4 w = make_uint4(0, 0, 0, 0);
      if (h < H) {
        const int64_t qrow = (int64_t)n * H + h;
        const int c0 = kc * 64 + u * 8;
        const uint32_t cw =
            *reinterpret_cast<const uint32_t *>(q_codes + qrow * kCodeBytes + c0 / 2);
        const uint32_t s2 = e4m3_to_f16x2_dup(q_sf[qrow * kSfBytes + c0 / 16]);
        w.x = f16x2_mul(e2m1x2_to_f16x2(cw & 0xFF), s2);
        w.y = f16x2_mul(e2m1x2_to_f16x2((cw >> 8) & 0xFF), s2);
        w.z = f16x2_mul(e2m1x2_to_f16x2((cw >> 16) & 0xFF), s2);
        w.w = f16x2_mul(e2m1x2_to_f16x2(cw >> 24), s2);
      }
      *reinterpret_cast<uint4 *>(sm + kPfOffQ + kc * 8192 + h * 128 + ((u ^ (h & 7)) << 4)) = w;
    }
    // per-head softmax state: warps 0,1 (columns 0..31 of S) and 4,5 (columns 32..63) share
    // each head (thread = head = TMEM lane of S); both halves keep the same reference maximum
    // and their own running sums
    float m_ref = -INFINITY, l_run = 0.0f;
    for (int t = 0; t < n_tiles; ++t) {
      const int buf = t & 1;
      uint8_t *raw = sm + kPfOffRaw + buf * kPfRawBytes;
      asm volatile("cp.async.wait_all;" ::: "memory");  // this tile's rows (own copies)
      asm volatile("bar.sync 2, 256;" ::: "memory");      // ... and everyone's
      // prefetch the next tile's rows into the other raw buffer (dequantised last tile)
      if (t + 1 < n_tiles)
        pf_gather_tile(sm + kPfOffRaw + (buf ^ 1) * kPfRawBytes, ms.rows[buf ^ 1], tid, base,
                       codes, sf);
      // dequantise two chunks at a time, each pair once PV(t-1) no longer reads it
      for (int cp = 0; cp < 4; ++cp) {
        if (t > 0) ok = mbar_wait(&ms.bar_pv[cp], (t - 1) & 1) && ok;
#pragma unroll 4
        for (int v = tid; v < kPfTS * 16; v += kPfWorkers) {
          const int j = v >> 4, rest = v & 15, kc = 2 * cp + (rest >> 3), u = rest & 7;
          const int c0 = kc * 64 + u * 8;
          const uint32_t cw = *reinterpret_cast<const uint32_t *>(raw + j * 256 + c0 / 2);
          const uint32_t s2 = e4m3_to_f16x2_dup(raw[kPfTS * 256 + j * 32 + c0 / 16]);
          uint4 w;
          w.x = f16x2_mul(e2m1x2_to_f16x2(cw & 0xFF), s2);
          w.y = f16x2_mul(e2m1x2_to_f16x2((cw >> 8) & 0xFF), s2);
          w.z = f16x2_mul(e2m1x2_to_f16x2((cw >> 16) & 0xFF), s2);
          w.w = f16x2_mul(e2m1x2_to_f16x2(cw >> 24), s2);
          *reinterpret_cast<uint4 *>(sm + kPfOffK + kc * 8192 + j * 128 + ((u ^ (j & 7)) << 4)) =
              w;
        }
        fence_async_smem();
        mbar_arrive(&ms.bar_dq[cp]);
      }
      if ((warp & 3) < 2) {  // softmax rows: warps 0,1 columns 0..31, warps 4,5 columns 32..63
        ok = __all_sync(0xffffffffu, mbar_wait(&ms.bar_s, t & 1)) && ok;
        tc_fence_after();
        const int h = (warp & 3) * 32 + lane;
        const int sh = warp >> 2, j0 = sh * 32;
        float s[32];
        const uint32_t la = tS + j0 + ((uint32_t)((warp & 3) * 32) << 16);
        {
          uint32_t r[2][16];
          tmem_ld16(la, r[0]);
          tmem_ld16(la + 16, r[1]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int i = 0; i < 16; ++i) s[16 * c + i] = __uint_as_float(r[c][i]) * scale_log2e;
        }
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (ms.rows[buf][j0 + j] >= 0) mt = fmaxf(mt, s[j]);
        ms.mhalf[sh][h] = mt;
        asm volatile("bar.sync 1, 128;" ::: "memory");  // the four softmax warps
        mt = fmaxf(ms.mhalf[0][h], ms.mhalf[1][h]);
        float factor = 1.0f;
        if (mt > m_ref + kPfRescale) {  // (also true the first time: m_ref = -inf)
          if (m_ref != -INFINITY) {
            factor = exp2f(m_ref - mt);
            if (sh == 0) atomicOr(&ms.any_rescale[buf], 1);
          }
          l_run *= factor;
          m_ref = mt;
        }
        if (sh == 0) ms.factor[h] = factor;
        // numerators as fp16 hi + lo parts (p = hi + lo to ~2^-22): one fp16 operand alone
        // (2^-12) is too coarse when large rows of opposite sign nearly cancel.  P(t-1) is no
        // longer read: PV(t-1) is complete (every bar_pv of t-1 was waited above).
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float p0 = ms.rows[buf][j0 + j] >= 0 ? exp2f(s[j] - m_ref) : 0.0f;
          const float p1 = ms.rows[buf][j0 + j + 1] >= 0 ? exp2f(s[j + 1] - m_ref) : 0.0f;
          l_run += p0 + p1;
          const __half b0 = __float2half_rn(p0), b1 = __float2half_rn(p1);
          hi[j / 2] = (uint32_t)__half_as_ushort(b0) | ((uint32_t)__half_as_ushort(b1) << 16);
          lo[j / 2] = pack_f16x2(p0 - __half2float(b0), p1 - __half2float(b1));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int off = h * 128 + (((4 * sh + u) ^ (h & 7)) << 4);
          *reinterpret_cast<uint4 *>(sm + kPfOffPhi + off) =
              make_uint4(hi[4 * u], hi[4 * u + 1], hi[4 * u + 2], hi[4 * u + 3]);
          *reinterpret_cast<uint4 *>(sm + kPfOffPlo + off) =
              make_uint4(lo[4 * u], lo[4 * u + 1], lo[4 * u + 2], lo[4 * u + 3]);
        }
      }
      fence_async_smem();
      asm volatile("bar.sync 2, 256;" ::: "memory");  // the workers: P, factors, flag visible
      if (tid == 0) ms.any_rescale[buf ^ 1] = 0;      // its readers (tile t-1) are all past
      if (ms.any_rescale[buf] && warp < 4) {  // O^T[:, h] *= factor[h]: thread = channel lane
        tc_fence_after();
        const uint32_t la = tmem + ((uint32_t)(warp * 32) << 16);
        for (int c = 0; c < 256; c += 16) {
          uint32_t r[16];
          tmem_ld16(la + c, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            r[i] = __float_as_uint(__uint_as_float(r[i]) * ms.factor[(c + i) & 63]);
          tmem_st16(la + c, r);
        }
        tmem_st_wait();
      }
      // the slots of tile t+2 go where tile t's were (tile t's readers are past the barrier
      // above); the barrier below publishes them for the gather issued at tile t+1
      if (tid < kPfTS) {
        ms.rows[buf][tid] = r_next;
        const int slot = (t + 3) * kPfTS + tid;
        r_next = slot < topk ? idx_n[slot] : -1;
      }
      tc_fence_before();
      asm volatile("bar.sync 2, 256;" ::: "memory");  // factors read before they change
      mbar_arrive(&ms.bar_p);
    }
    // ---- epilogue: thread = channel lane; column 64*qb + h of O^T is channel 128*qb + lane'
    ok = mbar_wait(&ms.bar_pv[3], (n_tiles - 1) & 1) && ok;
    tc_fence_after();
    if ((warp & 3) < 2) {  // publish the final per-head state through shared memory
      const int h = (warp & 3) * 32 + lane;
      if (warp >= 4) ms.mhalf[1][h] = l_run;  // the second half's running sum
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (warp < 4) {
        const float l = l_run + ms.mhalf[1][h];
        ms.factor[h] = (l > 0.0f && ok) ? 1.0f / l : 0.0f;
        if (h < H && lse)
          lse[(int64_t)n * H + h] = (l > 0.0f && ok) ? (m_ref + log2f(l)) * 0.69314718055994531f
                                                     : -INFINITY;
      }
    }
    asm volatile("bar.sync 2, 256;" ::: "memory");
    if (warp < 4) {
      const uint32_t la = tmem + ((uint32_t)(warp * 32) << 16);
      const int cl = warp * 32 + lane;  // channel within a 128-channel block
      for (int qb = 0; qb < 4; ++qb) {
        for (int h0 = 0; h0 < 64; h0 += 16) {
          uint32_t r[16];
          tmem_ld16(la + qb * 64 + h0, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int h = h0 + i;
            if (h < H)
              out[((int64_t)n * H + h) * kD + qb * 128 + cl] =
                  __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[i]) * ms.factor[h]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kPfMmaWarp) tmem_dealloc(tmem, 512);
}

bool attn_prefill_supported(int H) { return H <= 64 && encode_fn() != nullptr; }

cudaError_t launch_attn_prefill(const uint8_t *q_codes, const uint8_t *q_sf, int T, int H,
                                const int32_t *q_seq, const uint8_t *codes, const uint8_t *sf,
                                const int64_t *cu_ctx, const int32_t *idx, int topk, float scale,
                                void *out_bf16, float *lse, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  cudaError_t e = set_smem_once(attn_prefill_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attn_prefill_kernel, dim3(T), dim3(kPfThreads), kPfSmem, st, q_codes, q_sf, H,
                 q_seq, codes, sf, cu_ctx, idx, topk, scale * 1.4426950408889634f,
                 static_cast<uint16_t *>(out_bf16), lse);
  note_launches(1);
  return e;
}

}  // namespace csa2

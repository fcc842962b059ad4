// attn_prefill.cu -- sparse attention for chunked prefill on the tensor cores (tcgen05).
//
// Each query token has its own Top-K rows (the indexer's causal selection); the query is
// quantised to FP4 with the main-KV rule (16-channel E4M3 scales, E2M1 values) and used exactly
// dequantised.  One CTA owns one query token (all heads, H <= 64) and walks its selected rows in
// tiles of 128 with an online softmax, so no partial result leaves the CTA:
//   S^T = Khat Qhat^T   kind::f16, M=128 rows x N=64 heads x K=512, fp32 in TMEM cols 448..511
//                       (rows on the M side: no padding of the 64 heads up to M=128)
//   O^T = Vhat^T P^T    kind::f16, M=128 channels x K=16 rows per MMA, four channel blocks
//                       (channels on TMEM lanes, heads on columns), accumulated over all tiles.
//                       Blocks 0..2 take P_hi and P_lo side by side as one N=128 operand and keep
//                       two accumulators (cols 128qb + h and 128qb + 64 + h, summed at the end);
//                       block 3 adds both into one N=64 accumulator (cols 384 + h), two MMAs.
// Khat is the tile's dequantised rows [row][channel] in eight 128B-swizzled chunks of 64
// channels: the K-major A operand of S^T and, read channel-major, the MN-major A operand Vhat^T
// of O^T.  P^T is written by the softmax threads one tile row per thread (64 heads = one 128-byte
// line), the MN-major B operand of O^T, in fp16 hi + lo parts (P = hi + lo to ~2^-22; a single
// fp16 operand, 2^-11 relative, is too coarse for the stated output tolerance).
// The FP4-dequantised query and rows are exact in fp16 (at most 6 significant bits, magnitudes
// 2^-10..2688), so both products run as f16 x f16 with fp32 accumulation.
//
// Softmax: a thread holds one tile row (a TMEM lane of S^T) and 32 heads.  Each head keeps a
// reference maximum m_ref (shared memory); numerators are 2^(s - m_ref) and each thread keeps its
// rows' partial sums per head in registers, reduced across rows once per token.  m_ref moves only
// when some score exceeds it by more than 2^8 (always on the first tile with a valid row): then
// the tile's maximum per head is reduced across rows, and that head's O^T column and partial sums
// are rescaled.  The output is O / l in bf16, lse = (m_ref + log2 l) * ln 2.
//
// Local window (the sliding-window branch: "DeepSeek V4.1-Flash", aiwiki.ai, section "Compressed
// Sparse Attention 2", every layer's own local keys and values, stored in FP8 per section
// "KV-cache formats and bounded replay"): after the selected rows' tiles come tiles of 64 local
// E4M3 rows (the last n_win positions the token sees; rows 64..127 of those tiles are empty),
// decoded exactly to fp16, so one softmax covers the selected rows and the window.
//
// Roles: warps 0..7 load the next tile's rows from L2 into registers (16-byte loads, one tile
// ahead, row numbers two tiles ahead), dequantise them into Khat one 128-channel chunk pair at a
// time as the previous tile's O^T MMAs release it, run the softmax and the epilogue; warp 8
// allocates TMEM and issues every MMA.
#include "sm100.cuh"

namespace csa2 {

constexpr int kPfRows = 128;                   // selected rows per tile (M of S^T)
constexpr int kPfWorkers = 256;                // warps 0..7
constexpr int kPfMmaWarp = 8;                  // warp 8: TMEM allocation and MMA issue
constexpr int kPfThreads = kPfWorkers + 32;
constexpr float kPfHeadroom = 8.0f;            // log2 headroom above the reference maximum
constexpr int kPfWinRows = 64;                 // local rows per window tile

constexpr int kPfQChunk = 64 * 128;            // one 64-channel chunk of Qhat: 64 heads x 128 B
constexpr int kPfKChunk = kPfRows * 128;       // one 64-channel chunk of Khat: 128 rows x 128 B
constexpr int kPfOffQ = 0;                     // 8 Q chunks = 64 KB
constexpr int kPfOffK = 8 * kPfQChunk;         // 8 K chunks = 128 KB
constexpr int kPfOffPhi = kPfOffK + 8 * kPfKChunk;  // P^T hi: 128 rows x 128 B = 16 KB
constexpr int kPfOffPlo = kPfOffPhi + kPfRows * 128;
constexpr int kPfOffMisc = kPfOffPlo + kPfRows * 128;
constexpr int kPfSmem = kPfOffMisc + 1024 + 1024;  // misc block + 1024-byte alignment slack
static_assert(kPfSmem <= 232448, "shared memory per CTA");

struct PfMisc {
  uint64_t bar_q, bar_s, bar_p, bar_dq[4], bar_pv[4];
  uint64_t bar_v[2];  // full-FP4 PV variant: channel blocks 0-1 / 2-3 re-quantised
  uint32_t tmem_base;
  int flag[2];   // per tile parity: some score exceeded its reference maximum
  __align__(16) float mref[64];    // per-head reference maximum (log2 domain); read as float4
  __align__(16) float factor[64];  // per-head rescale factor of the current tile; read as float4
  float inv_l[64];
};
static_assert(offsetof(PfMisc, mref) % 16 == 0 && offsetof(PfMisc, factor) % 16 == 0,
              "float4 reads of mref / factor");
static_assert(sizeof(PfMisc) <= 1024, "misc block");

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
// Two E4M3 bytes (low byte = lower channel) -> f16x2 of their values (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)two));
  return r;
}
// One E4M3 scale byte -> f16x2 holding it twice (exact: E4M3 values are fp16 normals).
__device__ __forceinline__ uint32_t e4m3_to_f16x2_dup(uint32_t byte) {
  uint32_t r;
  const uint16_t two = (uint16_t)(byte | (byte << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
  return r;
}
// Eight E2M1 codes (one 32-bit word, channel 2j in nibble 2j) times one scale -> 8 fp16 values.
__device__ __forceinline__ uint4 dequant8(uint32_t word, uint32_t s2) {
  uint4 w;
  w.x = f16x2_mul(e2m1x2_to_f16x2(word & 0xFF), s2);
  w.y = f16x2_mul(e2m1x2_to_f16x2((word >> 8) & 0xFF), s2);
  w.z = f16x2_mul(e2m1x2_to_f16x2((word >> 16) & 0xFF), s2);
  w.w = f16x2_mul(e2m1x2_to_f16x2(word >> 24), s2);
  return w;
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  sm100::tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
      "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
      "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
      "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
      "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x on the special-function unit (approximate to a few ulp; -inf gives +0).  The numerators
// are then rounded to fp16 hi + lo parts, and both the output and its normaliser use them.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Warp-wide reduce-scatter of 32 values per lane: afterwards lane i holds op over the 32 lanes
// of value i (31 shuffles: at each step a lane keeps half of its values and sends the other
// half to its partner).
template <bool MAX>
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = lane & o;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float keep = upper ? v[i + o] : v[i], send = upper ? v[i] : v[i + o];
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

__device__ __forceinline__ void pf_bar_workers() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// WIN: the local window's tiles follow the selected rows' (compiled separately so the kernel
// without a window keeps its registers).
template <bool WIN>
__global__ void __launch_bounds__(kPfThreads, 1) attn_prefill_kernel(
    const uint16_t *__restrict__ q_bf16, int H, const int32_t *__restrict__ q_seq,
    const uint8_t *__restrict__ codes, const uint8_t *__restrict__ sf,
    const int64_t *__restrict__ cu_ctx, const int32_t *__restrict__ idx, int topk,
    float scale_log2e, uint16_t *__restrict__ out, float *__restrict__ lse,
    const int32_t *__restrict__ q_vis, const uint8_t *__restrict__ swa_kv, int ring, int n_win) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t *sm = smem_raw + ((1024 - (raw_u32 & 1023)) & 1023);
  PfMisc &ms = *reinterpret_cast<PfMisc *>(sm + kPfOffMisc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = blockIdx.x;
  const int32_t *idx_n = idx + (int64_t)n * topk;
  const int n_sel = (topk + kPfRows - 1) / kPfRows;  // tiles of selected rows
  const int n_tiles = n_sel + (WIN ? (n_win + kPfWinRows - 1) / kPfWinRows : 0);

  if (tid == 0) {
    mbar_init(&ms.bar_q, kPfWorkers);
    mbar_init(&ms.bar_s, 1);
    mbar_init(&ms.bar_p, kPfWorkers);
    for (int c = 0; c < 4; ++c) {
      mbar_init(&ms.bar_dq[c], kPfWorkers);
      mbar_init(&ms.bar_pv[c], 1);
    }
    ms.flag[0] = 0;
    ms.flag[1] = 0;
    fence_barrier_init();
  }
  if (tid < 64) ms.mref[tid] = -INFINITY;
  if (warp == kPfMmaWarp) {
    tmem_alloc(&ms.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;  // O^T: columns 0..447; S^T: columns 448..511
  const uint32_t tS = tmem + 448;
  pdl_wait();
  pdl_trigger();
  bool ok = true;

  if (warp == kPfMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f32acc(0, 0, 128, 64);  // f16 x f16, both K-major
      constexpr uint32_t mn = (1u << 15) | (1u << 16);            // A and B MN-major
      constexpr uint32_t idesc_pv2 = idesc_f32acc(0, 0, 128, 128) | mn;  // [P_hi | P_lo]
      constexpr uint32_t idesc_pv1 = idesc_f32acc(0, 0, 128, 64) | mn;
      const uint32_t qa = smem_u32(sm + kPfOffQ), ka = smem_u32(sm + kPfOffK);
      const uint32_t ph = smem_u32(sm + kPfOffPhi), pl = smem_u32(sm + kPfOffPlo);
      constexpr uint32_t kHiLo = kPfOffPlo - kPfOffPhi;  // P_lo is P_hi's second N atom
      ok = mbar_wait(&ms.bar_q, 0) && ok;
      for (int t = 0; t < n_tiles; ++t) {
        // S^T = Khat Qhat^T, chunk pair by chunk pair as the workers dequantise them
        for (int cp = 0; cp < 4; ++cp) {
          ok = mbar_wait(&ms.bar_dq[cp], t & 1) && ok;
          tc_fence_after();
#pragma unroll
          for (int kc = 2 * cp; kc < 2 * cp + 2; ++kc)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_f16(tS, desc_k128_sw128(ka + kc * kPfKChunk + 32 * ks),
                      desc_k128_sw128(qa + kc * kPfQChunk + 32 * ks), idesc_s, (kc | ks) != 0);
        }
        mma_commit(&ms.bar_s);
        // O^T += Vhat^T (P_hi + P_lo)^T, committed per 128-channel block so the next tile's
        // dequantisation can reuse chunks 2qb, 2qb+1 as soon as block qb is done
        ok = mbar_wait(&ms.bar_p, t & 1) && ok;
        tc_fence_after();
        for (int qb = 0; qb < 4; ++qb) {
#pragma unroll
          for (int ks = 0; ks < kPfRows / 16; ++ks) {
            const uint64_t ad =
                desc_mn_sw128_atoms(ka + (2 * qb) * kPfKChunk + ks * 16 * 128, kPfKChunk);
            const uint32_t acc = (t > 0 || ks > 0) ? 1u : 0u;
            if (qb < 3) {
              mma_f16(tmem + qb * 128, ad, desc_mn_sw128_atoms(ph + ks * 16 * 128, kHiLo),
                      idesc_pv2, acc);
            } else {
              mma_f16(tmem + 384, ad, desc_mn_sw128_atoms(ph + ks * 16 * 128, kHiLo), idesc_pv1,
                      acc);
              mma_f16(tmem + 384, ad, desc_mn_sw128_atoms(pl + ks * 16 * 128, kHiLo), idesc_pv1,
                      1u);
            }
          }
          mma_commit(&ms.bar_pv[qb]);
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ workers (warps 0..7)
    const int64_t base = cu_ctx[q_seq[n]];
    // dequantisation role: in every 128-channel chunk pair a thread owns the 32-channel segment
    // `seg` of rows jr and jr + 64
    const int seg = tid & 3, jr = tid >> 2;
    // softmax role: TMEM lane quarter and head half
    const int quarter = warp & 3, hh = warp >> 2;
    const int jrow = quarter * 32 + lane;  // the tile row this thread's S^T lane holds
    uint4 rc[8];     // codes of (chunk pair cp, row half) at 2 cp + half
    uint32_t rs[8];  // the two scales of each
    // Row numbers run two tiles ahead of the row data, so issuing a tile's data loads never
    // waits for its index loads.  For a window tile, ri[0] is the local row of this thread's
    // window slot (rows 64..127 of the tile are empty) and win_next is set.
    int ri[2], rrow = -1, rrow_next = -1;
    bool win_ri = false;
    const int64_t vis = WIN ? q_vis[n] : 0;
    const int64_t nw = vis < n_win ? vis : n_win;  // window length of this token
    const int64_t lbase = (int64_t)q_seq[n] * ring;
    auto load_idx = [&](int t) {
      if (!WIN || t < n_sel) {
        win_ri = false;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int slot = t * kPfRows + jr + 64 * hf;
          ri[hf] = slot < topk ? __ldg(idx_n + slot) : -1;
        }
        const int slot = t * kPfRows + jrow;
        rrow_next = slot < topk ? __ldg(idx_n + slot) : -1;
      } else {  // window tile: slot wi of the last nw positions t = vis - nw + wi
        win_ri = true;
        const int64_t w0 = (int64_t)(t - n_sel) * kPfWinRows;
        const int64_t wi = w0 + jr;
        ri[0] = (t < n_tiles && wi < nw) ? (int)((vis - nw + wi) % ring) : -1;
        ri[1] = -1;
        rrow_next = (t < n_tiles && jrow < kPfWinRows && w0 + jrow < nw) ? 0 : -1;
      }
    };
    auto load_rows = [&]() {
      if (WIN && win_ri) {  // 32 channels of E4M3 per chunk pair: two 16-byte loads
        const int64_t row = lbase + (ri[0] >= 0 ? ri[0] : 0);
#pragma unroll
        for (int cp = 0; cp < 4; ++cp) {
#pragma unroll
          for (int k = 0; k < 2; ++k)
            rc[2 * cp + k] = ri[0] >= 0 ? __ldg(reinterpret_cast<const uint4 *>(
                                              swa_kv + row * kD + cp * 128 + seg * 32 + 16 * k))
                                        : make_uint4(0, 0, 0, 0);
        }
        return;
      }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int64_t row = base + (ri[hf] >= 0 ? ri[hf] : 0);
#pragma unroll
        for (int cp = 0; cp < 4; ++cp) {
          if (ri[hf] >= 0) {
            rc[2 * cp + hf] = __ldg(reinterpret_cast<const uint4 *>(
                codes + row * kCodeBytes + cp * 64 + seg * 16));
            rs[2 * cp + hf] = __ldg(reinterpret_cast<const uint16_t *>(
                sf + row * kSfBytes + cp * 8 + seg * 2));
          } else {
            rc[2 * cp + hf] = make_uint4(0, 0, 0, 0);
            rs[2 * cp + hf] = 0;
          }
        }
      }
    };
    load_idx(0);
    load_rows();  // tile 0's rows
    rrow = rrow_next;
    load_idx(1);  // tile 1's row numbers

    // ---- the query: FP4-quantised per (token, head) row with the main-KV rule, then exactly
    //      dequantised into the eight swizzled Q chunks (heads >= H are zero).  Thread: eight
    //      16-channel groups of one head (all loads first).
    {
      constexpr int kGroups = 64 * 32 / kPfWorkers;  // 8
      uint4 qa[kGroups], qb[kGroups];
#pragma unroll
      for (int k = 0; k < kGroups; ++k) {
        const int gi = tid + k * kPfWorkers, h = gi >> 5, grp = gi & 31;
        if (h < H) {
          const uint4 *src = reinterpret_cast<const uint4 *>(
              q_bf16 + ((int64_t)n * H + h) * kD + 16 * grp);
          qa[k] = __ldg(src);
          qb[k] = __ldg(src + 1);
        }
      }
#pragma unroll
      for (int k = 0; k < kGroups; ++k) {
        const int gi = tid + k * kPfWorkers, h = gi >> 5, grp = gi & 31;
        uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0;
        if (h < H) {
          const uint32_t v[8] = {qa[k].x, qa[k].y, qa[k].z, qa[k].w,
                                 qb[k].x, qb[k].y, qb[k].z, qb[k].w};
          uint64_t packed;
          const uint32_t s2 = e4m3_to_f16x2_dup(quant_group16(v, &packed));
          w0 = dequant8((uint32_t)packed, s2);
          w1 = dequant8((uint32_t)(packed >> 32), s2);
        }
        const int kc = grp >> 2, u = (grp & 3) * 2;
        uint8_t *dst = sm + kPfOffQ + kc * kPfQChunk + h * 128;
        *reinterpret_cast<uint4 *>(dst + ((u ^ (h & 7)) << 4)) = w0;
        *reinterpret_cast<uint4 *>(dst + (((u + 1) ^ (h & 7)) << 4)) = w1;
      }
    }
    fence_async_smem();
    mbar_arrive(&ms.bar_q);

    float lpart[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) lpart[i] = 0.0f;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;

    for (int t = 0; t < n_tiles; ++t) {
      // ---- dequantise this tile into Khat, one chunk pair at a time as O^T(t-1) releases it
#pragma unroll
      for (int cp = 0; cp < 4; ++cp) {
        if (t > 0) ok = mbar_wait(&ms.bar_pv[cp], (t - 1) & 1) && ok;
        const int kc = 2 * cp + (seg >> 1), u0 = (seg & 1) * 4;
        if (!WIN || t < n_sel) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int j = jr + 64 * hf;
            const uint4 c = rc[2 * cp + hf];
            const uint32_t r = rs[2 * cp + hf];
            const uint32_t sa = e4m3_to_f16x2_dup(r & 0xFF), sb = e4m3_to_f16x2_dup(r >> 8);
            uint8_t *row = sm + kPfOffK + kc * kPfKChunk + j * 128;
            *reinterpret_cast<uint4 *>(row + (((u0 + 0) ^ (j & 7)) << 4)) = dequant8(c.x, sa);
            *reinterpret_cast<uint4 *>(row + (((u0 + 1) ^ (j & 7)) << 4)) = dequant8(c.y, sa);
            *reinterpret_cast<uint4 *>(row + (((u0 + 2) ^ (j & 7)) << 4)) = dequant8(c.z, sb);
            *reinterpret_cast<uint4 *>(row + (((u0 + 3) ^ (j & 7)) << 4)) = dequant8(c.w, sb);
          }
        } else {  // window tile: row jr from 32 E4M3 bytes, row jr + 64 empty
          uint8_t *row = sm + kPfOffK + kc * kPfKChunk + jr * 128;
          uint8_t *row2 = row + 64 * 128;
          const uint32_t b[8] = {rc[2 * cp].x, rc[2 * cp].y, rc[2 * cp].z, rc[2 * cp].w,
                                 rc[2 * cp + 1].x, rc[2 * cp + 1].y, rc[2 * cp + 1].z,
                                 rc[2 * cp + 1].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 w;
            w.x = e4m3x2_to_f16x2(b[2 * k] & 0xFFFF);
            w.y = e4m3x2_to_f16x2(b[2 * k] >> 16);
            w.z = e4m3x2_to_f16x2(b[2 * k + 1] & 0xFFFF);
            w.w = e4m3x2_to_f16x2(b[2 * k + 1] >> 16);
            *reinterpret_cast<uint4 *>(row + (((u0 + k) ^ (jr & 7)) << 4)) = w;
            *reinterpret_cast<uint4 *>(row2 + (((u0 + k) ^ (jr & 7)) << 4)) =
                make_uint4(0, 0, 0, 0);
          }
        }
        fence_async_smem();
        mbar_arrive(&ms.bar_dq[cp]);
      }
      const bool row_ok = rrow >= 0;
      if (t + 1 < n_tiles) {  // tile t+1's rows in flight during this tile's softmax
        load_rows();
        rrow = rrow_next;
        load_idx(t + 2);
      }

      // ---- softmax of tile t: this thread's row, heads 32hh..32hh+31; x = log2 numerator
      ok = __all_sync(0xffffffffu, mbar_wait(&ms.bar_s, t & 1)) && ok;
      tc_fence_after();
      float x[32];
      tmem_ld32(tS + 32 * hh + lane_off, x);
      const float *mref = &ms.mref[32 * hh];
      bool exceed = false;
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 m4 = *reinterpret_cast<const float4 *>(mref + i);
        const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          x[i + k] = row_ok ? fmaf(x[i + k], scale_log2e, -mv[k]) : -INFINITY;
          exceed |= x[i + k] > kPfHeadroom;
        }
      }
      if (__any_sync(0xffffffffu, exceed) && lane == 0) ms.flag[t & 1] = 1;
      pf_bar_workers();
      const bool slow = ms.flag[t & 1] != 0;
      if (tid == 0) ms.flag[(t + 1) & 1] = 0;  // its readers (tile t-1) are past the barrier
      if (slow) {
        // the tile's maximum per head: over this warp's 32 rows, then over the four quarters
        float *scratch = reinterpret_cast<float *>(sm + kPfOffPlo);  // [4][64], P(t) not yet written
        tmem_ld32(tS + 32 * hh + lane_off, x);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = row_ok ? x[i] * scale_log2e : -INFINITY;
        scratch[quarter * 64 + 32 * hh + lane] = reduce_scatter32<true>(x, lane);
        pf_bar_workers();
        if (quarter == 0) {  // warps 0 and 4: head 32hh + lane
          const int h = 32 * hh + lane;
          const float tm = fmaxf(fmaxf(scratch[h], scratch[64 + h]),
                                 fmaxf(scratch[128 + h], scratch[192 + h]));
          const float old = ms.mref[h];
          const float nm = tm > old + kPfHeadroom ? tm : old;
          ms.factor[h] = nm == old ? 1.0f : exp2f(old - nm);  // old = -inf: 0 (nothing yet)
          ms.mref[h] = nm;
        }
        pf_bar_workers();
        const float *fac = &ms.factor[32 * hh];
        bool any_change = false;
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 f4 = *reinterpret_cast<const float4 *>(fac + i);
          lpart[i] *= f4.x, lpart[i + 1] *= f4.y, lpart[i + 2] *= f4.z, lpart[i + 3] *= f4.w;
          any_change |= f4.x != 1.0f || f4.y != 1.0f || f4.z != 1.0f || f4.w != 1.0f;
        }
        if (t > 0 && __any_sync(0xffffffffu, any_change)) {
          // O^T[:, h] *= factor[h] for every accumulator column of head h (O^T(t-1) is
          // complete: S^T(t) was committed after it); this warp: lane quarter `quarter`, heads
          // 32hh..32hh+31
#pragma unroll 1
          for (int c = 0; c < 7; ++c) {  // column groups 0, 64, ..., 384 (+32hh)
            const uint32_t ta = tmem + c * 64 + 32 * hh + lane_off;
            float o[32];
            tmem_ld32(ta, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= fac[i];
            tmem_st32(ta, o);
          }
        }
        tmem_ld32(tS + 32 * hh + lane_off, x);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          x[i] = row_ok ? fmaf(x[i], scale_log2e, -mref[i]) : -INFINITY;
      }
      // numerators 2^x as fp16 hi + lo parts, eight heads (one 16-byte unit) at a time; P^T row
      // jrow, heads 32hh..32hh+31 = units 4hh..4hh+3.  An empty row has x = -inf, so 0.
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
          const int i = 8 * u + k;
          const float p0 = ex2_approx(x[i]), p1 = ex2_approx(x[i + 1]);
          const __half2 h2 = __floats2half2_rn(p0, p1);
          const float2 f2 = __half22float2(h2);
          const __half2 l2 = __floats2half2_rn(p0 - f2.x, p1 - f2.y);
          lpart[i] += p0;
          lpart[i + 1] += p1;
          hi[k / 2] = *reinterpret_cast<const uint32_t *>(&h2);
          lo[k / 2] = *reinterpret_cast<const uint32_t *>(&l2);
        }
        const int off = jrow * 128 + (((4 * hh + u) ^ (jrow & 7)) << 4);
        *reinterpret_cast<uint4 *>(sm + kPfOffPhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(sm + kPfOffPlo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&ms.bar_p);
    }

    // ---- epilogue: row sums per head, lse, O / l in bf16
    ok = __all_sync(0xffffffffu, mbar_wait(&ms.bar_pv[3], (n_tiles - 1) & 1)) && ok;
    tc_fence_after();
    float *scratch = reinterpret_cast<float *>(sm + kPfOffPlo);  // P is no longer read
    scratch[quarter * 64 + 32 * hh + lane] = reduce_scatter32<false>(lpart, lane);
    pf_bar_workers();
    if (quarter == 0) {
      const int h = 32 * hh + lane;
      const float l = scratch[h] + scratch[64 + h] + scratch[128 + h] + scratch[192 + h];
      ms.inv_l[h] = (l > 0.0f && ok) ? 1.0f / l : 0.0f;
      if (h < H && lse)
        lse[(int64_t)n * H + h] =
            (l > 0.0f && ok) ? (ms.mref[h] + log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
    pf_bar_workers();
    float inv[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) inv[i] = ms.inv_l[32 * hh + i];
    const int hn = min(32, H - 32 * hh);  // real heads of this half
#pragma unroll 1
    for (int qb = 0; qb < 4; ++qb) {
      float o[32];
      tmem_ld32(tmem + (qb < 3 ? qb * 128 : 384) + 32 * hh + lane_off, o);
      if (qb < 3) {
        float o2[32];
        tmem_ld32(tmem + qb * 128 + 64 + 32 * hh + lane_off, o2);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] += o2[i];
      }
      uint16_t *oc = out + ((int64_t)n * H + 32 * hh) * kD + qb * 128 + quarter * 32 + lane;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < hn) oc[(int64_t)i * kD] = __bfloat16_as_ushort(__float2bfloat16_rn(o[i] * inv[i]));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kPfMmaWarp) tmem_dealloc(tmem, 512);
}

bool attn_prefill_supported(int H) { return H <= 64 && encode_fn() != nullptr; }

cudaError_t launch_attn_prefill(const void *q_bf16, int T, int H, const int32_t *q_seq,
                                const uint8_t *codes, const uint8_t *sf, const int64_t *cu_ctx,
                                const int32_t *idx, int topk, float scale, void *out_bf16,
                                float *lse, cudaStream_t st, const int32_t *q_vis,
                                const uint8_t *swa_kv, int ring, int n_win) {
  if (T == 0) return cudaSuccess;
  auto go = [&](auto kern) {
    cudaError_t err = set_smem_once(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(T), dim3(kPfThreads), kPfSmem, st,
                      static_cast<const uint16_t *>(q_bf16), H, q_seq, codes, sf, cu_ctx, idx,
                      topk, scale * 1.4426950408889634f, static_cast<uint16_t *>(out_bf16), lse,
                      q_vis, swa_kv, ring, n_win);
  };
  const cudaError_t e = n_win > 0 ? go(attn_prefill_kernel<true>) : go(attn_prefill_kernel<false>);
  note_launches(1);
  return e;
}

}  // namespace csa2

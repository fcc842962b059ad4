// attn_small.cu -- the decode attention's tile kernel for few tiles (one or two decoding
// sequences): small tiles that spread one query over many SMs.  attn_mma.cu holds the
// tile kernel for many tiles; both produce the same partials for their combine.
//
// For sequence n, head h: softmax_j(scale * q_h . khat_j) over the selected rows j, applied to
// the same rows (K = V = the dequantised latent row; the model card's Introduction, CSA2
// paragraph: the sparse attention reads the FP4 main-KV rows that a shared Top-K index set names).
//
// One CTA = one query (sequence) x one tile of 32 selected rows x one group of 32 heads (M=128
// MMA shape, heads padded).  Small tiles keep the chain of dependent steps short and spread one
// query over many SMs (64 x 2 CTAs for 2,048 rows and 64 heads).  Steps:
//   1. Q [32 heads x 512] bf16 arrives by TMA as eight 128B-swizzled K-chunks of 64 channels;
//      the selected rows (256 B of codes, 32 B of scales each) arrive as 16-byte cp.async copies
//      spread over all threads (many small copies issue faster this way than one bulk copy
//      per row).
//   2. Every row is dequantised exactly (E2M1 x E4M3 has <= 6 significant bits) to bf16 and
//      stored once, as eight 128B-swizzled chunks [32 rows x 64 channels].
//   3. S = Q Khat^T: kind::f16, M=128 (heads) x N=32 (rows) x K=512, fp32 in TMEM.
//   4. Softmax rows (exp2 domain; two warps, one per 16-column half of S), P split into bf16
//      hi + lo parts (P ~ hi + lo to 2^-17).
//   5. O^T = Vhat^T (P_hi + P_lo)^T: kind::f16, the same dequantised chunks read as the
//      MN-major A operand (channels contiguous, M=128 channels = two chunks), P as the K-major
//      B operand (N=32 heads, K=32 rows), fp32 in TMEM columns 0..127 (S lives in 128..159).
//   6. Channels on TMEM lanes make the epilogue coalesced: a warp stores 32 consecutive channels
//      of one head per instruction.  The unnormalised O rows and the per-head (max, sum) go to
//      workspace; a combine kernel merges the tiles of each query.
// With a local window (the sliding-window branch: "DeepSeek V4.1-Flash", aiwiki.ai, section
// "Compressed Sparse Attention 2", every layer's own local keys and values; section "KV-cache
// formats and bounded replay", stored in FP8), the tiles after the selected rows' hold the
// window's local E4M3 rows instead (decoded exactly to bf16 through a table), so the combine's
// merge of all tiles is one softmax over the selected rows and the window.
#include <cstring>

#include "sm100.cuh"

namespace csa2 {

constexpr int kSmRows = 32;          // selected rows per CTA
constexpr int kSmHeads = 32;          // heads per CTA
constexpr int kSmThreads = 256;
constexpr int kSmTmemCols = 256;
constexpr int kSmColS = 128;          // S [heads x rows]; O^T takes columns 0..127
constexpr int kSmChunk = kSmRows * 128;  // one 64-channel chunk of the row tile (4 KB)
constexpr int kSmQChunk = kSmHeads * 128;  // one 64-channel chunk of Q (4 KB)

// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr int kSmOffQ = 0;                              // 8 chunks x (32 heads x 128 B) = 32 KB
constexpr int kSmOffK = 8 * kSmQChunk;               // 8 chunks x (32 rows x 128 B) = 32 KB
constexpr int kSmOffPhi = kSmOffK + 8 * kSmChunk;      // 32 heads x 128 B (64 B used)
constexpr int kSmOffPlo = kSmOffPhi + 4096;
constexpr int kSmOffRawC = kSmOffPlo + 4096;              // 32 rows x 256 B codes
constexpr int kSmOffRawS = kSmOffRawC + kSmRows * 256;     // 32 rows x 32 B scales
constexpr int kSmOffLut = kSmOffRawS + kSmRows * 32;       // 256 x u32
constexpr int kSmOffLut8 = kSmOffLut + 1024;              // 256 x u16: E4M3 byte -> bf16
constexpr int kSmOffRaw8 = kSmOffLut8 + 512;              // window tiles: 32 rows x 512 B of E4M3
constexpr int kSmOffMisc = kSmOffRaw8 + kSmRows * 512;
constexpr int kSmSmem = kSmOffMisc + 1024 + 1024;      // + alignment slack
// The M=128 operand read of a Q chunk covers 128 rows of 128 B from the chunk's start, i.e. up
// to 12 KB past its 32 real rows (into the following chunks and the row tile): readable, and it
// only feeds unused accumulator lanes.
static_assert(kSmOffQ + 7 * kSmQChunk + 128 * 128 <= kSmOffMisc, "Q over-read stays in smem");

struct SmMisc {
  uint64_t bar_q, bar_s, bar_o;
  uint32_t tmem_base;
  int slot_ok[kSmRows];
  float m2[kSmHeads];
  float mh[2][kSmHeads], lh[2][kSmHeads];  // per-half row max / sum of the softmax
};




__global__ void __launch_bounds__(kSmThreads, 1) attn_small_kernel(
    const __grid_constant__ CUtensorMap qmap, int H, const uint8_t *__restrict__ codes,
    const uint8_t *__restrict__ sf, const int64_t *__restrict__ cu_ctx,
    const int32_t *__restrict__ idx, int topk, float scale_log2e, int n_tiles,
    float *__restrict__ o_part, float *__restrict__ m_part, float *__restrict__ l_part,
    const uint8_t *__restrict__ swa_kv, int ring, int n_win, int n_sel_tiles) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t *sm = smem_raw + ((1024 - (raw_u32 & 1023)) & 1023);
  SmMisc &ms = *reinterpret_cast<SmMisc *>(sm + kSmOffMisc);
  uint32_t *lut = reinterpret_cast<uint32_t *>(sm + kSmOffLut);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, hg = blockIdx.y, n = blockIdx.z;
  const int h0 = hg * kSmHeads;  // first head of this CTA

  if (tid == 0) {
    mbar_init(&ms.bar_q, 1);
    mbar_init(&ms.bar_s, 1);
    mbar_init(&ms.bar_o, 1);
    fence_barrier_init();
    prefetch_tensormap(&qmap);
  }
  if (warp == 0) {
    tmem_alloc(&ms.tmem_base, kSmTmemCols);
    tmem_relinquish();
  }
  // byte of two E2M1 codes -> bf16x2 of their values (exact)
  lut[tid] = pack_bf16x2(e2m1_to_float(tid & 15), e2m1_to_float(tid >> 4));
  // E4M3 byte -> bf16 (exact: at most 4 significant bits, magnitudes 2^-9..448)
  reinterpret_cast<uint16_t *>(sm + kSmOffLut8)[tid] =
      __bfloat16_as_ushort(__float2bfloat16_rn(e4m3_to_float(tid)));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;
  pdl_wait();
  pdl_trigger();
  const int64_t base = cu_ctx[n];

  // ---- 1. loads
  if (tid == 0) {
    mbar_arrive_expect_tx(&ms.bar_q, 8 * kSmQChunk);
    for (int kc = 0; kc < 8; ++kc)
      tma_load_2d(sm + kSmOffQ + kc * kSmQChunk, &qmap, &ms.bar_q, kc * 64, n * H + h0);
  }
  const bool win = tile >= n_sel_tiles;  // a tile of the local window
  if (!win) {
    // the 32 rows as 32 x 18 16-byte cp.async copies (256 B codes + 32 B scales per row) spread
    // over all threads; an empty slot is a zero row (value 0, never NaN), masked in the softmax.
    // A thread's row numbers are all loaded first, so their latencies overlap.
    constexpr int kCopies = kSmRows * 18, kIters = (kCopies + kSmThreads - 1) / kSmThreads;
    int rr[kIters];
#pragma unroll
    for (int k = 0; k < kIters; ++k) {
      const int i = tid + k * kSmThreads, slot = tile * kSmRows + i / 18;
      rr[k] = (i < kCopies && slot < topk) ? idx[(int64_t)n * topk + slot] : -1;
    }
#pragma unroll
    for (int k = 0; k < kIters; ++k) {
      const int i = tid + k * kSmThreads;
      if (i >= kCopies) break;
      const int j = i / 18, part = i - j * 18;
      const int r = rr[k];
      if (part == 0) ms.slot_ok[j] = r >= 0;
      uint8_t *dst = part < 16 ? sm + kSmOffRawC + j * 256 + part * 16
                               : sm + kSmOffRawS + j * 32 + (part - 16) * 16;
      if (r >= 0) {
        const int64_t row = base + r;
        const uint8_t *src = part < 16 ? codes + row * kCodeBytes + part * 16
                                       : sf + row * kSfBytes + (part - 16) * 16;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
                     "l"(reinterpret_cast<uint64_t>(src))
                     : "memory");
      } else {
        *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
  } else {
    // window tile: slots wi = 32 (tile - n_sel_tiles) + j of the last nw = min(n_win, L) positions
    // t = L - nw + wi; position t's local row is n * ring + t % ring.  32 rows x 32 copies.
    const int64_t L = cu_ctx[n + 1] - base;
    const int64_t nw = L < n_win ? L : n_win;
    const int w0 = (tile - n_sel_tiles) * kSmRows;
#pragma unroll
    for (int k = 0; k < kSmRows * 32 / kSmThreads; ++k) {
      const int i = tid + k * kSmThreads, j = i >> 5, part = i & 31;
      const int wi = w0 + j;
      const bool ok_slot = wi < nw;
      if (part == 0) ms.slot_ok[j] = ok_slot;
      uint8_t *dst = sm + kSmOffRaw8 + j * 512 + part * 16;
      if (ok_slot) {
        const int64_t t = L - nw + wi;
        const uint8_t *src = swa_kv + ((int64_t)n * ring + t % ring) * kD + part * 16;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
                     "l"(reinterpret_cast<uint64_t>(src))
                     : "memory");
      } else {
        *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_all;" ::: "memory");
  bool ok = true;
  __syncthreads();

  // ---- 2./3. dequantise the rows once (chunk kc holds channels 64kc..64kc+63 of all 32 rows)
  //           and S = Q Khat^T: the MMAs over chunks 0..3 run while chunks 4..7 are dequantised
  constexpr uint32_t idesc = idesc_f32acc(1, 1, 128, kSmRows);
  for (int half = 0; half < 2; ++half) {
    for (int v = tid; v < kSmRows * 32; v += kSmThreads) {
      const int j = v >> 5, rest = v & 31, kc = half * 4 + (rest >> 3), u = rest & 7;
      const int c0 = kc * 64 + u * 8;
      uint4 w;
      if (!win) {
        const uint32_t cw = *reinterpret_cast<const uint32_t *>(sm + kSmOffRawC + j * 256 + c0 / 2);
        const float sc = e4m3_to_float(sm[kSmOffRawS + j * 32 + c0 / 16]);
        const uint32_t s2 = pack_bf16x2(sc, sc);
        w.x = bf16x2_mul(lut[cw & 0xFF], s2);
        w.y = bf16x2_mul(lut[(cw >> 8) & 0xFF], s2);
        w.z = bf16x2_mul(lut[(cw >> 16) & 0xFF], s2);
        w.w = bf16x2_mul(lut[cw >> 24], s2);
      } else {
        const uint16_t *lut8 = reinterpret_cast<const uint16_t *>(sm + kSmOffLut8);
        const uint2 b = *reinterpret_cast<const uint2 *>(sm + kSmOffRaw8 + j * 512 + c0);
        w.x = lut8[b.x & 0xFF] | ((uint32_t)lut8[(b.x >> 8) & 0xFF] << 16);
        w.y = lut8[(b.x >> 16) & 0xFF] | ((uint32_t)lut8[b.x >> 24] << 16);
        w.z = lut8[b.y & 0xFF] | ((uint32_t)lut8[(b.y >> 8) & 0xFF] << 16);
        w.w = lut8[(b.y >> 16) & 0xFF] | ((uint32_t)lut8[b.y >> 24] << 16);
      }
      *reinterpret_cast<uint4 *>(sm + kSmOffK + kc * kSmChunk + j * 128 + ((u ^ (j & 7)) << 4)) =
          w;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      if (half == 0) ok = ok && mbar_wait(&ms.bar_q, 0);
      const uint32_t qa = smem_u32(sm + kSmOffQ), ka = smem_u32(sm + kSmOffK);
      for (int kc = half * 4; kc < half * 4 + 4; ++kc)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_f16(tmem + kSmColS, desc_k128_sw128(qa + kc * kSmQChunk + 32 * ks),
                  desc_k128_sw128(ka + kc * kSmChunk + 32 * ks), idesc, (kc | ks) != 0);
      if (half == 1) mma_commit(&ms.bar_s);
    }
  }

  // ---- 4. softmax: warps 0 and 4 read TMEM lanes 0..31 (= heads); warp 0 takes the columns
  //         (rows) 0..15 of S, warp 4 the columns 16..31
  if ((warp & 3) == 0) {
    ok = __all_sync(0xffffffffu, mbar_wait(&ms.bar_s, 0)) && ok;
    tc_fence_after();
    const int h = lane;
    const int half = warp >> 2, j0 = half * 16;
    float s[16];
    {
      uint32_t r[16];
      tmem_ld16(tmem + kSmColS + j0, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) s[i] = __uint_as_float(r[i]) * scale_log2e;
    }
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (ms.slot_ok[j0 + j]) m = fmaxf(m, s[j]);
    ms.mh[half][h] = m;
    asm volatile("bar.sync 1, 64;" ::: "memory");  // the two softmax warps
    m = fmaxf(ms.mh[0][h], ms.mh[1][h]);
    float l = 0.0f;
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      const float p0 = ms.slot_ok[j0 + j] ? exp2f(s[j] - m) : 0.0f;
      const float p1 = ms.slot_ok[j0 + j + 1] ? exp2f(s[j + 1] - m) : 0.0f;
      l += p0 + p1;
      const __nv_bfloat16 b0 = __float2bfloat16_rn(p0), b1 = __float2bfloat16_rn(p1);
      hi[j / 2] = (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
      lo[j / 2] = pack_bf16x2(p0 - __bfloat162float(b0), p1 - __bfloat162float(b1));
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int off = h * 128 + (((2 * half + u) ^ (h & 7)) << 4);
      *reinterpret_cast<uint4 *>(sm + kSmOffPhi + off) =
          make_uint4(hi[4 * u], hi[4 * u + 1], hi[4 * u + 2], hi[4 * u + 3]);
      *reinterpret_cast<uint4 *>(sm + kSmOffPlo + off) =
          make_uint4(lo[4 * u], lo[4 * u + 1], lo[4 * u + 2], lo[4 * u + 3]);
    }
    if (half == 0) ms.m2[h] = m;
    ms.lh[half][h] = l;
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- 5. O^T = Vhat^T P^T: M=128 channels (two chunks), N=32 heads, K=16 rows per MMA
  if (tid == 0) {
    constexpr uint32_t idesc_pv = idesc_f32acc(1, 1, 128, kSmHeads) | (1u << 15);  // A MN-major
    const uint32_t ka = smem_u32(sm + kSmOffK);
    const uint32_t ph = smem_u32(sm + kSmOffPhi), pl = smem_u32(sm + kSmOffPlo);
    for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
      for (int ks = 0; ks < kSmRows / 16; ++ks) {
        const uint64_t ad =
            desc_mn_sw128_atoms(ka + (2 * mb) * kSmChunk + ks * 16 * 128, kSmChunk);
        mma_f16(tmem + mb * kSmHeads, ad, desc_k128_sw128(ph + 32 * ks), idesc_pv, ks != 0);
        mma_f16(tmem + mb * kSmHeads, ad, desc_k128_sw128(pl + 32 * ks), idesc_pv, 1);
      }
    }
    mma_commit(&ms.bar_o);
  }

  // ---- 6. epilogue: warp w reads lanes 32(w%4).. (channels) of M blocks 2(w/4), 2(w/4)+1;
  //         column 32*mb + h of O^T is channel 128*mb + lane
  ok = __all_sync(0xffffffffu, mbar_wait(&ms.bar_o, 0)) && ok;
  tc_fence_after();
  {
    const int q4 = warp & 3, mb0 = (warp >> 2) * 2;
    const uint32_t la = tmem + ((uint32_t)(q4 * 32) << 16);
    float *obase = o_part + (((int64_t)n * n_tiles + tile) * H + h0) * kD;
    const int hn = min(kSmHeads, H - h0);  // real heads of this group
#pragma unroll 1
    for (int mb = mb0; mb < mb0 + 2; ++mb) {
      uint32_t r0[16], r1[16];
      tmem_ld16(la + mb * kSmHeads, r0);
      tmem_ld16(la + mb * kSmHeads + 16, r1);
      tmem_ld_wait();
      float *oc = obase + mb * 128 + q4 * 32 + lane;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (i < hn) oc[(int64_t)i * kD] = __uint_as_float(r0[i]);
        if (i + 16 < hn) oc[(int64_t)(i + 16) * kD] = __uint_as_float(r1[i]);
      }
    }
    if (tid < hn) {
      const int64_t pr = ((int64_t)n * n_tiles + tile) * H + h0 + tid;
      m_part[pr] = ok ? ms.m2[tid] : -INFINITY;
      l_part[pr] = ok ? ms.lh[0][tid] + ms.lh[1][tid] : 0.0f;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kSmTmemCols);
}

// Merge the tiles of each (query, head): out = sum_t O_t 2^(m_t - M) / sum_t l_t 2^(m_t - M);
// lse = (M + log2 L) * ln 2.  m is in the log2 domain (logits * scale * log2 e).
// Grid (kD / 128, H, nq), 128 threads: thread = one channel.  The channel's partials are read 64
// tiles at a time with unconditional loads (indices clamped, so all 64 are in flight at once;
// the first batch before the weights are known), then summed in tile order.
constexpr int kSmCombBatch = 64;
__global__ void __launch_bounds__(128) attn_small_combine_kernel(
    int H, int n_tiles, const float *__restrict__ o_part, const float *__restrict__ m_part,
    const float *__restrict__ l_part, uint16_t *__restrict__ out, float *__restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  __shared__ float wgt[256];
  __shared__ float sM, sL;
  const int h = blockIdx.y, n = blockIdx.z, tid = threadIdx.x, lane = tid & 31;
  const int c = blockIdx.x * 128 + tid;
  const int64_t tstride = (int64_t)H * kD;  // floats between consecutive tiles
  const float *op = o_part + ((int64_t)n * n_tiles * H + h) * kD + c;
  float acc = 0.0f;
  for (int t0 = 0; t0 < n_tiles; t0 += kSmCombBatch) {
    float o[kSmCombBatch];
#pragma unroll
    for (int u = 0; u < kSmCombBatch; ++u) {
      const int t = min(t0 + u, n_tiles - 1);
      o[u] = op[t * tstride];
    }
    if (t0 == 0) {
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
    }
#pragma unroll
    for (int u = 0; u < kSmCombBatch; ++u)
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
// Few tiles in all: every query's small tiles (and head groups) fit in about one wave of CTAs
// (two per SM on a B300's 148 SMs), which the 128-row tiles of attn_mma.cu would leave idle.
bool attn_small_preferred(int nq, int H, int topk, int n_win) {
  const int64_t tiles = (topk + kSmRows - 1) / kSmRows + (n_win + kSmRows - 1) / kSmRows;
  const int64_t ctas = (int64_t)nq * tiles * ((H + kSmHeads - 1) / kSmHeads);
  return H <= 64 && tiles <= 256 && ctas <= 2 * 148 && encode_fn() != nullptr;
}

size_t attn_small_workspace_bytes(int nq, int H, int topk, int n_win) {
  const size_t tiles =
      (size_t)(topk + kSmRows - 1) / kSmRows + (size_t)(n_win + kSmRows - 1) / kSmRows;
  const size_t rows = (size_t)nq * tiles * H;
  return rows * kD * sizeof(float) + 2 * rows * sizeof(float) + 1024;
}

static bool make_q_map_small(CUtensorMap *m, const void *q, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rows <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, kSmHeads};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(q), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

cudaError_t launch_attn_small(const void *q_bf16, int nq, int H, const uint8_t *codes,
                              const uint8_t *sf, const int64_t *cu_ctx, const int32_t *idx,
                              int topk, float scale, void *out_bf16, float *lse, void *workspace,
                              cudaStream_t st, const uint8_t *swa_kv, int ring, int n_win) {
  if (nq == 0) return cudaSuccess;
  const int n_sel = (topk + kSmRows - 1) / kSmRows;
  const int n_tiles = n_sel + (n_win + kSmRows - 1) / kSmRows;
  const size_t rows = (size_t)nq * n_tiles * H;
  float *o_part = static_cast<float *>(workspace);
  float *m_part = o_part + rows * kD;
  float *l_part = m_part + rows;
  CUtensorMap qm;
  memset(&qm, 0, sizeof(qm));
  if (!make_q_map_small(&qm, q_bf16, (int64_t)nq * H)) return cudaErrorInvalidValue;
  const float scale_log2e = scale * 1.4426950408889634f;
  const int n_hg = (H + kSmHeads - 1) / kSmHeads;
  cudaError_t e = set_smem_once(attn_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmSmem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attn_small_kernel, dim3(n_tiles, n_hg, nq), dim3(kSmThreads), (size_t)kSmSmem,
                 st, qm, H, codes, sf, cu_ctx, idx, topk, scale_log2e, n_tiles, o_part, m_part,
                 l_part, swa_kv, ring, n_win, n_sel);
  note_launches(1);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attn_small_combine_kernel, dim3(kD / 128, H, nq), dim3(128), 0, st, H, n_tiles,
                 (const float *)o_part, (const float *)m_part, (const float *)l_part,
                 static_cast<uint16_t *>(out_bf16), lse);
  note_launches(1);
  return e;
}

}  // namespace csa2

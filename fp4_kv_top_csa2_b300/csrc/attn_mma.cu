// attn_mma.cu -- sparse decode attention over gathered FP4 rows on the tensor cores (tcgen05).
//
// For sequence n, head h: softmax_j(scale * q_h . khat_j) over the selected rows j, applied to
// the same rows (K = V = the dequantised latent row; the model card's Introduction, CSA2
// paragraph: the sparse attention reads the FP4 main-KV rows that a shared Top-K index set names).
//
// One CTA = one query (sequence) x one tile of 128 selected rows, all heads (H <= 64).  Steps:
//   1. Q [64 heads x 512] bf16 arrives by TMA as eight 128B-swizzled chunks of 64 channels; the
//      tile's rows are loaded from L2 into registers (16-byte code loads and 2-byte scale loads,
//      a thread per 32-channel segment of two rows) and dequantised exactly (E2M1 x E4M3 has <= 6
//      significant bits) to bf16 into eight chunks [128 rows x 64 channels]: the E2M1 pair by
//      cvt to fp16 and a move of the bit fields (the value times 2^-112), then one bf16 multiply
//      by the block scale times 2^112.
//   2. S = Q Khat^T: kind::f16 (bf16), M=128 (64 heads, padded) x N=128 rows x K=512, 32 MMAs,
//      issued chunk pair by chunk pair as the rows are dequantised; TMEM columns 256..383.
//   3. Softmax: a thread holds one head and 64 of the 128 rows (two threads per head, the maximum
//      and sum exchanged through shared memory); the numerators p = 2^(s - m) are split into bf16
//      hi + lo parts (P ~ hi + lo to 2^-16), written as the A operand [P_hi; P_lo]: M=128 rows =
//      the 64 heads' hi parts, then their lo parts, K = the tile's 128 rows.
//   4. O = [P_hi; P_lo] Vhat: M=128 x N=256 channels x K=16 rows per MMA, the same dequantised
//      chunks read as the MN-major B operand (channels contiguous), two channel halves into TMEM
//      columns 0..255 and 256..511 (the second half reuses S's columns once it is read): 16 MMAs
//      for the whole tile.  The M rows put each lane quarter's 16 heads' hi rows, then their lo
//      rows, so a head's two products sit 16 TMEM lanes apart in one warp.
//   5. One shuffle adds a head's hi and lo products in registers, and the tile's unnormalised
//      O [H x 512] fp32 goes to workspace (each pair of lanes fills whole 128-byte lines), with
//      the per-head (max, sum); a combine kernel merges the tiles with the softmax weights and
//      normalises.
// With a local window (the sliding-window branch: "DeepSeek V4.1-Flash", aiwiki.ai, section
// "Compressed Sparse Attention 2", every layer's own local keys and values; section "KV-cache
// formats and bounded replay", stored in FP8), the tiles after the selected rows' hold the
// window's local E4M3 rows instead (decoded exactly to bf16), so the combine's merge of all tiles
// is one softmax over the selected rows and the window.
#include <cstring>

#include "sm100.cuh"

namespace csa2 {

constexpr int kAttRows = 128;        // selected rows per CTA (MMA N of S, K of O)
constexpr int kAttWorkers = 256;     // warps 0..7
constexpr int kAttMmaWarp = 8;       // warp 8: TMEM allocation, TMA of Q, MMA issue
constexpr int kAttThreads = kAttWorkers + 32;
constexpr int kAttQChunk = 64 * 128;           // one 64-channel chunk of Q: 64 heads x 128 B
constexpr int kAttKChunk = kAttRows * 128;     // one 64-channel chunk of the rows
constexpr int kAttPChunk = 128 * 128;          // one 64-row chunk of [P_hi; P_lo]
constexpr int kAttOffQ = 0;                                // 64 KB
constexpr int kAttOffK = 8 * kAttQChunk;                   // 128 KB
constexpr int kAttOffP = kAttOffK + 8 * kAttKChunk;        // 32 KB
constexpr int kAttOffMisc = kAttOffP + 2 * kAttPChunk;
constexpr int kAttSmem = kAttOffMisc + 2048 + 1024;        // + alignment slack
// The M=128 operand read of a Q chunk covers 128 rows of 128 B from the chunk's start, i.e. up
// to 8 KB past its 64 real rows (into the next chunk, or the row tile after the last one):
// readable, and it only feeds accumulator lanes 64..127 of S, which are never read.
static_assert(kAttOffQ + 7 * kAttQChunk + 128 * 128 <= kAttOffMisc, "Q over-read stays in smem");
static_assert(kAttSmem <= 232448, "shared memory per CTA");

struct AttMisc {
  uint64_t bar_q, bar_dq[4], bar_s, bar_p, bar_o;
  uint32_t tmem_base;
  int slot_ok[kAttRows];
  float mx[2][64], sm[2][64];  // per column half: head maximum, head sum
};
static_assert(sizeof(AttMisc) <= 2048, "misc block");

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

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Two E4M3 bytes (low byte = lower channel) -> bf16x2 of their values (exact: at most 4
// significant bits, magnitudes 2^-9..448).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)two));
  const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
  return pack_bf16x2(f.x, f.y);
}

// E2M1 code byte (low nibble = lower channel) -> bf16x2 of the two values times 2^-112, exact:
// cvt gives the fp16 pair; its sign, exponent field and top 7 mantissa bits moved into bf16
// positions (mantissa >> 3) read as the same value scaled by 2^(15 - 127), the two exponent
// biases.  An E2M1 value uses one mantissa bit, so the three bits shifted out (and the three
// that cross from the upper half into the lower one) are zero; zero stays zero.  The
// 2^112 goes back in with the block scale (s * 2^112 <= 448 * 2^112 fits bf16).
__device__ __forceinline__ uint32_t e2m1x2_bf16x2_m112(uint32_t byte) {
  uint32_t h;
  asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(h) : "r"(byte));
  return ((h & 0x7FFF7FFFu) >> 3) | (h & 0x80008000u);
}

__global__ void __launch_bounds__(kAttThreads, 1) attn_mma_kernel(
    const __grid_constant__ CUtensorMap qmap, int H, const uint8_t *__restrict__ codes,
    const uint8_t *__restrict__ sf, const int64_t *__restrict__ cu_ctx,
    const int32_t *__restrict__ idx, int topk, float scale_log2e, int n_tiles,
    float *__restrict__ o_part, float *__restrict__ m_part, float *__restrict__ l_part,
    const uint8_t *__restrict__ swa_kv, int ring, int n_win, int n_sel_tiles) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  AttMisc &ms = *reinterpret_cast<AttMisc *>(sm + kAttOffMisc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, n = blockIdx.y;

  if (tid == 0) {
    mbar_init(&ms.bar_q, 1);
    for (int c = 0; c < 4; ++c) mbar_init(&ms.bar_dq[c], kAttWorkers);
    mbar_init(&ms.bar_s, 1);
    mbar_init(&ms.bar_p, kAttWorkers);
    mbar_init(&ms.bar_o, 1);
    fence_barrier_init();
    prefetch_tensormap(&qmap);
  }
  if (warp == kAttMmaWarp) {
    tmem_alloc(&ms.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;  // O half 0: cols 0..255; S: 256..383; O half 1: 256..511
  pdl_wait();
  pdl_trigger();
  const int64_t base = cu_ctx[n];
  bool ok = true;

  if (warp == kAttMmaWarp) {
    // ------------------------------------------------------------------ TMA of Q, MMA issue
    if (lane == 0) {
      mbar_arrive_expect_tx(&ms.bar_q, 8 * kAttQChunk);
      for (int kc = 0; kc < 8; ++kc)
        tma_load_2d(sm + kAttOffQ + kc * kAttQChunk, &qmap, &ms.bar_q, kc * 64, n * H);
      constexpr uint32_t idesc_s = idesc_f32acc(1, 1, 128, kAttRows);             // bf16
      constexpr uint32_t idesc_o = idesc_f32acc(1, 1, 128, 256) | (1u << 16);     // B MN-major
      const uint32_t qa = smem_u32(sm + kAttOffQ), ka = smem_u32(sm + kAttOffK);
      const uint32_t pa = smem_u32(sm + kAttOffP);
      ok = mbar_wait(&ms.bar_q, 0) && ok;
      for (int cp = 0; cp < 4; ++cp) {
        ok = mbar_wait(&ms.bar_dq[cp], 0) && ok;
        tc_fence_after();
#pragma unroll
        for (int kc = 2 * cp; kc < 2 * cp + 2; ++kc)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_f16(tmem + 256, desc_k128_sw128(qa + kc * kAttQChunk + 32 * ks),
                    desc_k128_sw128(ka + kc * kAttKChunk + 32 * ks), idesc_s, (kc | ks) != 0);
      }
      mma_commit(&ms.bar_s);
      ok = mbar_wait(&ms.bar_p, 0) && ok;  // [P_hi; P_lo] written, S read
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < 2; ++half)
#pragma unroll
        for (int ks = 0; ks < kAttRows / 16; ++ks)
          mma_f16(tmem + 256 * half,
                  desc_k128_sw128(pa + (ks >> 2) * kAttPChunk + 32 * (ks & 3)),
                  desc_mn_sw128_atoms(ka + 4 * half * kAttKChunk + ks * 16 * 128, kAttKChunk),
                  idesc_o, ks != 0);
      mma_commit(&ms.bar_o);
    }
  } else {
    // ------------------------------------------------------------------ workers (warps 0..7)
    // a thread owns the 32-channel segment `seg` of rows jr and jr + 64 in every chunk pair
    const int seg = tid & 3, jr = tid >> 2;
    const bool win = tile >= n_sel_tiles;  // a tile of the local window
    uint4 rc[16];                          // FP4: codes of (pair cp, row half) at 2 cp + half;
    uint32_t rs[8];                        // E4M3 window rows: 32 bytes of (cp, half) at 4 cp ..
    if (!win) {
      int r[2];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int slot = tile * kAttRows + jr + 64 * hf;
        r[hf] = slot < topk ? __ldg(idx + (int64_t)n * topk + slot) : -1;
        if (seg == 0) ms.slot_ok[jr + 64 * hf] = r[hf] >= 0;
      }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int64_t row = base + (r[hf] >= 0 ? r[hf] : 0);
#pragma unroll
        for (int cp = 0; cp < 4; ++cp) {
          rc[2 * cp + hf] = r[hf] >= 0 ? __ldg(reinterpret_cast<const uint4 *>(
                                             codes + row * kCodeBytes + cp * 64 + seg * 16))
                                       : make_uint4(0, 0, 0, 0);
          rs[2 * cp + hf] = r[hf] >= 0 ? (uint32_t)__ldg(reinterpret_cast<const uint16_t *>(
                                             sf + row * kSfBytes + cp * 8 + seg * 2))
                                       : 0u;
        }
      }
    } else {
      // window slot wi of the last nw = min(n_win, L) positions t = L - nw + wi; position t's
      // local row is n * ring + t % ring
      const int64_t L = cu_ctx[n + 1] - base;
      const int64_t nw = L < n_win ? L : n_win;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int64_t wi = (int64_t)(tile - n_sel_tiles) * kAttRows + jr + 64 * hf;
        const bool valid = wi < nw;
        if (seg == 0) ms.slot_ok[jr + 64 * hf] = valid;
        const int64_t lrow = (int64_t)n * ring + (valid ? (L - nw + wi) % ring : 0);
#pragma unroll
        for (int cp = 0; cp < 4; ++cp)
#pragma unroll
          for (int k = 0; k < 2; ++k)
            rc[4 * cp + 2 * hf + k] =
                valid ? __ldg(reinterpret_cast<const uint4 *>(swa_kv + lrow * kD + cp * 128 +
                                                              seg * 32 + 16 * k))
                      : make_uint4(0, 0, 0, 0);
      }
    }
    // ---- dequantise into the eight K chunks, a chunk pair at a time (the MMAs follow)
#pragma unroll
    for (int cp = 0; cp < 4; ++cp) {
      const int kc = 2 * cp + (seg >> 1), u0 = (seg & 1) * 4;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int j = jr + 64 * hf;
        uint8_t *row = sm + kAttOffK + kc * kAttKChunk + j * 128;
        uint4 w[4];
        if (!win) {
          const uint4 c = rc[2 * cp + hf];
          const uint32_t r = rs[2 * cp + hf];
          const float fa = e4m3_to_float(r & 0xFF) * 0x1p112f;
          const float fb = e4m3_to_float(r >> 8) * 0x1p112f;
          const uint32_t sa = pack_bf16x2(fa, fa), sb = pack_bf16x2(fb, fb);
          const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t sc = u < 2 ? sa : sb;
            w[u].x = bf16x2_mul(e2m1x2_bf16x2_m112(cw[u] & 0xFF), sc);
            w[u].y = bf16x2_mul(e2m1x2_bf16x2_m112((cw[u] >> 8) & 0xFF), sc);
            w[u].z = bf16x2_mul(e2m1x2_bf16x2_m112((cw[u] >> 16) & 0xFF), sc);
            w[u].w = bf16x2_mul(e2m1x2_bf16x2_m112(cw[u] >> 24), sc);
          }
        } else {
          const uint4 a = rc[4 * cp + 2 * hf], b = rc[4 * cp + 2 * hf + 1];
          const uint32_t by[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            w[u].x = e4m3x2_to_bf16x2(by[2 * u] & 0xFFFF);
            w[u].y = e4m3x2_to_bf16x2(by[2 * u] >> 16);
            w[u].z = e4m3x2_to_bf16x2(by[2 * u + 1] & 0xFFFF);
            w[u].w = e4m3x2_to_bf16x2(by[2 * u + 1] >> 16);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4 *>(row + (((u0 + u) ^ (j & 7)) << 4)) = w[u];
      }
      fence_async_smem();
      mbar_arrive(&ms.bar_dq[cp]);
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");  // slot_ok visible to every worker

    // ---- softmax: warps 0,1 (columns 0..63) and 4,5 (columns 64..127) hold heads 0..63
    const int quarter = warp & 3, c2 = warp >> 2;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    if (quarter < 2) {
      const int h = quarter * 32 + lane;
      ok = __all_sync(0xffffffffu, mbar_wait(&ms.bar_s, 0)) && ok;
      tc_fence_after();
      float x[64];
      {
        uint32_t r0[16], r1[16], r2[16], r3[16];
        const uint32_t ta = tmem + 256 + 64 * c2 + lane_off;
        tmem_ld16(ta, r0);
        tmem_ld16(ta + 16, r1);
        tmem_ld16(ta + 32, r2);
        tmem_ld16(ta + 48, r3);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          x[i] = __uint_as_float(r0[i]);
          x[16 + i] = __uint_as_float(r1[i]);
          x[32 + i] = __uint_as_float(r2[i]);
          x[48 + i] = __uint_as_float(r3[i]);
        }
      }
      float m = -INFINITY;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        x[i] = ms.slot_ok[64 * c2 + i] ? x[i] * scale_log2e : -INFINITY;
        m = fmaxf(m, x[i]);
      }
      ms.mx[c2][h] = m;
      asm volatile("bar.sync 2, 128;" ::: "memory");  // the four softmax warps
      m = fmaxf(ms.mx[0][h], ms.mx[1][h]);
      const float mm = m == -INFINITY ? 0.0f : m;  // no valid slot: every numerator 0
      float l = 0.0f;
      // M rows: lane quarter h / 16 holds heads 16 (h / 16) .. + 15, their hi rows then their lo
      // rows (row & 7 == h & 7 for both, so the swizzle below keeps h & 7)
      const int mr_hi = 32 * (h >> 4) + (h & 15);
      uint8_t *phi = sm + kAttOffP + c2 * kAttPChunk + mr_hi * 128;
      uint8_t *plo = phi + 16 * 128;  // row mr_hi + 16
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
          const float p0 = exp2f(x[8 * u + k] - mm), p1 = exp2f(x[8 * u + k + 1] - mm);
          l += p0 + p1;
          const __nv_bfloat16 b0 = __float2bfloat16_rn(p0), b1 = __float2bfloat16_rn(p1);
          hi[k / 2] = (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
          lo[k / 2] = pack_bf16x2(p0 - __bfloat162float(b0), p1 - __bfloat162float(b1));
        }
        *reinterpret_cast<uint4 *>(phi + ((u ^ (h & 7)) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(plo + ((u ^ (h & 7)) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      ms.sm[c2][h] = l;
      asm volatile("bar.sync 2, 128;" ::: "memory");
      if (c2 == 0 && h < H) {
        const int64_t pr = ((int64_t)n * n_tiles + tile) * H + h;
        m_part[pr] = ok ? m : -INFINITY;
        l_part[pr] = ok ? ms.sm[0][h] + ms.sm[1][h] : 0.0f;
      }
    }
    fence_async_smem();
    tc_fence_before();
    mbar_arrive(&ms.bar_p);

    // ---- epilogue: warp = (lane quarter q: heads 16 q .. + 15, hi products in lanes 0..15 and
    // lo in 16..31; channel half c2).  One shuffle adds a head's hi and lo values: the hi lane
    // keeps columns 0..15 of each 32-column block, the lo lane 16..31, and each stores its 64
    // bytes of the head's partial row (two lanes fill one 128-byte line).
    ok = __all_sync(0xffffffffu, mbar_wait(&ms.bar_o, 0)) && ok;
    tc_fence_after();
    {
      const bool lo = lane >= 16;
      const int ho = 16 * quarter + (lane & 15);
      const uint32_t ta = tmem + 256 * c2 + lane_off;
      float *orow = o_part + (((int64_t)n * n_tiles + tile) * H + ho) * kD + 256 * c2 + 16 * lo;
#pragma unroll 1
      for (int c0 = 0; c0 < 256; c0 += 32) {
        uint32_t v0[16], v1[16];
        tmem_ld16(ta + c0, v0);
        tmem_ld16(ta + c0 + 16, v1);
        tmem_ld_wait();
        float o[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float send = __uint_as_float(lo ? v0[k] : v1[k]);
          const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
          o[k] = __uint_as_float(lo ? v1[k] : v0[k]) + recv;
        }
        if (ho < H) {
          float4 *d = reinterpret_cast<float4 *>(orow + c0);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            d[k] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kAttMmaWarp) tmem_dealloc(tmem, 512);
}

// Merge the tiles of each (query, head): out = sum_t O_t 2^(m_t - M) / sum_t l_t 2^(m_t - M),
// M = max_t m_t over tiles with l_t > 0, m in the log2 domain (logits * scale * log2 e);
// lse = (M + log2 L) ln 2 with L the denominator, -inf with no valid slot.  One CTA per (head, query), a thread per four channels: the tiles' rows are read
// as float4 (each tile's row 2 KB contiguous), the first batch in flight while warp 0 forms the
// weights (24 tiles: one round trip for up to 3,072 rows).
constexpr int kCombBatch = 24;

__global__ void __launch_bounds__(128) attn_mma_combine_kernel(
    int H, int n_tiles, const float *__restrict__ o_part, const float *__restrict__ m_part,
    const float *__restrict__ l_part, uint16_t *__restrict__ out, float *__restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  __shared__ float wgt[256];
  __shared__ float sM, sL;
  const int h = blockIdx.x, n = blockIdx.y, tid = threadIdx.x, lane = tid & 31;
  const int64_t ts4 = (int64_t)H * kD / 4;  // float4s between consecutive tiles
  const float4 *op =
      reinterpret_cast<const float4 *>(o_part + ((int64_t)n * n_tiles * H + h) * kD) + tid;
  float4 o[kCombBatch];
#pragma unroll
  for (int u = 0; u < kCombBatch; ++u)
    if (u < n_tiles) o[u] = op[u * ts4];
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
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int t0 = 0; t0 < n_tiles; t0 += kCombBatch) {
    if (t0 > 0) {
#pragma unroll
      for (int u = 0; u < kCombBatch; ++u)
        if (t0 + u < n_tiles) o[u] = op[(t0 + u) * ts4];
    }
#pragma unroll
    for (int u = 0; u < kCombBatch; ++u) {
      if (t0 + u < n_tiles) {
        const float wv = wgt[t0 + u];
        acc.x = fmaf(o[u].x, wv, acc.x);
        acc.y = fmaf(o[u].y, wv, acc.y);
        acc.z = fmaf(o[u].z, wv, acc.z);
        acc.w = fmaf(o[u].w, wv, acc.w);
      }
    }
  }
  const float L = sL, M = sM;
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  uint2 pk;
  pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2 *>(out + ((int64_t)n * H + h) * kD)[tid] = pk;
  if (tid == 0 && lse)
    lse[(int64_t)n * H + h] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

bool attn_mma_supported(int H, int topk, int n_win) {
  return H <= 64 && (topk + kAttRows - 1) / kAttRows + (n_win + kAttRows - 1) / kAttRows <= 256 &&
         encode_fn() != nullptr;
}

size_t attn_mma_workspace_bytes(int nq, int H, int topk, int n_win) {
  if (attn_small_preferred(nq, H, topk, n_win))
    return attn_small_workspace_bytes(nq, H, topk, n_win);
  const size_t tiles =
      (size_t)(topk + kAttRows - 1) / kAttRows + (size_t)(n_win + kAttRows - 1) / kAttRows;
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

cudaError_t launch_attn_mma(const void *q_bf16, int nq, int H, const uint8_t *codes,
                            const uint8_t *sf, const int64_t *cu_ctx, const int32_t *idx,
                            int topk, float scale, void *out_bf16, float *lse, void *workspace,
                            cudaStream_t st, const uint8_t *swa_kv, int ring, int n_win) {
  if (nq == 0) return cudaSuccess;
  if (attn_small_preferred(nq, H, topk, n_win))
    return launch_attn_small(q_bf16, nq, H, codes, sf, cu_ctx, idx, topk, scale, out_bf16, lse,
                             workspace, st, swa_kv, ring, n_win);
  const int n_sel = (topk + kAttRows - 1) / kAttRows;
  const int n_tiles = n_sel + (n_win + kAttRows - 1) / kAttRows;
  const size_t rows = (size_t)nq * n_tiles * H;
  float *o_part = static_cast<float *>(workspace);
  float *m_part = o_part + rows * kD;
  float *l_part = m_part + rows;
  const float scale_log2e = scale * 1.4426950408889634f;
  cudaError_t e;
  CUtensorMap qm;
  memset(&qm, 0, sizeof(qm));
  if (!make_q_map(&qm, q_bf16, (int64_t)nq * H)) return cudaErrorInvalidValue;
  e = set_smem_once(attn_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttSmem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attn_mma_kernel, dim3(n_tiles, nq), dim3(kAttThreads), (size_t)kAttSmem, st, qm,
                 H, codes, sf, cu_ctx, idx, topk, scale_log2e, n_tiles, o_part, m_part, l_part,
                 swa_kv, ring, n_win, n_sel);
  note_launches(1);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attn_mma_combine_kernel, dim3(H, nq), dim3(kD / 4), 0, st, H, n_tiles,
                 (const float *)o_part, (const float *)m_part, (const float *)l_part,
                 static_cast<uint16_t *>(out_bf16), lse);
  note_launches(1);
  return e;
}

}  // namespace csa2

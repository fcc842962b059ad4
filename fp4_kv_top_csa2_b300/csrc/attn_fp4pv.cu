// attn_fp4pv.cu -- the full-FP4 PV variant of prefill attention: the probability-value product
// as a block-scaled FP4 contraction too (the workload names both products of prefill attention
// as block-scaled FP4).  Per query token and head, with the token's selected slots j in tiles of
// 128 and blocks of 16 consecutive slots:
//   s_j = scale <qhat_h, khat_j>  (as the prefill kernel: FP4 query and rows, exact fp16 values)
//   m_h = max_j s_j,  p_j = 2^((s_j - m_h) log2 e)
//   Pt_j  = FP4(p_j; 16-slot block of head h):  sc = E4M3(max p / 6),  Pt = E2M1(p / sc) * sc
//   Vt_jc = FP4(khat_jc; channel c, 16-slot block): sc = E4M3(max |khat| / 6), same rule
//   out_h = sum_j Pt_j Vt_j / sum_j Pt_j,   lse_h = m_h + ln sum_j Pt_j
// The maximum must be known before any numerator is quantised, so the kernel makes two passes
// over the token's tiles: the first computes S^T only and keeps each head's maximum; the second
// recomputes S^T, quantises P (a 16-slot block is 16 lanes: block maxima by a half-warp
// reduce-scatter, one scale and its reciprocal rounded per lane) and re-quantises the tile's rows
// in place in shared memory (a thread per 8 channels of a 16-row block), in two steps of two
// 128-channel blocks, so the MMAs O^T += Vt^T Pt^T of the first two blocks run while the last two
// are re-quantised.  Both roundings take the quotient x / sc to within an ulp (a product with the
// reciprocal, corrected once by the exact remainder) and the hardware E2M1 conversion (nearest,
// ties to even, saturating); the rows' quotients are formed in packed fp16.  A row value has at
// most 6 significant bits and sc at most 4, so x / sc equals a decision point exactly or lies
// more than 2^-7 (relative) from one: Vt is exactly the rounding of the quotient.  A numerator
// p has 24 bits: Pt can differ from that rounding only where p / sc lies within an ulp of a
// decision point.  Pt and Vt are exact in fp16 (at most 6
// significant bits), so O^T is one kind::f16 MMA per (channel block, 16 rows): the products a
// block-scaled FP4 MMA would form, accumulated in fp32.
//
// Structure and roles as attn_prefill_kernel (warps 0..7 load, dequantise, softmax, epilogue;
// warp 8 allocates TMEM and issues the MMAs); O^T takes TMEM columns 0..255, S^T 256..319.
#include "sm100.cuh"

namespace csa2 {

// The E4M3 scale of a block whose largest magnitude is amax (the main-KV rule: amax / 6, fp32
// division, round to nearest even, saturating).
__device__ __forceinline__ float fp4_scale(float amax) {
  return e4m3_to_float(float_to_e4m3_sat(__fdiv_rn(amax, 6.0f)));
}

// The quotient x / sc to within an ulp, without a division: q0 = x * rcp, corrected once by the
// remainder (exact in an fma), written so that x = -0 gives -0.  rcp = 0 for sc = 0 gives 0.
__device__ __forceinline__ float fp4_quot(float x, float sc, float rcp) {
  const float q0 = x * rcp;
  return fmaf(-fmaf(q0, sc, -x), rcp, q0);
}

// Two quotients -> their E2M1 values (round to nearest even, saturating at 6, sign kept) as an
// fp16 pair, lo in the low half, by the conversion instructions.
__device__ __forceinline__ uint32_t e2m1_round_f16x2(float lo, float hi) {
  uint32_t r;
  asm("{\n .reg .b8 b;\n cvt.rn.satfinite.e2m1x2.f32 b, %2, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}\n"
      : "=r"(r)
      : "f"(lo), "f"(hi));
  return r;
}

// The same for a pair of fp16 row values (at most 6 significant bits) under fp16 scales and
// reciprocals: the quotient to within an fp16 ulp, exact at a decision point, then E2M1 and back
// to fp16 by the conversion instructions.  Every such x / sc lies on a decision point or more than
// 2^-7 (relative) from one, so the fp16 quotient decides as the exact one does.
__device__ __forceinline__ uint32_t fp4_level_f16x2(__half2 x, __half2 sc, __half2 rcp) {
  const __half2 q0 = __hmul2(x, rcp);
  const __half2 q = __hfma2(__hneg2(__hfma2(q0, sc, __hneg2(x))), rcp, q0);
  uint32_t r;
  asm("{\n .reg .b8 b;\n cvt.rn.satfinite.e2m1x2.f16x2 b, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}\n"
      : "=r"(r)
      : "r"(*reinterpret_cast<const uint32_t *>(&q)));
  return r;
}

// The main-KV scale rule E4M3(fp32(amax / 6)) for a pair of fp16 block maxima of row values (at
// most 6 significant bits), as an fp16 pair (exact: E4M3 values are fp16 normals).  The fp16
// quotient amax * fp16(1/6), corrected once by the remainder, is exact where amax / 6 lies on an
// E4M3 rounding boundary (a few maxima do, in the subnormal range) and within an ulp elsewhere,
// far from every boundary; the hardware E4M3 conversion then rounds it as the fp32 quotient
// rounds (checked for every possible maximum).
__device__ __forceinline__ __half2 fp4_scale_f16x2(__half2 amax) {
  const __half2 six = __float2half2_rn(6.0f), r6 = __float2half2_rn(1.0f / 6.0f);
  const __half2 q0 = __hmul2(amax, r6);
  const __half2 q = __hfma2(__hneg2(__hfma2(q0, six, __hneg2(amax))), r6, q0);
  uint16_t e;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;"
      : "=h"(e)
      : "r"(*reinterpret_cast<const uint32_t *>(&q)));
  const uint32_t h = e4m3x2_to_f16x2(e);
  return *reinterpret_cast<const __half2 *>(&h);
}

__global__ void __launch_bounds__(kPfThreads, 1) attn_fp4pv_kernel(
    const uint16_t *__restrict__ q_bf16, int H, const int32_t *__restrict__ q_seq,
    const uint8_t *__restrict__ codes, const uint8_t *__restrict__ sf,
    const int64_t *__restrict__ cu_ctx, const int32_t *__restrict__ idx, int topk,
    float scale_log2e, uint16_t *__restrict__ out, float *__restrict__ lse) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  PfMisc &ms = *reinterpret_cast<PfMisc *>(sm + kPfOffMisc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = blockIdx.x;
  const int32_t *idx_n = idx + (int64_t)n * topk;
  const int n_tiles = (topk + kPfRows - 1) / kPfRows;

  if (tid == 0) {
    mbar_init(&ms.bar_q, kPfWorkers);
    mbar_init(&ms.bar_s, 1);
    mbar_init(&ms.bar_p, kPfWorkers);
    for (int c = 0; c < 4; ++c) {
      mbar_init(&ms.bar_dq[c], kPfWorkers);
      mbar_init(&ms.bar_pv[c], 1);
    }
    mbar_init(&ms.bar_v[0], kPfWorkers);
    mbar_init(&ms.bar_v[1], kPfWorkers);
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
      constexpr uint32_t idesc_s = idesc_f32acc(0, 0, 128, 64);
      constexpr uint32_t idesc_pv = idesc_f32acc(0, 0, 128, 64) | (1u << 15) | (1u << 16);
      const uint32_t qa = smem_u32(sm + kPfOffQ), ka = smem_u32(sm + kPfOffK);
      const uint32_t ph = smem_u32(sm + kPfOffPhi);
      ok = mbar_wait(&ms.bar_q, 0) && ok;
      for (int g = 0; g < 2 * n_tiles; ++g) {  // pass 1: g < n_tiles; pass 2: the rest
        const bool second = g >= n_tiles;
        for (int cp = 0; cp < 4; ++cp) {
          ok = mbar_wait(&ms.bar_dq[cp], g & 1) && ok;
          tc_fence_after();
#pragma unroll
          for (int kc = 2 * cp; kc < 2 * cp + 2; ++kc)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_f16(tS, desc_k128_sw128(ka + kc * kPfKChunk + 32 * ks),
                      desc_k128_sw128(qa + kc * kPfQChunk + 32 * ks), idesc_s, (kc | ks) != 0);
          if (!second) mma_commit(&ms.bar_pv[cp]);  // pass 1: the chunk pair is free again
        }
        mma_commit(&ms.bar_s);
        ok = mbar_wait(&ms.bar_p, g & 1) && ok;  // S^T read (and, pass 2, Pt written)
        tc_fence_after();
        if (second) {
          const int t = g - n_tiles;
          for (int qb = 0; qb < 4; ++qb) {
            if ((qb & 1) == 0) {  // Vt of channel blocks qb, qb + 1 written
              ok = mbar_wait(&ms.bar_v[qb >> 1], t & 1) && ok;
              tc_fence_after();
            }
#pragma unroll
            for (int ks = 0; ks < kPfRows / 16; ++ks)
              mma_f16(tmem + qb * 64,
                      desc_mn_sw128_atoms(ka + (2 * qb) * kPfKChunk + ks * 16 * 128, kPfKChunk),
                      desc_mn_sw128_atoms(ph + ks * 16 * 128, kPfKChunk), idesc_pv,
                      (t > 0 || ks > 0) ? 1u : 0u);
            mma_commit(&ms.bar_pv[qb]);
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ workers (warps 0..7)
    const int64_t base = cu_ctx[q_seq[n]];
    const int seg = tid & 3, jr = tid >> 2;             // dequantisation: rows jr, jr + 64
    const int quarter = warp & 3, hh = warp >> 2;       // softmax: TMEM lane quarter, head half
    const int jrow = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint4 rc[8];
    uint32_t rs[8];
    auto load_rows = [&](int t) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int slot = t * kPfRows + jr + 64 * hf;
        const int r = slot < topk ? __ldg(idx_n + slot) : -1;
        const int64_t row = base + (r >= 0 ? r : 0);
#pragma unroll
        for (int cp = 0; cp < 4; ++cp) {
          rc[2 * cp + hf] = r >= 0 ? __ldg(reinterpret_cast<const uint4 *>(
                                         codes + row * kCodeBytes + cp * 64 + seg * 16))
                                   : make_uint4(0, 0, 0, 0);
          rs[2 * cp + hf] = r >= 0 ? (uint32_t)__ldg(reinterpret_cast<const uint16_t *>(
                                         sf + row * kSfBytes + cp * 8 + seg * 2))
                                   : 0u;
        }
      }
    };
    auto row_valid = [&](int t) {
      const int slot = t * kPfRows + jrow;
      return slot < topk && __ldg(idx_n + slot) >= 0;
    };
    load_rows(0);

    // ---- the query: FP4-quantised with the main-KV rule, exactly dequantised (as the prefill
    //      kernel)
    for (int k = 0; k < 64 * 32 / kPfWorkers; ++k) {
      const int gi = tid + k * kPfWorkers, h = gi >> 5, grp = gi & 31;
      uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0;
      if (h < H) {
        const uint4 *src =
            reinterpret_cast<const uint4 *>(q_bf16 + ((int64_t)n * H + h) * kD + 16 * grp);
        const uint4 a = __ldg(src), b = __ldg(src + 1);
        const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
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
    fence_async_smem();
    mbar_arrive(&ms.bar_q);

    float mrow[32], lpart[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) mrow[i] = -INFINITY, lpart[i] = 0.0f;

    for (int g = 0; g < 2 * n_tiles; ++g) {
      const bool second = g >= n_tiles;
      const int t = second ? g - n_tiles : g;
      // ---- dequantise tile t into Khat (chunk pair by chunk pair as it is released)
#pragma unroll
      for (int cp = 0; cp < 4; ++cp) {
        if (g > 0) ok = mbar_wait(&ms.bar_pv[cp], (g - 1) & 1) && ok;
        const int kc = 2 * cp + (seg >> 1), u0 = (seg & 1) * 4;
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
        fence_async_smem();
        mbar_arrive(&ms.bar_dq[cp]);
      }
      const bool row_ok = row_valid(t);
      if (g + 1 < 2 * n_tiles) load_rows((g + 1) % n_tiles);

      // ---- S^T of tile t: this thread's row, heads 32hh..32hh+31 (log2 domain)
      ok = __all_sync(0xffffffffu, mbar_wait(&ms.bar_s, g & 1)) && ok;
      tc_fence_after();
      float x[32];
      tmem_ld32(tS + 32 * hh + lane_off, x);
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = row_ok ? x[i] * scale_log2e : -INFINITY;
      if (!second) {  // pass 1: the running maximum of this thread's rows
#pragma unroll
        for (int i = 0; i < 32; ++i) mrow[i] = fmaxf(mrow[i], x[i]);
        tc_fence_before();
        mbar_arrive(&ms.bar_p);
        if (g == n_tiles - 1) {  // each head's maximum over every slot of the token
          float *scratch = reinterpret_cast<float *>(sm + kPfOffPlo);  // [4][64]
          scratch[quarter * 64 + 32 * hh + lane] = reduce_scatter32<true>(mrow, lane);
          pf_bar_workers();
          if (quarter == 0) {
            const int h = 32 * hh + lane;
            ms.mref[h] = fmaxf(fmaxf(scratch[h], scratch[64 + h]),
                               fmaxf(scratch[128 + h], scratch[192 + h]));
          }
          pf_bar_workers();
        }
        continue;
      }
      // ---- pass 2: numerators, FP4 per (head, 16-slot block) = 16 lanes.  Per 16 heads the
      //      block maxima are reduce-scattered over the half-warp (lane l ends with head l's),
      //      each lane rounds one scale, and the scales are broadcast back by shuffles.
      const float *mref = &ms.mref[32 * hh];
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        float p[16], t[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          p[i] = row_ok ? ex2_approx(x[16 * hb + i] - mref[16 * hb + i]) : 0.0f;
          t[i] = p[i];
        }
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) {
          const bool upper = lane & o;
#pragma unroll
          for (int i = 0; i < o; ++i) {
            const float keep = upper ? t[i + o] : t[i], send = upper ? t[i] : t[i + o];
            t[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
          }
        }
        const float sc_mine = fp4_scale(t[0]);
        const float rcp_mine = sc_mine == 0.0f ? 0.0f : __frcp_rn(sc_mine);
#pragma unroll
        for (int uh = 0; uh < 2; ++uh) {
          uint32_t hv[4];
#pragma unroll
          for (int k = 0; k < 8; k += 2) {
            const int i = 8 * uh + k;
            const int src = (lane & 16) | i;
            const float sc0 = __shfl_sync(0xffffffffu, sc_mine, src);
            const float sc1 = __shfl_sync(0xffffffffu, sc_mine, src + 1);
            const float r0 = __shfl_sync(0xffffffffu, rcp_mine, src);
            const float r1 = __shfl_sync(0xffffffffu, rcp_mine, src + 1);
            // Pt = E2M1(p / sc) * sc, exact in fp16 (at most 6 significant bits)
            const uint32_t lv =
                e2m1_round_f16x2(fp4_quot(p[i], sc0, r0), fp4_quot(p[i + 1], sc1, r1));
            const __half2 sc2 = __floats2half2_rn(sc0, sc1);  // exact: E4M3 values
            const __half2 pt = __hmul2(*reinterpret_cast<const __half2 *>(&lv), sc2);
            const float2 ptf = __half22float2(pt);
            lpart[16 * hb + i] += ptf.x;
            lpart[16 * hb + i + 1] += ptf.y;
            hv[k / 2] = *reinterpret_cast<const uint32_t *>(&pt);
          }
          const int u = 2 * hb + uh;
          const int off = jrow * 128 + (((4 * hh + u) ^ (jrow & 7)) << 4);
          *reinterpret_cast<uint4 *>(sm + kPfOffPhi + off) =
              make_uint4(hv[0], hv[1], hv[2], hv[3]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&ms.bar_p);
      // ---- V re-quantised in place, in two steps of two 128-channel blocks (the PV MMAs of
      //      blocks 0-1 run during the second step): thread = 8 channels of one 16-row block.
      //      S^T(t) is complete (its commit arrived), so Khat is no longer read by it.  The
      //      level E2M1(x / sc) times sc is exact in fp16.
      {
        const int b = tid >> 5;  // 16-row block 0..7
        const int u = lane & 7;  // 16-byte unit of the chunk
#pragma unroll 1
        for (int step = 0; step < 2; ++step) {
          const int kc = 4 * step + (lane >> 3);  // chunks 0..3, then 4..7
          uint8_t *chunk = sm + kPfOffK + kc * kPfKChunk;
          __half2 amax[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) amax[e] = __float2half2_rn(0.0f);
#pragma unroll 4
          for (int rr = 0; rr < 16; ++rr) {
            const int j = 16 * b + rr;
            const uint4 v =
                *reinterpret_cast<const uint4 *>(chunk + j * 128 + ((u ^ (j & 7)) << 4));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              amax[e] = __hmax2(amax[e], __habs2(*reinterpret_cast<const __half2 *>(&w[e])));
          }
          __half2 sc2[4], rc2[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            sc2[e] = fp4_scale_f16x2(amax[e]);
            const float2 sf2 = __half22float2(sc2[e]);
            rc2[e] = __floats2half2_rn(sf2.x == 0.0f ? 0.0f : __frcp_rn(sf2.x),
                                       sf2.y == 0.0f ? 0.0f : __frcp_rn(sf2.y));
          }
#pragma unroll 4
          for (int rr = 0; rr < 16; ++rr) {
            const int j = 16 * b + rr;
            uint4 *pv = reinterpret_cast<uint4 *>(chunk + j * 128 + ((u ^ (j & 7)) << 4));
            const uint4 v = *pv;
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t lv =
                  fp4_level_f16x2(*reinterpret_cast<const __half2 *>(&w[e]), sc2[e], rc2[e]);
              const __half2 q = __hmul2(*reinterpret_cast<const __half2 *>(&lv), sc2[e]);  // exact
              w[e] = *reinterpret_cast<const uint32_t *>(&q);
            }
            *pv = make_uint4(w[0], w[1], w[2], w[3]);
          }
          fence_async_smem();
          mbar_arrive(&ms.bar_v[step]);
        }
      }
    }

    // ---- epilogue: sums of the quantised numerators, lse, O / l in bf16
    ok = __all_sync(0xffffffffu, mbar_wait(&ms.bar_pv[3], (2 * n_tiles - 1) & 1)) && ok;
    tc_fence_after();
    float *scratch = reinterpret_cast<float *>(sm + kPfOffPlo);
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
    const int hn = min(32, H - 32 * hh);
#pragma unroll 1
    for (int qb = 0; qb < 4; ++qb) {
      float o[32];
      tmem_ld32(tmem + qb * 64 + 32 * hh + lane_off, o);
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

cudaError_t launch_attn_fp4pv(const void *q_bf16, int T, int H, const int32_t *q_seq,
                              const uint8_t *codes, const uint8_t *sf, const int64_t *cu_ctx,
                              const int32_t *idx, int topk, float scale, void *out_bf16,
                              float *lse, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  cudaError_t e = set_smem_once(attn_fp4pv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kPfSmem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attn_fp4pv_kernel, dim3(T), dim3(kPfThreads), kPfSmem, st,
                 static_cast<const uint16_t *>(q_bf16), H, q_seq, codes, sf, cu_ctx, idx, topk,
                 scale * 1.4426950408889634f, static_cast<uint16_t *>(out_bf16), lse);
  note_launches(1);
  return e;
}

}  // namespace csa2

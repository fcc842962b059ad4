// attn_simt.cu -- sparse attention over gathered FP4 rows on CUDA cores (general path).
//
// For each query n and head h: softmax(scale * q_h . khat_j) over the selected rows j, applied
// to the same rows (K = V = the dequantised latent row; the model card's Introduction, CSA2
// paragraph: the sparse attention reads the FP4 main-KV rows that a shared Top-K index set names).
//
// Grid: (split, head group of 16, query).  A CTA walks its share of the Top-K slots in chunks of
// 32 rows: gather codes + scales, dequantise exactly into fp32 shared memory, scores for 16 heads
// x 32 rows, online-softmax update, P.V accumulate in registers.  With one split per query the
// CTA writes the final bf16 output and lse; otherwise it writes (O, m, l) partials that
// attn_combine_kernel merges.
#include "common.cuh"

namespace csa2 {

constexpr int kChunk = 32;   // rows per step
constexpr int kHG = 16;      // heads per CTA
constexpr int kAT = 256;     // threads per CTA
constexpr int kKsStride = kD + 1;

struct AttnSmem {
  uint16_t q[kHG * kD];          // bf16 query rows of this head group
  float ks[kChunk * kKsStride];  // dequantised rows
  float p[kHG * (kChunk + 1)];   // scores, then probabilities
  float alpha[kHG];
  int valid[kChunk];
};

__device__ __forceinline__ uint16_t float_to_bf16_bits_exact(float f) {
  return (uint16_t)(__float_as_uint(f) >> 16);  // exact for dequantised FP4 values
}

__global__ void __launch_bounds__(kAT) attn_partial_kernel(
    const uint16_t *__restrict__ q_bf16, const uint8_t *__restrict__ q_codes,
    const uint8_t *__restrict__ q_sf, int H, const int32_t *__restrict__ q_seq,
    const uint8_t *__restrict__ codes, const uint8_t *__restrict__ sf,
    const int64_t *__restrict__ cu_ctx, const int32_t *__restrict__ idx, int topk, float scale,
    int slots_per_split, int n_split, float *__restrict__ o_part, float *__restrict__ m_part,
    float *__restrict__ l_part, uint16_t *__restrict__ out, float *__restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  AttnSmem &sm = *reinterpret_cast<AttnSmem *>(smem_raw);
  const int s = blockIdx.x, hg = blockIdx.y, n = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int h0 = hg * kHG;
  const int nh = min(kHG, H - h0);
  const int64_t base = cu_ctx[q_seq ? q_seq[n] : n];

  // query rows -> bf16 in shared memory
  for (int i = tid; i < kHG * kD; i += kAT) {
    const int h = i / kD, c = i % kD;
    uint16_t v = 0;
    if (h < nh) {
      const int64_t qrow = (int64_t)n * H + h0 + h;
      if (q_bf16) {
        v = q_bf16[qrow * kD + c];
      } else {
        const uint32_t byte = q_codes[qrow * kCodeBytes + c / 2];
        const float x = e2m1_to_float((c & 1) ? (byte >> 4) : (byte & 15u)) *
                        e4m3_to_float(q_sf[qrow * kSfBytes + c / 16]);
        v = float_to_bf16_bits_exact(x);
      }
    }
    sm.q[i] = v;
  }

  float o0[kHG], o1[kHG];
#pragma unroll
  for (int h = 0; h < kHG; ++h) o0[h] = o1[h] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f;  // per head, owned by (warp, half): see softmax below

  const int j_begin = s * slots_per_split;
  const int j_end = min(topk, j_begin + slots_per_split);
  const int32_t *idx_n = idx + (int64_t)n * topk;

  for (int jc = j_begin; jc < j_end; jc += kChunk) {
    __syncthreads();  // previous chunk fully consumed
    // gather + dequantise: thread -> (row tid/8, 64-channel segment tid%8)
    {
      const int j = tid >> 3, seg = tid & 7;
      const int slot = jc + j;
      const int r = (slot < j_end) ? idx_n[slot] : -1;
      float *dst = sm.ks + j * kKsStride + seg * 64;
      if (r >= 0) {
        const int64_t row = base + r;
        const uint4 *cp = reinterpret_cast<const uint4 *>(codes + row * kCodeBytes + seg * 32);
        const uint32_t sfw = *reinterpret_cast<const uint32_t *>(sf + row * kSfBytes + seg * 4);
        const uint4 c0 = __ldg(cp), c1 = __ldg(cp + 1);
        const uint32_t wds[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float sc = e4m3_to_float((sfw >> (8 * g)) & 0xFFu);
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            const uint32_t wv = wds[2 * g + b];
#pragma unroll
            for (int k = 0; k < 8; ++k) dst[16 * g + 8 * b + k] = e2m1_to_float((wv >> (4 * k)) & 15u) * sc;
          }
        }
      } else {
#pragma unroll 8
        for (int k = 0; k < 64; ++k) dst[k] = 0.0f;
      }
      if (seg == 0) sm.valid[j] = (r >= 0);
    }
    __syncthreads();
    // scores: thread -> row j = lane, heads 2*wid, 2*wid+1
    {
      const float *kr = sm.ks + lane * kKsStride;
      const int ha = 2 * wid, hb = 2 * wid + 1;
      const uint32_t *qa = reinterpret_cast<const uint32_t *>(sm.q + ha * kD);
      const uint32_t *qb = reinterpret_cast<const uint32_t *>(sm.q + hb * kD);
      float da = 0.0f, db = 0.0f;
#pragma unroll 4
      for (int c2 = 0; c2 < kD / 2; ++c2) {
        const float k0 = kr[2 * c2], k1 = kr[2 * c2 + 1];
        const uint32_t va = qa[c2], vb = qb[c2];
        da = fmaf(bf16_lo(va), k0, da);
        da = fmaf(bf16_hi(va), k1, da);
        db = fmaf(bf16_lo(vb), k0, db);
        db = fmaf(bf16_hi(vb), k1, db);
      }
      const bool v = sm.valid[lane];
      sm.p[ha * (kChunk + 1) + lane] = v ? da * scale : -INFINITY;
      sm.p[hb * (kChunk + 1) + lane] = v ? db * scale : -INFINITY;
    }
    __syncthreads();
    // online softmax: warp wid owns heads 2*wid and 2*wid+1, lane = row
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int h = 2 * wid + e;
      const float sv = sm.p[h * (kChunk + 1) + lane];
      const float cmax = warp_max(sv);
      const float m_old = __shfl_sync(0xffffffffu, m_run, e);
      const float m_new = fmaxf(m_old, cmax);
      const float pv = (sv == -INFINITY) ? 0.0f : expf(sv - m_new);
      const float alpha = (m_old == -INFINITY) ? 0.0f : expf(m_old - m_new);
      const float psum = warp_sum(pv);
      sm.p[h * (kChunk + 1) + lane] = pv;
      if (lane == e) {
        m_run = m_new;
        l_run = l_run * alpha + psum;
      }
      if (lane == 0) sm.alpha[h] = (m_new == -INFINITY) ? 1.0f : alpha;
    }
    __syncthreads();
    // O update: thread -> channels tid and tid + 256, all heads of the group
    {
      const int c0 = tid, c1 = tid + 256;
#pragma unroll
      for (int h = 0; h < kHG; ++h) {
        const float a = sm.alpha[h];
        o0[h] *= a;
        o1[h] *= a;
      }
#pragma unroll 4
      for (int j = 0; j < kChunk; ++j) {
        const float k0 = sm.ks[j * kKsStride + c0], k1 = sm.ks[j * kKsStride + c1];
#pragma unroll
        for (int h = 0; h < kHG; ++h) {
          const float p = sm.p[h * (kChunk + 1) + j];
          o0[h] = fmaf(p, k0, o0[h]);
          o1[h] = fmaf(p, k1, o1[h]);
        }
      }
    }
  }
  __syncthreads();
  // publish per-head (m, l) through shared memory: lanes 0/1 of warp w hold heads 2w, 2w+1
  float *ml = sm.p;  // reuse: [kHG] m then [kHG] l
  if (lane < 2) {
    ml[2 * wid + lane] = m_run;
    ml[kHG + 2 * wid + lane] = l_run;
  }
  __syncthreads();
  const int c0 = tid, c1 = tid + 256;
  if (n_split == 1) {
    for (int h = 0; h < nh; ++h) {
      const float m = ml[h], l = ml[kHG + h];
      const int64_t orow = ((int64_t)n * H + h0 + h) * kD;
      float r0 = 0.0f, r1 = 0.0f;
      if (l > 0.0f) {
        r0 = o0[h] / l;
        r1 = o1[h] / l;
      }
      out[orow + c0] = __bfloat16_as_ushort(__float2bfloat16_rn(r0));
      out[orow + c1] = __bfloat16_as_ushort(__float2bfloat16_rn(r1));
      if (tid == 0 && lse) lse[(int64_t)n * H + h0 + h] = (l > 0.0f) ? m + logf(l) : -INFINITY;
    }
  } else {
    for (int h = 0; h < nh; ++h) {
      const int64_t prow = (((int64_t)n * n_split + s) * H + h0 + h);
      o_part[prow * kD + c0] = o0[h];
      o_part[prow * kD + c1] = o1[h];
      if (tid == 0) {
        m_part[prow] = ml[h];
        l_part[prow] = ml[kHG + h];
      }
    }
  }
}

// Merge split partials: out = sum_s O_s e^{m_s - M} / sum_s l_s e^{m_s - M}.
__global__ void __launch_bounds__(128) attn_combine_kernel(
    int H, int n_split, const float *__restrict__ o_part, const float *__restrict__ m_part,
    const float *__restrict__ l_part, uint16_t *__restrict__ out, float *__restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  const int h = blockIdx.x, n = blockIdx.y;
  float M = -INFINITY;
  for (int s = 0; s < n_split; ++s) M = fmaxf(M, m_part[((int64_t)n * n_split + s) * H + h]);
  float L = 0.0f;
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int s = 0; s < n_split; ++s) {
    const int64_t prow = ((int64_t)n * n_split + s) * H + h;
    const float l = l_part[prow];
    if (!(l > 0.0f)) continue;
    const float wgt = expf(m_part[prow] - M);
    L += l * wgt;
    const float4 o = reinterpret_cast<const float4 *>(o_part + prow * kD)[threadIdx.x];
    acc[0] = fmaf(o.x, wgt, acc[0]);
    acc[1] = fmaf(o.y, wgt, acc[1]);
    acc[2] = fmaf(o.z, wgt, acc[2]);
    acc[3] = fmaf(o.w, wgt, acc[3]);
  }
  const int64_t orow = ((int64_t)n * H + h) * kD + 4 * threadIdx.x;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    out[orow + k] = __bfloat16_as_ushort(__float2bfloat16_rn(L > 0.0f ? acc[k] / L : 0.0f));
  if (threadIdx.x == 0 && lse) lse[(int64_t)n * H + h] = (L > 0.0f) ? M + logf(L) : -INFINITY;
}

static void attn_plan(int nq, int H, int topk, int *slots_per_split, int *n_split) {
  const int hgs = (H + kHG - 1) / kHG;
  const int chunks = (topk + kChunk - 1) / kChunk;
  const int64_t ctas = (int64_t)nq * hgs;
  int want = (int)((4 * 148 + ctas - 1) / ctas);  // aim for ~4 CTAs per SM
  want = max(1, min(want, chunks));
  const int chunks_per = (chunks + want - 1) / want;
  *slots_per_split = chunks_per * kChunk;
  *n_split = (chunks + chunks_per - 1) / chunks_per;
}

size_t attn_workspace_bytes(int nq, int H, int topk) {
  int sps, ns;
  attn_plan(nq, H, topk, &sps, &ns);
  if (ns == 1) return 0;
  const size_t rows = (size_t)nq * ns * H;
  return rows * kD * sizeof(float) + 2 * rows * sizeof(float) + 512;
}

cudaError_t launch_attn(const void *q_bf16, const uint8_t *q_codes, const uint8_t *q_sf, int nq,
                        int H, const int32_t *q_seq, const uint8_t *codes, const uint8_t *sf,
                        const int64_t *cu_ctx, const int32_t *idx, int topk, float scale,
                        void *out_bf16, float *lse, void *workspace, cudaStream_t st) {
  if (nq == 0) return cudaSuccess;
  int sps, ns;
  attn_plan(nq, H, topk, &sps, &ns);
  const size_t rows = (size_t)nq * ns * H;
  float *o_part = static_cast<float *>(workspace);
  float *m_part = o_part ? o_part + rows * kD : nullptr;
  float *l_part = m_part ? m_part + rows : nullptr;
  const size_t smem = sizeof(AttnSmem);
  static_assert(sizeof(AttnSmem) <= 227 * 1024, "shared memory");
  cudaError_t e = set_smem_once(attn_partial_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(ns, (H + kHG - 1) / kHG, nq);
  e = launch_pdl(attn_partial_kernel, grid, dim3(kAT), smem, st,
                 static_cast<const uint16_t *>(q_bf16), q_codes, q_sf, H, q_seq, codes, sf,
                 cu_ctx, idx, topk, scale, sps, ns, o_part, m_part, l_part,
                 static_cast<uint16_t *>(out_bf16), lse);
  note_launches(1);
  if (e != cudaSuccess || ns == 1) return e;
  e = launch_pdl(attn_combine_kernel, dim3(H, nq), dim3(128), 0, st, H, ns,
                 (const float *)o_part, (const float *)m_part, (const float *)l_part,
                 static_cast<uint16_t *>(out_bf16), lse);
  note_launches(1);
  return e;
}

}  // namespace csa2

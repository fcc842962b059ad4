// kv_quant.cu -- FP4 main-KV quantisation: bf16 rows -> E2M1 codes + one E4M3 scale per 16
// channels (DeepSeek-V4.1-Flash model card, Introduction, CSA2 paragraph).
//
// One warp per row, one lane per 16-channel group (a 512-channel row is exactly 32 groups, so a
// warp moves 1 KB in with two 16-byte loads per lane and 256 + 32 bytes out with one 8-byte and
// one 1-byte store per lane, all coalesced).  HBM-bound: 1024 B read + 288 B written per row.
//
// The code of x is E2M1(fp32(x / s)) rounded to nearest even.  x is bf16 (8 significant bits)
// and s an E4M3 value (4), so x / s either equals a decision point T (a midpoint between E2M1
// neighbours: 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5) or differs from it by more than 2^-9
// relative -- far more than an fp32 rounding.  The kernel forms the quotient without a division:
// q0 = x * rcp(s), then one correction q = q0 - (q0 s - x) rcp(s) (the remainder is exact in an
// fma).  q is within an ulp of x / s, and equals T exactly when x = T s, so the hardware
// conversion to E2M1 (round to nearest even, saturating at 6) takes the decision the rounded
// quotient takes, ties included.  A group holding an infinity takes the comparison path instead
// (|x| against the exact products T * s, three comparisons per value), which saturates it.
#include "common.cuh"

namespace csa2 {

// Eight fp32 values -> eight E2M1 codes in one word (value 2k in the low nibble of byte k), by
// the conversion instruction: round to nearest even, saturating at +-6, sign kept.
__device__ __forceinline__ uint32_t e2m1x8_rn(const float *q) {
  uint32_t w;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}\n"
      : "=r"(w)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return w;
}

// Quantise one 16-channel group held as 8 packed bf16 pairs.  Returns the scale code and writes
// the 8 code bytes (channel 2j low nibble, 2j+1 high nibble) into *codes64.
__device__ __forceinline__ uint32_t quant_group16(const uint32_t (&v)[8], uint64_t *codes64) {
  // amax by packed bf16 maxima of the magnitudes (exact)
  uint32_t m = v[0] & 0x7FFF7FFFu;
#pragma unroll
  for (int i = 1; i < 8; ++i) {
    const uint32_t a = v[i] & 0x7FFF7FFFu;
    __nv_bfloat162 r = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&m),
                               *reinterpret_cast<const __nv_bfloat162 *>(&a));
    m = *reinterpret_cast<const uint32_t *>(&r);
  }
  const float amax = fmaxf(bf16_lo(m), bf16_hi(m));
  const uint32_t scode = float_to_e4m3_sat(__fdiv_rn(amax, 6.0f));
  const float sd = e4m3_to_float(scode);
  uint64_t packed = 0;
  if (sd != 0.0f && amax < INFINITY) {
    const float rcp = __frcp_rn(sd);
    float q[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float x = (i & 1) ? bf16_hi(v[i >> 1]) : bf16_lo(v[i >> 1]);
      const float q0 = x * rcp;
      // q0 - (q0 s - x) rcp: the remainder's sign is chosen so that x = -0 keeps its sign
      // (-0 + -0); written as x - q0 s it would come out +0
      q[i] = fmaf(-fmaf(q0, sd, -x), rcp, q0);
    }
    packed = ((uint64_t)e2m1x8_rn(q + 8) << 32) | e2m1x8_rn(q);
  } else if (sd != 0.0f) {
    const float t1 = 0.25f * sd, t2 = 0.75f * sd, t3 = 1.25f * sd, t4 = 1.75f * sd;
    const float t5 = 2.5f * sd, t6 = 3.5f * sd, t7 = 5.0f * sd;
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float x = (i & 1) ? bf16_hi(v[i >> 1]) : bf16_lo(v[i >> 1]);
      const float a = fabsf(x);
      const bool ge4 = a >= t4;
      const bool ge2 = a >= (ge4 ? t6 : t2);
      const bool gt1 = a > (ge2 ? (ge4 ? t7 : t3) : (ge4 ? t5 : t1));
      const uint32_t code = (ge4 ? 4u : 0u) | (ge2 ? 2u : 0u) | (gt1 ? 1u : 0u) |
                            ((__float_as_uint(x) >> 28) & 8u);
      if (i < 8) lo |= code << (4 * i);
      else hi |= code << (4 * (i - 8));
    }
    packed = ((uint64_t)hi << 32) | lo;
  }
  *codes64 = packed;
  return scode;
}

__global__ void __launch_bounds__(256) kv_quant_kernel(const uint16_t *__restrict__ x,
                                                       int64_t n_rows, int d,
                                                       const int64_t *__restrict__ out_rows,
                                                       uint8_t *__restrict__ codes,
                                                       uint8_t *__restrict__ sf) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= n_rows) return;
  const int64_t orow = out_rows ? out_rows[row] : row;
  const int groups = d >> 4;
  const uint16_t *xr = x + row * d;
  for (int g = lane; g < groups; g += 32) {
    const uint4 *src = reinterpret_cast<const uint4 *>(xr + 16 * g);
    uint4 a = __ldg(src), b = __ldg(src + 1);
    uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint64_t packed;
    uint32_t scode = quant_group16(v, &packed);
    *reinterpret_cast<uint64_t *>(codes + orow * (d >> 1) + 8 * g) = packed;
    sf[orow * groups + g] = (uint8_t)scode;
  }
}

cudaError_t launch_kv_quant(const void *x, int64_t n_rows, int d, const int64_t *out_rows,
                            uint8_t *codes, uint8_t *sf, cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  const int rows_per_cta = 8;
  const int64_t grid = (n_rows + rows_per_cta - 1) / rows_per_cta;
  const cudaError_t e = launch_pdl(kv_quant_kernel, dim3((unsigned)grid), dim3(32 * rows_per_cta),
                                   0, st, static_cast<const uint16_t *>(x), n_rows, d, out_rows,
                                   codes, sf);
  note_launches(1);
  return e;
}

}  // namespace csa2

// ------------------------------------------------------------------------------------------
// FP8 local sliding-window rows ("DeepSeek V4.1-Flash", aiwiki.ai, section "KV-cache formats and
// bounded replay": the local sliding-window KV is stored in FP8): every bf16 element -> E4M3
// ("fn"), round to nearest even, saturating at +-448, sign kept, no scale.  One thread per 16
// elements: two 16-byte loads, eight two-element conversions, one 16-byte store.
// ------------------------------------------------------------------------------------------
namespace csa2 {

__device__ __forceinline__ uint32_t bf16x2_to_e4m3x2(uint32_t v) {
  uint16_t r;
  // the first source lands in the upper byte: channel 2i (low bf16) goes to the low byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(bf16_hi(v)), "f"(bf16_lo(v)));
  return r;
}

__global__ void __launch_bounds__(256) fp8_quant_kernel(const uint16_t *__restrict__ x,
                                                        int64_t n_rows, int d,
                                                        const int64_t *__restrict__ out_rows,
                                                        uint8_t *__restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int per_row = d >> 4;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_rows * per_row) return;
  const int64_t row = i / per_row;
  const int g = (int)(i - row * per_row);
  const int64_t orow = out_rows ? out_rows[row] : row;
  const uint4 *src = reinterpret_cast<const uint4 *>(x + row * d + 16 * g);
  const uint4 a = __ldg(src), b = __ldg(src + 1);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    o[k] = bf16x2_to_e4m3x2(w[2 * k]) | (bf16x2_to_e4m3x2(w[2 * k + 1]) << 16);
  *reinterpret_cast<uint4 *>(out + orow * d + 16 * g) = make_uint4(o[0], o[1], o[2], o[3]);
}

cudaError_t launch_fp8_quant(const void *x, int64_t n_rows, int d, const int64_t *out_rows,
                             uint8_t *out, cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  const int64_t threads = n_rows * (d >> 4);
  const cudaError_t e = launch_pdl(fp8_quant_kernel, dim3((unsigned)((threads + 255) / 256)),
                                   dim3(256), 0, st, static_cast<const uint16_t *>(x), n_rows, d,
                                   out_rows, out);
  note_launches(1);
  return e;
}

}  // namespace csa2

// kv_quant.cu -- FP4 main-KV quantisation: bf16 rows -> E2M1 codes + one E4M3 scale per 16
// channels (DeepSeek-V4.1-Flash model card, Introduction, CSA2 paragraph).
//
// One warp per row, one lane per 16-channel group (a 512-channel row is exactly 32 groups, so a
// warp moves 1 KB in with two 16-byte loads per lane and 256 + 32 bytes out with one 8-byte and
// one 1-byte store per lane, all coalesced).  HBM-bound: 1024 B read + 288 B written per row.
//
// The code of x is E2M1(fp32(x / s)) rounded to nearest even.  It is computed without the
// division: x is bf16 (8 significant bits) and s an E4M3 value (4), so x / s either equals a
// decision point T (a midpoint between E2M1 neighbours: 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5) or
// differs from it by more than 2^-11 relative -- far more than one fp32 rounding -- and T * s
// (at most 7 significant bits) is exact in fp32.  So comparing |x| with T * s takes exactly the
// decision the rounded quotient takes, ties included.  Three comparisons find the code: against
// 1.75 s, then 0.75 s or 3.5 s (all "at least": the even code wins a tie there), then 0.25 s,
// 1.25 s, 2.5 s or 5 s ("greater than": the even code is below).
#include "common.cuh"

namespace csa2 {

// Quantise one 16-channel group held as 8 packed bf16 pairs.  Returns the scale code and writes
// the 8 code bytes (channel 2j low nibble, 2j+1 high nibble) into *codes64.
__device__ __forceinline__ uint32_t quant_group16(const uint32_t (&v)[8], uint64_t *codes64) {
  float x[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = bf16_lo(v[i]);
    x[2 * i + 1] = bf16_hi(v[i]);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const uint32_t scode = float_to_e4m3_sat(__fdiv_rn(amax, 6.0f));
  const float sd = e4m3_to_float(scode);
  uint64_t packed = 0;
  if (sd != 0.0f) {
    const float t1 = 0.25f * sd, t2 = 0.75f * sd, t3 = 1.25f * sd, t4 = 1.75f * sd;
    const float t5 = 2.5f * sd, t6 = 3.5f * sd, t7 = 5.0f * sd;
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float a = fabsf(x[i]);
      const bool ge4 = a >= t4;
      const bool ge2 = a >= (ge4 ? t6 : t2);
      const bool gt1 = a > (ge2 ? (ge4 ? t7 : t3) : (ge4 ? t5 : t1));
      const uint32_t code = (ge4 ? 4u : 0u) | (ge2 ? 2u : 0u) | (gt1 ? 1u : 0u) |
                            ((__float_as_uint(x[i]) >> 28) & 8u);
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

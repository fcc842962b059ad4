// kv_quant.cu -- FP4 main-KV quantisation: bf16 rows -> E2M1 codes + one E4M3 scale per 16
// channels (DeepSeek-V4.1-Flash model card, Introduction, CSA2 paragraph).
//
// One warp per row, one lane per 16-channel group (a 512-channel row is exactly 32 groups, so a
// warp moves 1 KB in with two 16-byte loads per lane and 256 + 32 bytes out with one 8-byte and
// one 1-byte store per lane, all coalesced).  HBM-bound: 1024 B read + 288 B written per row.
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
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float q = __fdiv_rn(x[i], sd);
      const uint32_t code = e2m1_mag_code(fabsf(q)) | ((__float_as_uint(q) >> 28) & 8u);
      packed |= (uint64_t)code << (4 * i);
    }
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

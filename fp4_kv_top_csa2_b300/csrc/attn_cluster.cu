// attn_cluster.cu -- the decode attention's tile kernel for few tiles: one thread-block cluster
// of 8 CTAs per tile of 128 selected rows, CTA r owning the 64-channel slice [64 r, 64 r + 64).
//
// Same result as attn_mma.cu's tile kernel (sequence n, head h: softmax_j(scale * q_h . khat_j)
// over the tile's rows j, applied to the same rows; the model card's Introduction, CSA2
// paragraph: the sparse attention reads the FP4 main-KV rows that a shared Top-K index set
// names), and the same partials for its combine kernel.  A single CTA per tile is a chain of
// 48 tensor-core instructions plus a 128 KB epilogue; when a step has only a few tiles (one
// decoding sequence: 16 tiles for 2,048 rows) most SMs idle while that chain runs.  Splitting
// the channels over a cluster cuts every per-CTA term by the cluster size except the exchanges:
//   1. CTA r loads Q[:, slice r] (64 heads x 64 channels, bf16) and the slice of the tile's 128
//      rows (32 code bytes + 4 scales each, or 64 E4M3 bytes of a local window row), dequantised
//      exactly to bf16 (the E2M1 pair through cvt to fp16 and a move of the bit fields).
//   2. S_r = Q_r Khat_r^T: kind::f16, M=128 (64 heads, padded) x N=128 rows x K=64: 4 MMAs.
//   3. S = sum_r S_r, all-reduced through distributed shared memory with bulk copies (the DMA
//      engine, not per-thread remote accesses): S_r is staged as 8 contiguous 4 KB slices of 16
//      rows; slice k goes to CTA k, which sums the 8 partials of its slice in rank order and
//      sends the sum back to all 8 CTAs.  Every CTA then holds the whole S of the tile.
//   4. Every CTA forms the softmax numerators of all 128 rows itself (the tile's per-head
//      maximum m, p = 2^(s - m), split into bf16 hi + lo by truncation) as the A operand
//      [P_hi; P_lo] (M row = head and plane, K = the tile's row); CTA 0 writes m and the sums.
//   5. O_r = [P_hi; P_lo] Vhat_r: M=128 x N=64 channels x K=128 rows: 8 MMAs.  The M rows put a
//      head's hi and lo products 16 TMEM lanes apart in one warp's lane quarter, so one shuffle
//      adds them; each CTA stores 64 channels of every head's partial row.
// Every wait on a copy or on the tensor core is bounded (sm100.cuh mbar_wait); the two cluster
// barriers (peers' barriers initialised before the first copy; every copy landed before any CTA
// exits) are hardware barriers over co-resident CTAs.
#include "sm100.cuh"

namespace csa2 {

constexpr int kClR = 8;           // CTAs per cluster = 64-channel slices of a row
constexpr int kClRows = 128;      // rows per tile
constexpr int kClThreads = 256;
constexpr int kClSlice = 64 * 16 * 4;             // 16 rows of S for 64 heads, fp32 (4 KB)
constexpr int kClOffQ = 0;                        // Q slice: 64 heads x 128 B (8 KB)
constexpr int kClOffK = 8 * 1024;                 // row slice: 128 rows x 128 B (16 KB)
// S_r as 8 slices (32 KB); slice k becomes the reduced slice k in place: this CTA's own slice
// element by element as it sums, slice k != r when CTA k's all-gather copy lands, which CTA k
// sends only after this CTA's copy of slice k has reached it
constexpr int kClOffSB = kClOffK + 16 * 1024;
constexpr int kClOffRB = kClOffSB + 8 * kClSlice; // peers' partials of this CTA's slice (32 KB)
// [P_hi; P_lo]: 2 chunks x 128 x 128 B (32 KB) over the peers' partials, dead once summed
constexpr int kClOffP = kClOffRB;
constexpr int kClPChunk = 128 * 128;
constexpr int kClOffMisc = kClOffRB + 8 * kClSlice;
constexpr int kClSmem = kClOffMisc + 1024 + 1024;  // + alignment slack
// The M=128 read of Q covers 16 KB from its start (64 real rows, then the row slice): readable,
// and it only feeds accumulator lanes 64..127 of S, which are never read.
static_assert(kClOffQ + 128 * 128 <= kClOffSB, "Q over-read stays in shared memory");
static_assert(kClOffK % 1024 == 0 && kClOffP % 1024 == 0, "swizzled operands 1024-aligned");

struct ClMisc {
  uint8_t slot_ok[kClRows];  // first: read as 16-byte vectors
  uint64_t bar_s, bar_o;     // tensor core: S_r, O_r complete
  uint64_t bar_rs, bar_ag;   // the 7 peers' partials of this slice; the 7 reduced slices
  uint32_t tmem_base, pad;
};
static_assert(sizeof(ClMisc) <= 1024, "misc block");

// Float4 index of (head h, float4 u of its 16 rows) inside a slice: rows of 64 B, u XORed with
// bits 1..2 of h so that 32 consecutive heads writing one u hit 8 different bank groups.
__device__ __forceinline__ int cl_sidx(int h, int u) { return h * 4 + (u ^ ((h >> 1) & 3)); }

// M row of the PV operand for (head h, plane pl): lane quarter h / 16 holds the 16 heads' hi
// rows, then their lo rows.
__device__ __forceinline__ int cl_mrow(int h, int pl) { return 32 * (h >> 4) + 16 * pl + (h & 15); }

// 2^x on the special-function unit (relative error a few 2^-23; -inf gives +0).
__device__ __forceinline__ float cl_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __cluster_dims__(kClR, 1, 1) __launch_bounds__(kClThreads, 2)
    attn_cluster_kernel(const uint16_t *__restrict__ q, int H, const uint8_t *__restrict__ codes,
                        const uint8_t *__restrict__ sf, const int64_t *__restrict__ cu_ctx,
                        const int32_t *__restrict__ idx, int topk, float scale_log2e,
                        int n_tiles, int n_sel_tiles, float *__restrict__ o_part,
                        float *__restrict__ m_part, float *__restrict__ l_part,
                        const uint8_t *__restrict__ swa_kv, int ring, int n_win) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  // the same offset in every CTA of the cluster, so dsmem_map of a local address names the
  // peer's copy of the same object
  uint8_t *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  ClMisc &ms = *reinterpret_cast<ClMisc *>(sm + kClOffMisc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t r = cluster_ctarank();
  const int tile = blockIdx.x / kClR, n = blockIdx.y;

  if (tid == 0) {
    mbar_init(&ms.bar_s, 1);
    mbar_init(&ms.bar_o, 1);
    mbar_init(&ms.bar_rs, 1);
    mbar_init(&ms.bar_ag, 1);
    mbar_arrive_expect_tx(&ms.bar_rs, (kClR - 1) * kClSlice);
    mbar_arrive_expect_tx(&ms.bar_ag, (kClR - 1) * kClSlice);
    fence_barrier_init();
  }
  __syncthreads();
  // this CTA's barriers are initialised (released by fence_barrier_init; matched before the
  // first copy)
  cluster_arrive_relaxed();
  pdl_wait();
  const int64_t base = cu_ctx[n];
  bool ok = true;

  // ---- 1. loads: Q slice, thread = (head hq, 16 channels; heads >= H are zero rows); row
  // slice, thread = (row j, 32 channels 64 r + 32 hf ..)
  const int hq = tid >> 2, part = tid & 3;
  uint4 qa0 = make_uint4(0, 0, 0, 0), qa1 = qa0;
  if (hq < H) {
    const uint4 *src =
        reinterpret_cast<const uint4 *>(q + ((int64_t)n * H + hq) * kD + 64 * r + 16 * part);
    qa0 = __ldg(src);
    qa1 = __ldg(src + 1);
  }
  const int j = tid >> 1, hf = tid & 1;
  const bool win = tile >= n_sel_tiles;  // a tile of the local window
  bool valid;
  uint4 rc0 = make_uint4(0, 0, 0, 0), rc1 = rc0;  // FP4: codes in rc0; E4M3 window row: both
  uint32_t s2 = 0;                              // FP4: the two scales
  if (!win) {
    const int slot = tile * kClRows + j;
    const int rr = slot < topk ? __ldg(idx + (int64_t)n * topk + slot) : -1;
    valid = rr >= 0;
    if (valid) {
      const int64_t row = base + rr;
      rc0 = __ldg(reinterpret_cast<const uint4 *>(codes + row * kCodeBytes + 32 * r + 16 * hf));
      s2 = __ldg(reinterpret_cast<const uint16_t *>(sf + row * kSfBytes + 4 * r + 2 * hf));
    }
  } else {
    // window slot wi of the last nw = min(n_win, L) positions t = L - nw + wi; position t's
    // local row is n * ring + t % ring
    const int64_t L = cu_ctx[n + 1] - base;
    const int64_t nw = L < n_win ? L : n_win;
    const int64_t wi = (int64_t)(tile - n_sel_tiles) * kClRows + j;
    valid = wi < nw;
    if (valid) {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          swa_kv + ((int64_t)n * ring + (L - nw + wi) % ring) * kD + 64 * r + 32 * hf);
      rc0 = __ldg(src);
      rc1 = __ldg(src + 1);
    }
  }
  // TMEM while the rows are in flight; the next kernel may start once every CTA holds its own
  if (warp == 0) {
    tmem_alloc(&ms.tmem_base, 256);
    tmem_relinquish();
  }
  // ---- 1. dequantise (exact) into the swizzled operands
  {
    uint8_t *row = sm + kClOffQ + hq * 128;
    *reinterpret_cast<uint4 *>(row + (((2 * part) ^ (hq & 7)) << 4)) = qa0;
    *reinterpret_cast<uint4 *>(row + (((2 * part + 1) ^ (hq & 7)) << 4)) = qa1;
  }
  {
    uint4 w[4];
    if (!win) {
      const float fa = e4m3_to_float(s2 & 0xFF) * 0x1p112f;
      const float fb = e4m3_to_float(s2 >> 8) * 0x1p112f;
      const uint32_t sa = pack_bf16x2(fa, fa), sb2 = pack_bf16x2(fb, fb);
      const uint32_t cw[4] = {rc0.x, rc0.y, rc0.z, rc0.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t sc = u < 2 ? sa : sb2;
        w[u].x = bf16x2_mul(e2m1x2_bf16x2_m112(cw[u] & 0xFF), sc);
        w[u].y = bf16x2_mul(e2m1x2_bf16x2_m112((cw[u] >> 8) & 0xFF), sc);
        w[u].z = bf16x2_mul(e2m1x2_bf16x2_m112((cw[u] >> 16) & 0xFF), sc);
        w[u].w = bf16x2_mul(e2m1x2_bf16x2_m112(cw[u] >> 24), sc);
      }
    } else {
      const uint32_t by[8] = {rc0.x, rc0.y, rc0.z, rc0.w, rc1.x, rc1.y, rc1.z, rc1.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        w[u].x = e4m3x2_to_bf16x2(by[2 * u] & 0xFFFF);
        w[u].y = e4m3x2_to_bf16x2(by[2 * u] >> 16);
        w[u].z = e4m3x2_to_bf16x2(by[2 * u + 1] & 0xFFFF);
        w[u].w = e4m3x2_to_bf16x2(by[2 * u + 1] >> 16);
      }
    }
    if (hf == 0) ms.slot_ok[j] = valid;
    uint8_t *krow = sm + kClOffK + j * 128;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      *reinterpret_cast<uint4 *>(krow + (((4 * hf + u) ^ (j & 7)) << 4)) = w[u];
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;  // S_r: columns 0..127; O_r: 128..191
  pdl_trigger();

  // ---- 2. S_r = Q_r Khat_r^T
  const uint32_t qa = smem_u32(sm + kClOffQ), ka = smem_u32(sm + kClOffK);
  if (tid == 0) {
    tc_fence_after();
    constexpr uint32_t idesc_s = idesc_f32acc(1, 1, 128, kClRows);  // bf16, both K-major
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma_f16(tmem, desc_k128_sw128(qa + 32 * ks), desc_k128_sw128(ka + 32 * ks), idesc_s,
              ks != 0);
    mma_commit(&ms.bar_s);
  }
  // S_r -> 8 slices of 16 rows (cl_sidx layout): warps 0, 1, 4, 5 (TMEM lanes 0..63 = heads),
  // 64 columns each
  const int quarter = warp & 3, c2 = warp >> 2;
  float4 *sb = reinterpret_cast<float4 *>(sm + kClOffSB);
  constexpr int kSliceF4 = kClSlice / 16;
  if (quarter < 2) {
    ok = __all_sync(0xffffffffu, mbar_wait(&ms.bar_s, 0)) && ok;
    tc_fence_after();
    const int h = quarter * 32 + lane;
    const uint32_t ta = tmem + 64 * c2 + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 32) {
      uint32_t r0[16], r1[16];
      tmem_ld16(ta + c0, r0);
      tmem_ld16(ta + c0 + 16, r1);
      tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t *v = k < 4 ? r0 + 4 * k : r1 + 4 * (k - 4);
        const int col = 64 * c2 + c0 + 4 * k;  // S column = the tile's row
        sb[(col >> 4) * kSliceF4 + cl_sidx(h, (col >> 2) & 3)] =
            make_float4(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]),
                        __uint_as_float(v[3]));
      }
    }
  }
  fence_async_smem();  // the staged slices are read by bulk copies
  tc_fence_before();
  __syncthreads();
  cluster_wait();  // every peer's barriers are initialised

  // ---- 3. reduce-scatter (slice k of S_r to CTA k), local sums, all-gather of the sums
  if (tid < kClR && tid != (int)r)
    bulk_copy_to_peer(dsmem_map(smem_u32(sm + kClOffRB + r * kClSlice), tid),
                      sm + kClOffSB + tid * kClSlice, kClSlice,
                      dsmem_map(smem_u32(&ms.bar_rs), tid));
  ok = __all_sync(0xffffffffu, mbar_wait(&ms.bar_rs, 0)) && ok;
  {
    const int i = cl_sidx(tid >> 2, tid & 3);
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < kClR; ++k) {  // rank order: the same sum in every run
      const float4 v = k == (int)r ? sb[r * kSliceF4 + i]
                                   : reinterpret_cast<const float4 *>(sm + kClOffRB)[k * kSliceF4 + i];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    sb[r * kSliceF4 + i] = acc;
  }
  fence_async_smem();
  __syncthreads();
  if (tid < kClR && tid != (int)r)
    bulk_copy_to_peer(dsmem_map(smem_u32(sm + kClOffSB + r * kClSlice), tid),
                      sm + kClOffSB + r * kClSlice, kClSlice,
                      dsmem_map(smem_u32(&ms.bar_ag), tid));
  ok = __all_sync(0xffffffffu, mbar_wait(&ms.bar_ag, 0)) && ok;
  // every copy into this CTA has landed (execution order only; matched before the exit)
  cluster_arrive_relaxed();

  // ---- 4. numerators of all 128 rows: thread = (head h, rows 32 rq .. 32 rq + 31)
  const int h = tid >> 2, rq = tid & 3;
  float x[32];
  {
    const float4 *sf4 = reinterpret_cast<const float4 *>(sm + kClOffSB);
#pragma unroll
    for (int k = 0; k < 8; ++k) {  // rows 32 rq + 4 k ..: slice 2 rq + k / 4, float4 k % 4
      const float4 v = sf4[(2 * rq + (k >> 2)) * kSliceF4 + cl_sidx(h, k & 3)];
      x[4 * k] = v.x;
      x[4 * k + 1] = v.y;
      x[4 * k + 2] = v.z;
      x[4 * k + 3] = v.w;
    }
  }
  // validity of rows 32 rq .. + 31 as two 16-byte loads
  const uint4 v0 = *reinterpret_cast<const uint4 *>(&ms.slot_ok[32 * rq]);
  const uint4 v1 = *reinterpret_cast<const uint4 *>(&ms.slot_ok[32 * rq + 16]);
  const uint32_t vw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four independent chains
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    x[i] = ((vw[i >> 2] >> (8 * (i & 3))) & 0xFFu) ? x[i] * scale_log2e : -INFINITY;
    mq[i & 3] = fmaxf(mq[i & 3], x[i]);
  }
  float m = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  const float mm = m == -INFINITY ? 0.0f : m;  // no valid row in the tile: every p is 0
  float lq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int u = 0; u < 4; ++u) {  // K = 32 rq + 8 u .. + 7: one 16-byte unit per plane
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
      const float p0 = cl_ex2(x[8 * u + k] - mm), p1 = cl_ex2(x[8 * u + k + 1] - mm);
      lq[k >> 1] += p0 + p1;
      // hi = p truncated to bf16 (its upper 16 bits), lo = p - hi (exact in fp32) truncated:
      // |p - hi - lo| < 2^-14 p, with byte permutes instead of conversions
      const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
      hi[k / 2] = __byte_perm(u0, u1, 0x7632);
      lo[k / 2] = __byte_perm(__float_as_uint(p0 - __uint_as_float(u0 & 0xFFFF0000u)),
                              __float_as_uint(p1 - __uint_as_float(u1 & 0xFFFF0000u)), 0x7632);
    }
#pragma unroll
    for (int pl = 0; pl < 2; ++pl) {
      const int mr = cl_mrow(h, pl);
      uint8_t *dst = sm + kClOffP + (rq >> 1) * kClPChunk + mr * 128 +
                     (((4 * (rq & 1) + u) ^ (mr & 7)) << 4);
      *reinterpret_cast<uint4 *>(dst) = pl == 0 ? make_uint4(hi[0], hi[1], hi[2], hi[3])
                                                : make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
  float l = (lq[0] + lq[1]) + (lq[2] + lq[3]);
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();

  // ---- 5. O_r = [P_hi; P_lo] Vhat_r
  if (tid == 0) {
    tc_fence_after();
    const uint32_t pa = smem_u32(sm + kClOffP);
    constexpr uint32_t idesc_o = idesc_f32acc(1, 1, 128, 64) | (1u << 16);  // B MN-major
#pragma unroll
    for (int ks = 0; ks < kClRows / 16; ++ks)
      mma_f16(tmem + 128, desc_k128_sw128(pa + (ks >> 2) * kClPChunk + 32 * (ks & 3)),
              desc_mn_sw128_atoms(ka + ks * 16 * 128, 16 * 1024), idesc_o, ks != 0);
    mma_commit(&ms.bar_o);
  }
  if (r == 0 && rq == 0 && h < H) {
    const int64_t pr = ((int64_t)n * n_tiles + tile) * H + h;
    m_part[pr] = ok ? m : -INFINITY;
    l_part[pr] = ok ? l : 0.0f;
  }
  ok = __all_sync(0xffffffffu, mbar_wait(&ms.bar_o, 0)) && ok;
  tc_fence_after();
  {
    // warp = (lane quarter q4: heads 16 q4 .. + 15, hi in lanes 0..15, lo in 16..31;
    //         column half: channels 64 r + 32 half ..)
    const int q4 = warp & 3, half = warp >> 2;
    uint32_t v0[16], v1[16];
    const uint32_t ta = tmem + 128 + 32 * half + ((uint32_t)(32 * q4) << 16);
    tmem_ld16(ta, v0);
    tmem_ld16(ta + 16, v1);
    tmem_ld_wait();
    const bool lo = lane >= 16;  // hi lanes keep columns 0..15, lo lanes 16..31
    float o[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float send = __uint_as_float(lo ? v0[k] : v1[k]);
      const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
      o[k] = __uint_as_float(lo ? v1[k] : v0[k]) + recv;
    }
    const int ho = 16 * q4 + (lane & 15);
    if (ho < H) {
      float4 *dst = reinterpret_cast<float4 *>(
          o_part + (((int64_t)n * n_tiles + tile) * H + ho) * kD + 64 * r + 32 * half + 16 * lo);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        dst[k] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 256);
  cluster_wait();  // every peer has received this CTA's copies before its shared memory goes
}

bool attn_cluster_preferred(int nq, int n_tiles) {
  // up to two such CTAs per SM of a B300 (148 SMs) in one wave; beyond that the single-CTA
  // tile (fewer instructions in all) wins
  return (int64_t)nq * n_tiles * kClR <= 2 * 148;
}

cudaError_t launch_attn_cluster_tiles(const void *q_bf16, int nq, int H, const uint8_t *codes,
                                      const uint8_t *sf, const int64_t *cu_ctx,
                                      const int32_t *idx, int topk, float scale_log2e,
                                      int n_tiles, int n_sel_tiles, float *o_part, float *m_part,
                                      float *l_part, const uint8_t *swa_kv, int ring, int n_win,
                                      cudaStream_t st) {
  cudaError_t e = set_smem_once(attn_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kClSmem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attn_cluster_kernel, dim3(kClR * n_tiles, nq), dim3(kClThreads),
                 (size_t)kClSmem, st, static_cast<const uint16_t *>(q_bf16), H, codes, sf, cu_ctx,
                 idx, topk, scale_log2e, n_tiles, n_sel_tiles, o_part, m_part, l_part, swa_kv,
                 ring, n_win);
  note_launches(1);
  return e;
}

}  // namespace csa2

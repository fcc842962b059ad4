/*
 * csa2_oracle.c -- plain, slow, single-threaded CPU statement of the CSA2 hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU-baseline leg of
 * bench.py may load this library.  It shares no code, header, table or helper with the CUDA
 * library; neither includes nor links the other.
 *
 * Sources (the method is described in prose only; no formula or listing is printed there):
 *   [MC]   "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (Hugging Face model
 *          card), Introduction, paragraph "Compressed Sparse Attention 2 (CSA2)": three static
 *          modes Full / Reindex / Reuse; Hierarchical Sparse Indexer with a candidate pool built
 *          by the first Full layer; FP4 main KV = E2M1 values with one E4M3 scale per 16 channels.
 *   [WIKI] "DeepSeek V4.1-Flash" (aiwiki.ai), section "Compressed Sparse Attention 2": what each
 *          mode recomputes; the first Full layer scores all causally visible positions, selects
 *          blocks by their maximum index score, pool = 2,048 blocks of 8 positions; Reindex
 *          layers search that pool and select 512 positions; every layer also has its own local
 *          sliding-window keys and values.  Section "KV-cache formats and bounded replay": main
 *          global KV stored in FP4, local sliding-window KV in FP8.
 *   [SPEC] readings taken where the pages are silent (rounding rules, score formula, tie rule,
 *          softmax scale, packing); each is stated beside the function that uses it.
 *
 * Pins: tests/test_oracle_*.py check every function here against facts that do not come from
 * this file (the OCP E2M1/E4M3 format definitions, torch's float8/bf16 converters, exact
 * rational arithmetic, brute force, dense attention from torch).  Functions without a pin say
 * "parity unpinned" below; there are none at present.
 *
 * Floating point: build without -ffast-math and with -ffp-contract=off, so every float
 * operation is the correctly rounded IEEE operation it is written as.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------------ */
/* Number formats                                                                              */
/* ------------------------------------------------------------------------------------------ */

/* E2M1 ("FP4", [MC] Introduction): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no
 * inf/NaN.  Code layout sign<<3 | exp<<1 | man.  exp == 0 is subnormal: man * 0.5. */
double orc_e2m1_value(int code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : (1.0 + 0.5 * m) * ldexp(1.0, e - 1);
    return s ? -mag : mag;
}

/* E4M3 ("fn" variant; the scale format of [MC] Introduction): 1 sign, 4 exponent bits (bias 7),
 * 3 mantissa bits, no inf, S.1111.111 is NaN; exp == 0 is subnormal man * 2^-9. */
double orc_e4m3_value(int code)
{
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m, -9);
    else mag = (1.0 + m / 8.0) * ldexp(1.0, e - 7);
    return s ? -mag : mag;
}

/* Nearest representable value among codes [0, n_codes) of a monotone non-negative table, ties
 * to the even code (the code whose mantissa LSB is 0).  Values above the largest finite value
 * land on it: round-to-nearest-even followed by saturation to the largest finite value. */
static int nearest_even_code(double a, double (*value)(int), int n_codes)
{
    if (a >= value(n_codes - 1)) return n_codes - 1; /* saturation */
    int best = 0;
    double bestd = fabs(value(0) - a);
    for (int c = 1; c < n_codes; ++c) {
        double d = fabs(value(c) - a);
        if (d < bestd || (d == bestd && (c & 1) == 0)) { best = c; bestd = d; }
    }
    return best;
}

/* [SPEC] E2M1 encode: round to nearest, ties to even, saturate at 6, keep the sign bit (so a
 * negative value that rounds to zero is code 0x8). */
int orc_e2m1_encode(float v)
{
    int mag = nearest_even_code(fabs((double)v), orc_e2m1_value, 8);
    return (signbit(v) ? 8 : 0) | mag;
}

/* [SPEC] E4M3 encode of a non-negative value (scales are never negative): round to nearest,
 * ties to even, saturate at 448.  Codes 0..126 are the finite non-negative values. */
int orc_e4m3_encode(float v)
{
    return nearest_even_code((double)v, orc_e4m3_value, 127);
}

float orc_bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a double to bf16 (8 significant bits), to nearest, ties to even, in one step (no
 * intermediate float, so no double rounding).  Normal range only up to the bf16 maximum;
 * results that would overflow become +-inf. */
uint16_t orc_double_to_bf16(double x)
{
    double r;
    if (x == 0.0 || isnan(x) || isinf(x)) {
        float f = (float)x;
        uint32_t u;
        memcpy(&u, &f, 4);
        return (uint16_t)(u >> 16);
    }
    int e;
    double fr = frexp(fabs(x), &e); /* |x| = fr * 2^e, fr in [0.5, 1) */
    if (e - 1 >= -126) {
        r = ldexp(nearbyint(ldexp(fr, 8)), e - 8); /* 8 significant bits */
    } else {
        r = ldexp(nearbyint(ldexp(fabs(x), 133)), -133); /* subnormal quantum 2^-133 */
    }
    if (r > 3.3895313892515355e38) r = INFINITY;
    float f = (float)(x < 0 ? -r : r);
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------------------------ */
/* a1: FP4 main-KV quantisation ([MC] Introduction: E2M1 values, one E4M3 scale per 16 channels) */
/* ------------------------------------------------------------------------------------------ */

/* [SPEC] for each row and each group g of 16 consecutive channels:
 *   amax  = max |x_i| over the group (bf16 -> fp32 is exact)
 *   scode = E4M3_encode(fp32(amax / 6))            (6 = largest E2M1 magnitude)
 *   sd    = value(scode)
 *   code_i = 0 if sd == 0, else E2M1_encode(fp32(x_i / sd))
 * Packing: codes byte j of a row holds channel 2j in the low nibble and channel 2j+1 in the
 * high nibble (d/2 bytes per row); sf byte g holds the scale of channels 16g..16g+15 (d/16
 * bytes per row). */
void orc_kv_quant_fp4(const uint16_t *x, int64_t n_rows, int d, uint8_t *codes, uint8_t *sf)
{
    for (int64_t r = 0; r < n_rows; ++r) {
        const uint16_t *row = x + r * d;
        for (int g = 0; g < d / 16; ++g) {
            float amax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float a = fabsf(orc_bf16_to_float(row[16 * g + i]));
                if (a > amax) amax = a;
            }
            float s = amax / 6.0f;
            int scode = orc_e4m3_encode(s);
            float sd = (float)orc_e4m3_value(scode);
            sf[r * (d / 16) + g] = (uint8_t)scode;
            for (int i = 0; i < 16; ++i) {
                int c = 16 * g + i;
                int code = 0;
                if (sd != 0.0f) code = orc_e2m1_encode(orc_bf16_to_float(row[c]) / sd);
                uint8_t *byte = &codes[r * (d / 2) + c / 2];
                if (c % 2 == 0) *byte = (uint8_t)((*byte & 0xF0) | code);
                else *byte = (uint8_t)((*byte & 0x0F) | (code << 4));
            }
        }
    }
}

/* Dequantised value of channel c of one packed row: value(code) * value(scale).  The product
 * has at most 6 significant bits and is exact in double (and in fp32, bf16 and fp16). */
static double dequant_elem(const uint8_t *codes_row, const uint8_t *sf_row, int c)
{
    int byte = codes_row[c / 2];
    int code = (c % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    return orc_e2m1_value(code) * orc_e4m3_value(sf_row[c / 16]);
}

void orc_kv_dequant_fp4(const uint8_t *codes, const uint8_t *sf, int64_t n_rows, int d,
                        double *out)
{
    for (int64_t r = 0; r < n_rows; ++r)
        for (int c = 0; c < d; ++c)
            out[r * d + c] = dequant_elem(codes + r * (d / 2), sf + r * (d / 16), c);
}

/* ------------------------------------------------------------------------------------------ */
/* a2 / a5: indexer score ([WIKI] CSA2: the indexer has its own keys and queries; [SPEC] form) */
/* ------------------------------------------------------------------------------------------ */

/* dtype 0 = bf16 (2 bytes/element), 1 = E4M3 (1 byte/element). */
static double elem(const void *base, int dtype, int64_t i)
{
    if (dtype == 0) return (double)orc_bf16_to_float(((const uint16_t *)base)[i]);
    return orc_e4m3_value(((const uint8_t *)base)[i]);
}

/* [SPEC] score(t) = fp32( sum_h w_h * max(0, kscale_t * sum_c q[h,c] * k[t,c]) ), evaluated in
 * double.  With E4M3 inputs every product is a multiple of 2^-18 below 2^18, so the 128-term
 * dot product is exact in double.  q: [Hi, Di], w: [Hi], k: rows of Di elements.
 * Scores are written for positions pos[0..n) (sequence-local row numbers into k). */
void orc_index_scores(const void *q, int dtype, const float *w, int Hi, int Di, const void *k,
                      const float *k_scale, const int64_t *pos, int64_t n, float *out)
{
    double *qd = (double *)malloc(sizeof(double) * (size_t)Hi * Di);
    double *kd = (double *)malloc(sizeof(double) * (size_t)Di);
    for (int64_t i = 0; i < (int64_t)Hi * Di; ++i) qd[i] = elem(q, dtype, i);
    for (int64_t j = 0; j < n; ++j) {
        int64_t t = pos[j];
        for (int c = 0; c < Di; ++c) kd[c] = elem(k, dtype, t * Di + c);
        double score = 0.0;
        for (int h = 0; h < Hi; ++h) {
            double dot = 0.0;
            for (int c = 0; c < Di; ++c) dot += qd[(size_t)h * Di + c] * kd[c];
            if (k_scale) dot *= (double)k_scale[t];
            score += (double)w[h] * (dot > 0.0 ? dot : 0.0);
        }
        out[j] = (float)score;
    }
    free(qd);
    free(kd);
}

/* ------------------------------------------------------------------------------------------ */
/* a3 / a4: Top-K and block selection                                                          */
/* ------------------------------------------------------------------------------------------ */

typedef struct { float score; int64_t pos; } cand_t;

/* [SPEC] order: larger score first; equal scores (including -0 == +0) -> lower position first. */
static int cand_cmp(const void *a, const void *b)
{
    const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->pos < y->pos) ? -1 : (x->pos > y->pos);
}

static int pos_cmp(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* Top-K of n candidates (score, position): sort by the order above, keep the first min(K, n),
 * write their positions in ascending order, pad with -1 up to K.  Returns the count kept. */
int orc_topk(const float *scores, const int64_t *pos, int64_t n, int K, int32_t *out)
{
    cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (n > 0 ? n : 1));
    for (int64_t i = 0; i < n; ++i) { c[i].score = scores[i]; c[i].pos = pos[i]; }
    qsort(c, (size_t)n, sizeof(cand_t), cand_cmp);
    int kept = (int)(n < K ? n : K);
    for (int i = 0; i < kept; ++i) out[i] = (int32_t)c[i].pos;
    qsort(out, (size_t)kept, sizeof(int32_t), pos_cmp);
    for (int i = kept; i < K; ++i) out[i] = -1;
    free(c);
    return kept;
}

/* [WIKI] CSA2: blocks are ranked by the largest index score inside them.  Block b covers positions
 * [bs*b, bs*b+bs) intersected with [0, n); bm_b is the largest score in it. */
void orc_block_max(const float *scores, int64_t n, int bs, float *bm)
{
    int64_t nb = (n + bs - 1) / bs;
    for (int64_t b = 0; b < nb; ++b) {
        float m = scores[b * bs];
        for (int64_t t = b * bs + 1; t < b * bs + bs && t < n; ++t)
            if (scores[t] > m) m = scores[t];
        bm[b] = m;
    }
}

/* [WIKI] CSA2: the candidate pool is the n_pool blocks with the largest block maximum (2,048 in
 * the released configuration), ties to the lower block id; block ids ascending, -1 padded. */
int orc_candidate_pool(const float *bm, int64_t n_blocks, int n_pool, int32_t *out)
{
    int64_t *ids = (int64_t *)malloc(sizeof(int64_t) * (n_blocks > 0 ? n_blocks : 1));
    for (int64_t b = 0; b < n_blocks; ++b) ids[b] = b;
    int kept = orc_topk(bm, ids, n_blocks, n_pool, out);
    free(ids);
    return kept;
}

/* ------------------------------------------------------------------------------------------ */
/* a7 / a8: sparse attention over the selected FP4 rows                                        */
/* ------------------------------------------------------------------------------------------ */

/* [SPEC] For each head h (q: [H, d] in double):
 *   s_j   = scale * sum_c q[h,c] * khat[idx_j, c]       over slots j with idx_j >= 0
 *   out_h = sum_j exp(s_j - m) * khat[idx_j] / sum_j exp(s_j - m),  m = max_j s_j
 *   lse_h = m + log(sum_j exp(s_j - m))
 * K = V = the dequantised latent row.  No valid slot: out = 0, lse = -inf.
 * codes/sf point at row 0 of the sequence; idx are sequence-local row numbers. */
void orc_sparse_attn(const double *q, int H, int d, const uint8_t *codes, const uint8_t *sf,
                     const int32_t *idx, int K, double scale, double *out, double *lse)
{
    int nv = 0;
    for (int j = 0; j < K; ++j) nv += idx[j] >= 0;
    double *rows = (double *)malloc(sizeof(double) * (size_t)(nv > 0 ? nv : 1) * d);
    double *s = (double *)malloc(sizeof(double) * (nv > 0 ? nv : 1));
    int v = 0;
    for (int j = 0; j < K; ++j) {
        if (idx[j] < 0) continue;
        orc_kv_dequant_fp4(codes + (int64_t)idx[j] * (d / 2), sf + (int64_t)idx[j] * (d / 16), 1,
                           d, rows + (size_t)v * d);
        ++v;
    }
    for (int h = 0; h < H; ++h) {
        double *o = out + (size_t)h * d;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        if (nv == 0) { lse[h] = -INFINITY; continue; }
        double m = -INFINITY;
        for (int j = 0; j < nv; ++j) {
            double dot = 0.0;
            for (int c = 0; c < d; ++c) dot += q[(size_t)h * d + c] * rows[(size_t)j * d + c];
            s[j] = scale * dot;
            if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (int j = 0; j < nv; ++j) {
            double p = exp(s[j] - m);
            l += p;
            for (int c = 0; c < d; ++c) o[c] += p * rows[(size_t)j * d + c];
        }
        for (int c = 0; c < d; ++c) o[c] /= l;
        lse[h] = m + log(l);
    }
    free(rows);
    free(s);
}

/* Helpers for callers: bf16 array -> double array; double array -> bf16 (RNE). */
void orc_bf16_to_double(const uint16_t *x, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (double)orc_bf16_to_float(x[i]);
}

void orc_double_to_bf16_array(const double *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_double_to_bf16(x[i]);
}

/* ------------------------------------------------------------------------------------------ */
/* f1: the local sliding-window branch ([WIKI] "Compressed Sparse Attention 2": every CSA2     */
/* layer creates its own local sliding-window keys and values; "KV-cache formats and bounded  */
/* replay": the local sliding-window KV is stored in FP8)                                      */
/* ------------------------------------------------------------------------------------------ */

/* [SPEC] local KV encoding: each bf16 element -> E4M3 "fn" (round to nearest, ties to even,
 * saturating at +-448, sign kept), no scale. */
void orc_fp8_quant(const uint16_t *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) {
        float v = orc_bf16_to_float(x[i]);
        int mag = orc_e4m3_encode(fabsf(v));
        out[i] = (uint8_t)((signbit(v) ? 0x80 : 0) | mag);
    }
}

/* [SPEC] one softmax over the union of the selected global rows (dequantised FP4, as
 * orc_sparse_attn) and n_loc local rows (E4M3, decoded exactly); K = V = each row.  For each
 * head h:  s = scale * <q_h, row> over every row of the union,
 *   out_h = sum softmax(s) * row,   lse_h = log sum exp(s)   (no row: out 0, lse -inf). */
void orc_sparse_swa_attn(const double *q, int H, int d, const uint8_t *codes, const uint8_t *sf,
                         const int32_t *idx, int K, const uint8_t *loc, int n_loc, double scale,
                         double *out, double *lse)
{
    int nv = 0;
    for (int j = 0; j < K; ++j) nv += idx[j] >= 0;
    int n = nv + n_loc;
    double *rows = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * d);
    double *s = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
    int v = 0;
    for (int j = 0; j < K; ++j) {
        if (idx[j] < 0) continue;
        orc_kv_dequant_fp4(codes + (int64_t)idx[j] * (d / 2), sf + (int64_t)idx[j] * (d / 16), 1,
                           d, rows + (size_t)v * d);
        ++v;
    }
    for (int j = 0; j < n_loc; ++j, ++v)
        for (int c = 0; c < d; ++c) rows[(size_t)v * d + c] = orc_e4m3_value(loc[(size_t)j * d + c]);
    for (int h = 0; h < H; ++h) {
        double *o = out + (size_t)h * d;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        if (n == 0) { lse[h] = -INFINITY; continue; }
        double m = -INFINITY;
        for (int j = 0; j < n; ++j) {
            double dot = 0.0;
            for (int c = 0; c < d; ++c) dot += q[(size_t)h * d + c] * rows[(size_t)j * d + c];
            s[j] = scale * dot;
            if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (int j = 0; j < n; ++j) {
            double p = exp(s[j] - m);
            l += p;
            for (int c = 0; c < d; ++c) o[c] += p * rows[(size_t)j * d + c];
        }
        for (int c = 0; c < d; ++c) o[c] /= l;
        lse[h] = m + log(l);
    }
    free(rows);
    free(s);
}

/* ------------------------------------------------------------------------------------------ */
/* f3: index keys derived from main-KV entries ([WIKI] "Compressed Sparse Attention 2": CSA2    */
/* derives index keys from main KV entries rather than through a separate hidden-state path)   */
/* ------------------------------------------------------------------------------------------ */

/* [SPEC] for each cached row t: x = the dequantised FP4 row (d channels), W the layer's index-key
 * projection [Di, d] (bf16):
 *   y_i   = fp32( sum_c W[i,c] * x[c] )     (exact in double: at most 8 x 6 significant bits per
 *                                            product, then one rounding to fp32)
 *   s     = fp32( max_i |y_i| / 448 )       (448 = largest E4M3 value; s = 1 if every y_i is 0)
 *   key_i = E4M3( fp32(y_i / s) )           (round to nearest even, saturating, sign kept)
 * keys [n, Di] E4M3 and k_scale [n] = s are the indexer's k_idx and k_scale: the score uses
 * s * <q_h, key>. */
void orc_index_keys_from_kv(const uint8_t *codes, const uint8_t *sf, int64_t n_rows, int d,
                            const uint16_t *W, int Di, uint8_t *keys, float *k_scale)
{
    double *x = (double *)malloc(sizeof(double) * (size_t)d);
    float *y = (float *)malloc(sizeof(float) * (size_t)Di);
    for (int64_t r = 0; r < n_rows; ++r) {
        orc_kv_dequant_fp4(codes + r * (d / 2), sf + r * (d / 16), 1, d, x);
        float amax = 0.0f;
        for (int i = 0; i < Di; ++i) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += (double)orc_bf16_to_float(W[(size_t)i * d + c]) * x[c];
            y[i] = (float)acc;
            if (fabsf(y[i]) > amax) amax = fabsf(y[i]);
        }
        float s = amax > 0.0f ? amax / 448.0f : 1.0f;
        k_scale[r] = s;
        for (int i = 0; i < Di; ++i) {
            float v = y[i] / s;
            keys[r * Di + i] = (uint8_t)((signbit(v) ? 0x80 : 0) | orc_e4m3_encode(fabsf(v)));
        }
    }
    free(x);
    free(y);
}

/* ------------------------------------------------------------------------------------------ */
/* f4: the full-FP4 PV variant of prefill attention (the workload asks for the PV product as a */
/* block-scaled FP4 contraction too)                                                           */
/* ------------------------------------------------------------------------------------------ */

/* [SPEC] block-scaled FP4 value of x within a block whose largest magnitude is amax, with the
 * main-KV rule: sc = E4M3(fp32(amax / 6)), value = E2M1(fp32(x / sc)) * sc (0 if sc == 0). */
static double fp4_block_value(float x, float amax)
{
    int scode = orc_e4m3_encode(amax / 6.0f);
    float sc = (float)orc_e4m3_value(scode);
    if (sc == 0.0f) return 0.0;
    return orc_e2m1_value(orc_e2m1_encode(x / sc)) * (double)sc;
}

/* [SPEC] For one query token (q = its FP4-dequantised query [H, d]) and its K selected slots
 * (idx[j] < 0: an empty slot, a zero row that takes part in the blocks):
 *   s_j = scale * <q_h, khat_j>;  m_h = max over valid slots;  p_j = fp32(exp(s_j - m_h)) (0 for
 *   empty slots);
 *   P: slots in blocks of 16 consecutive slots; per (head, block) Pt_j = fp4_block_value(p_j,
 *      max_block p);
 *   V: per (channel c, block) Vt_jc = fp4_block_value(khat_jc, max_block |khat_.c|);
 *   out_hc = sum_j Pt_j Vt_jc / sum_j Pt_j;   lse_h = m_h + log(sum_j Pt_j)
 * (no valid slot: out 0, lse -inf). */
void orc_attn_fp4pv(const double *q, int H, int d, const uint8_t *codes, const uint8_t *sf,
                    const int32_t *idx, int K, double scale, double *out, double *lse)
{
    int nb = (K + 15) / 16;
    int kp = nb * 16;
    double *rows = (double *)calloc((size_t)kp * d, sizeof(double));
    double *vt = (double *)calloc((size_t)kp * d, sizeof(double));
    double *s = (double *)malloc(sizeof(double) * kp);
    float *p = (float *)malloc(sizeof(float) * kp);
    double *pt = (double *)malloc(sizeof(double) * kp);
    int nv = 0;
    for (int j = 0; j < K; ++j) {
        if (idx[j] < 0) continue;
        ++nv;
        orc_kv_dequant_fp4(codes + (int64_t)idx[j] * (d / 2), sf + (int64_t)idx[j] * (d / 16), 1,
                           d, rows + (size_t)j * d);
    }
    for (int b = 0; b < nb; ++b)
        for (int c = 0; c < d; ++c) {
            float amax = 0.0f;
            for (int j = 16 * b; j < 16 * b + 16; ++j) {
                float a = fabsf((float)rows[(size_t)j * d + c]);
                if (a > amax) amax = a;
            }
            for (int j = 16 * b; j < 16 * b + 16; ++j)
                vt[(size_t)j * d + c] = fp4_block_value((float)rows[(size_t)j * d + c], amax);
        }
    for (int h = 0; h < H; ++h) {
        double *o = out + (size_t)h * d;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        if (nv == 0) { lse[h] = -INFINITY; continue; }
        double m = -INFINITY;
        for (int j = 0; j < kp; ++j) {
            s[j] = -INFINITY;
            if (j >= K || idx[j] < 0) continue;
            double dot = 0.0;
            for (int c = 0; c < d; ++c) dot += q[(size_t)h * d + c] * rows[(size_t)j * d + c];
            s[j] = scale * dot;
            if (s[j] > m) m = s[j];
        }
        for (int j = 0; j < kp; ++j) p[j] = (s[j] == -INFINITY) ? 0.0f : (float)exp(s[j] - m);
        double l = 0.0;
        for (int b = 0; b < nb; ++b) {
            float amax = 0.0f;
            for (int j = 16 * b; j < 16 * b + 16; ++j)
                if (p[j] > amax) amax = p[j];
            for (int j = 16 * b; j < 16 * b + 16; ++j) {
                pt[j] = fp4_block_value(p[j], amax);
                l += pt[j];
            }
        }
        for (int j = 0; j < kp; ++j)
            if (pt[j] != 0.0)
                for (int c = 0; c < d; ++c) o[c] += pt[j] * vt[(size_t)j * d + c];
        if (l > 0.0) {
            for (int c = 0; c < d; ++c) o[c] /= l;
            lse[h] = m + log(l);
        } else {
            lse[h] = -INFINITY;
        }
    }
    free(rows);
    free(vt);
    free(s);
    free(p);
    free(pt);
}

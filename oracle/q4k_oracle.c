/*
 * q4k_oracle.c -- CPU oracle for the Q4_K mixture-of-experts id-GEMV layer.
 *
 * TEST INFRASTRUCTURE: see q4k_oracle.h. Plain loops, fp64 accumulation,
 * no SIMD intrinsics, no blocking or reordering beyond the definitions.
 * Build with -ffp-contract=off so that the quantizer's binary32 steps are the
 * same single roundings on every host (aarch64 compilers contract a*b+c into
 * one fused operation otherwise).
 */
#include "q4k_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- IEEE binary16 ----------------------------------------------------------- */

float q4o_half_to_float(uint16_t h) {
    /* value = (-1)^s * 2^(e-15) * (1 + f/1024) for 0 < e < 31, (-1)^s * 2^-14 * f/1024 for e == 0 */
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);
    }
    return (float)(s ? -v : v);
}

uint16_t q4o_float_to_half_rne(float f) {
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    uint32_t sign = (x >> 16) & 0x8000u;
    int exp32 = (int)((x >> 23) & 0xFFu);
    uint32_t man = x & 0x7FFFFFu;
    if (exp32 == 0xFF) /* inf or nan */
        return (uint16_t)(sign | 0x7C00u | (man ? 0x200u : 0u));
    int e = exp32 - 127 + 15; /* biased binary16 exponent */
    if (e >= 31) return (uint16_t)(sign | 0x7C00u);
    if (e >= 1) {
        /* normal: keep 10 of 23 fraction bits, round the dropped 13 to nearest even;
         * a carry out of the fraction bumps the exponent (up to infinity) */
        uint32_t h = ((uint32_t)e << 10) | (man >> 13);
        uint32_t rem = man & 0x1FFFu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;
        return (uint16_t)(sign | h);
    }
    /* subnormal result: units of 2^-24. value = M * 2^(exp32-150) with M the
     * 24-bit significand, so the count of units is M >> (126 - exp32). */
    int shift = 126 - exp32;
    if (shift > 24) return (uint16_t)sign;
    uint32_t M = man | 0x800000u;
    uint32_t q = M >> shift;
    uint32_t rem = M & ((1u << shift) - 1u);
    uint32_t halfway = 1u << (shift - 1);
    if (rem > halfway || (rem == halfway && (q & 1u))) q += 1u;
    return (uint16_t)(sign | q);
}

void q4o_half_to_float_n(const uint16_t* h, float* f, int64_t n) {
    for (int64_t i = 0; i < n; ++i) f[i] = q4o_half_to_float(h[i]);
}

void q4o_float_to_half_rne_n(const float* f, uint16_t* h, int64_t n) {
    for (int64_t i = 0; i < n; ++i) h[i] = q4o_float_to_half_rne(f[i]);
}

/* ---- Q4_K decode --------------------------------------------------------------- */

static uint16_t load_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

void q4o_block_scale_min(const uint8_t* block, int j, int* sc, int* mn) {
    const uint8_t* s = block + 4; /* the 12 scale bytes */
    if (j < 4) {
        *sc = s[j] & 63;
        *mn = s[j + 4] & 63;
    } else {
        /* low four bits in byte j+4 (scale: low nibble, min: high nibble);
         * high two bits are the top bits of bytes j-4 (scale) and j (min) */
        *sc = (s[j + 4] & 0x0F) | ((s[j - 4] >> 6) << 4);
        *mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

void q4o_dequant_block(const uint8_t* block, float* w256) {
    const float d = q4o_half_to_float(load_u16(block));
    const float dmin = q4o_half_to_float(load_u16(block + 2));
    const uint8_t* qs = block + 16;
    for (int c = 0; c < 4; ++c) {          /* 64-weight groups */
        for (int half = 0; half < 2; ++half) { /* low nibble: sub-block 2c, high: 2c+1 */
            int j = 2 * c + half;
            int sc, mn;
            q4o_block_scale_min(block, j, &sc, &mn);
            float ds = d * (float)sc;
            float dm = dmin * (float)mn;
            for (int i = 0; i < 32; ++i) {
                int q = half ? (qs[32 * c + i] >> 4) : (qs[32 * c + i] & 0x0F);
                w256[64 * c + 32 * half + i] = ds * (float)q - dm;
            }
        }
    }
}

/* little-endian bit string: bit b of the row is bit (b % 8) of byte b / 8 */
static unsigned row_bits(const uint8_t* bytes, int64_t start, int len) {
    unsigned v = 0;
    for (int b = 0; b < len; ++b) {
        int64_t pos = start + b;
        v |= (unsigned)((bytes[pos >> 3] >> (pos & 7)) & 1) << b;
    }
    return v;
}

float q4o_weight_at(const uint8_t* row, int64_t k) {
    const int64_t blk = k / Q4O_QK;
    const int e = (int)(k % Q4O_QK);
    const int64_t base = blk * Q4O_BLOCK_BYTES * 8; /* bit offset of the block */
    /* fields: d at bit 0, dmin at bit 16, scale bytes from bit 32, codes from bit 128 */
    const float d = q4o_half_to_float((uint16_t)row_bits(row, base + 0, 16));
    const float dmin = q4o_half_to_float((uint16_t)row_bits(row, base + 16, 16));
    const int grp = e / 64, r = e % 64;
    const int code_byte = 32 * grp + (r % 32);
    const int q = (int)row_bits(row, base + 128 + 8 * code_byte + (r >= 32 ? 4 : 0), 4);
    const int j = e / 32;
    unsigned sc, mn;
    if (j < 4) {
        sc = row_bits(row, base + 32 + 8 * j, 6);
        mn = row_bits(row, base + 32 + 8 * (j + 4), 6);
    } else {
        sc = row_bits(row, base + 32 + 8 * (j + 4), 4) | (row_bits(row, base + 32 + 8 * (j - 4) + 6, 2) << 4);
        mn = row_bits(row, base + 32 + 8 * (j + 4) + 4, 4) | (row_bits(row, base + 32 + 8 * j + 6, 2) << 4);
    }
    float ds = d * (float)sc;
    float dm = dmin * (float)mn;
    return ds * (float)q - dm;
}

void q4o_dequant_rows(const uint8_t* w, int64_t rows, int64_t k, float* out, int elementwise) {
    const int64_t nb = k / Q4O_QK;
    const int64_t row_bytes = nb * Q4O_BLOCK_BYTES;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const uint8_t* row = w + r * row_bytes;
        if (elementwise) {
            for (int64_t c = 0; c < k; ++c) out[r * k + c] = q4o_weight_at(row, c);
        } else {
            for (int64_t b = 0; b < nb; ++b) q4o_dequant_block(row + b * Q4O_BLOCK_BYTES, out + r * k + b * Q4O_QK);
        }
    }
}

/* ---- quantizer ------------------------------------------------------------------ */

static void quantize_block(const float* x, uint8_t* out) {
    float scale[8], mnv[8];
    float max_scale = 0.0f, max_mn = 0.0f;
    for (int j = 0; j < 8; ++j) {
        float lo = 0.0f, hi = x[32 * j];
        for (int i = 0; i < 32; ++i) {
            float v = x[32 * j + i];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        scale[j] = (hi - lo) / 15.0f;
        mnv[j] = -lo;
        if (scale[j] > max_scale) max_scale = scale[j];
        if (mnv[j] > max_mn) max_mn = mnv[j];
    }
    uint16_t d16 = q4o_float_to_half_rne(max_scale / 63.0f);
    uint16_t dmin16 = q4o_float_to_half_rne(max_mn / 63.0f);
    float d = q4o_half_to_float(d16), dmin = q4o_half_to_float(dmin16);
    int sc[8], mn[8];
    for (int j = 0; j < 8; ++j) {
        int s = d > 0.0f ? (int)rintf(scale[j] / d) : 0;
        int m = dmin > 0.0f ? (int)rintf(mnv[j] / dmin) : 0;
        sc[j] = s > 63 ? 63 : s;
        mn[j] = m > 63 ? 63 : m;
    }
    memset(out, 0, Q4O_BLOCK_BYTES);
    out[0] = (uint8_t)(d16 & 0xFF);
    out[1] = (uint8_t)(d16 >> 8);
    out[2] = (uint8_t)(dmin16 & 0xFF);
    out[3] = (uint8_t)(dmin16 >> 8);
    uint8_t* s = out + 4;
    for (int j = 0; j < 4; ++j) {
        s[j] = (uint8_t)(sc[j] | ((sc[j + 4] >> 4) << 6));
        s[j + 4] = (uint8_t)(mn[j] | ((mn[j + 4] >> 4) << 6));
        s[j + 8] = (uint8_t)((sc[j + 4] & 0x0F) | ((mn[j + 4] & 0x0F) << 4));
    }
    uint8_t* qs = out + 16;
    for (int j = 0; j < 8; ++j) {
        float ds = d * (float)sc[j];
        float dm = dmin * (float)mn[j];
        for (int i = 0; i < 32; ++i) {
            int q = 0;
            if (ds > 0.0f) {
                float t = (x[32 * j + i] + dm) / ds;
                q = (int)rintf(t);
                q = q < 0 ? 0 : (q > 15 ? 15 : q);
            }
            int c = j / 2, half = j % 2;
            qs[32 * c + i] |= (uint8_t)(q << (4 * half));
        }
    }
}

void q4o_quantize_rows(const float* x, int64_t rows, int64_t k, uint8_t* out) {
    const int64_t nb = k / Q4O_QK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b)
            quantize_block(x + r * k + b * Q4O_QK, out + (r * nb + b) * Q4O_BLOCK_BYTES);
}

/* ---- MoE id-GEMV ---------------------------------------------------------------- */

/* One output: sum over the row's blocks of dequantized weight times activation. */
static double dot_row_f32(const uint8_t* row, const float* x, int k) {
    float w[Q4O_QK];
    double acc = 0.0;
    for (int b = 0; b < k / Q4O_QK; ++b) {
        q4o_dequant_block(row + (int64_t)b * Q4O_BLOCK_BYTES, w);
        for (int i = 0; i < Q4O_QK; ++i) acc += (double)w[i] * (double)x[b * Q4O_QK + i];
    }
    return acc;
}

static double dot_row_f64(const uint8_t* row, const double* x, int k) {
    float w[Q4O_QK];
    double acc = 0.0;
    for (int b = 0; b < k / Q4O_QK; ++b) {
        q4o_dequant_block(row + (int64_t)b * Q4O_BLOCK_BYTES, w);
        for (int i = 0; i < Q4O_QK; ++i) acc += (double)w[i] * x[b * Q4O_QK + i];
    }
    return acc;
}

static int count_invalid(const int32_t* ids, int n_pairs, int num_experts) {
    int bad = 0;
    for (int p = 0; p < n_pairs; ++p) bad += (ids[p] < 0 || ids[p] >= num_experts);
    return bad;
}

int q4o_moe_id_gemv(const uint8_t* w, int num_experts, const float* a, int64_t outer,
                    int64_t inner, const int32_t* ids, int m, int top_k, int n, int k,
                    double* out) {
    const int64_t row_bytes = (int64_t)(k / Q4O_QK) * Q4O_BLOCK_BYTES; /* nb01 */
    const int64_t expert_bytes = (int64_t)n * row_bytes;               /* nb02 */
    const int64_t n_pairs = (int64_t)m * top_k;
#pragma omp parallel for schedule(static)
    for (int64_t idx = 0; idx < n_pairs * n; ++idx) {
        int64_t p = idx / n, r = idx % n;
        int32_t e = ids[p];
        if (e < 0 || e >= num_experts) { out[idx] = 0.0; continue; }
        int64_t t = p / top_k, s = p % top_k;
        const float* x = a + t * outer + s * inner;
        out[idx] = dot_row_f32(w + e * expert_bytes + r * row_bytes, x, k);
    }
    return count_invalid(ids, (int)n_pairs, num_experts);
}

int q4o_moe_id_gemv_f64(const uint8_t* w, int num_experts, const double* a, int64_t outer,
                        int64_t inner, const int32_t* ids, int m, int top_k, int n, int k,
                        double* out) {
    const int64_t row_bytes = (int64_t)(k / Q4O_QK) * Q4O_BLOCK_BYTES;
    const int64_t expert_bytes = (int64_t)n * row_bytes;
    const int64_t n_pairs = (int64_t)m * top_k;
#pragma omp parallel for schedule(static)
    for (int64_t idx = 0; idx < n_pairs * n; ++idx) {
        int64_t p = idx / n, r = idx % n;
        int32_t e = ids[p];
        if (e < 0 || e >= num_experts) { out[idx] = 0.0; continue; }
        int64_t t = p / top_k, s = p % top_k;
        const double* x = a + t * outer + s * inner;
        out[idx] = dot_row_f64(w + e * expert_bytes + r * row_bytes, x, k);
    }
    return count_invalid(ids, (int)n_pairs, num_experts);
}

/* ---- expert FFN --------------------------------------------------------------------- */

double q4o_silu(double x) { return x / (1.0 + exp(-x)); }

int q4o_expert_ffn(const uint8_t* w_gate, const uint8_t* w_up, const uint8_t* w_down,
                   int num_experts, const float* h_post, const int32_t* ids, int m, int top_k,
                   int hidden, int inter, double* expert_out) {
    const int64_t n_pairs = (int64_t)m * top_k;
    double* g = (double*)malloc(sizeof(double) * n_pairs * inter);
    double* u = (double*)malloc(sizeof(double) * n_pairs * inter);
    if (!g || !u) { free(g); free(u); return -1; }
    /* gate and up: every slot of a token reads the token's row (outer = hidden, inner = 0) */
    int bad = q4o_moe_id_gemv(w_gate, num_experts, h_post, hidden, 0, ids, m, top_k, inter, hidden, g);
    q4o_moe_id_gemv(w_up, num_experts, h_post, hidden, 0, ids, m, top_k, inter, hidden, u);
    /* SwiGLU, in place in g: act = silu(g) * u, laid out [m, top_k, inter] */
    for (int64_t i = 0; i < n_pairs * inter; ++i) g[i] = q4o_silu(g[i]) * u[i];
    /* down: each pair reads its own act row (outer = top_k*inter, inner = inter) */
    q4o_moe_id_gemv_f64(w_down, num_experts, g, (int64_t)top_k * inter, inter, ids, m, top_k,
                        hidden, inter, expert_out);
    free(g);
    free(u);
    return bad;
}

/* ---- combine ---------------------------------------------------------------------------- */

void q4o_moe_combine(const double* h_mid, const double* expert_out, const double* weights,
                     const double* shared_out, const double* shared_gate, int shared_mode,
                     int m, int top_k, int hidden, double* y) {
    for (int t = 0; t < m; ++t) {
        double g = 0.0;
        if (shared_mode == 1) g = 1.0 / (1.0 + exp(-shared_gate[t]));
        else if (shared_mode == 2) g = 1.0;
        for (int h = 0; h < hidden; ++h) {
            double acc = h_mid[(int64_t)t * hidden + h];
            for (int s = 0; s < top_k; ++s) {
                int64_t p = (int64_t)t * top_k + s;
                acc += weights[p] * expert_out[p * hidden + h];
            }
            if (shared_mode != 0) acc += g * shared_out[(int64_t)t * hidden + h];
            y[(int64_t)t * hidden + h] = acc;
        }
    }
}

/* ---- whole layer -------------------------------------------------------------------------- */

int q4o_moe_layer(const uint8_t* w_gate, const uint8_t* w_up, const uint8_t* w_down,
                  int num_experts, const uint8_t* ws_gate, const uint8_t* ws_up,
                  const uint8_t* ws_down, int shared_inter, int shared_mode,
                  const float* h_post, const float* h_mid, const int32_t* ids,
                  const float* weights, const float* shared_gate, int m, int top_k,
                  int hidden, int inter, double* y) {
    const int64_t n_pairs = (int64_t)m * top_k;
    const int64_t mh = (int64_t)m * hidden;
    double* eo = (double*)malloc(sizeof(double) * n_pairs * hidden);
    double* so = (double*)calloc((size_t)mh, sizeof(double));
    double* hm = (double*)malloc(sizeof(double) * mh);
    double* wt = (double*)malloc(sizeof(double) * n_pairs);
    double* sg = (double*)calloc((size_t)m, sizeof(double));
    int32_t* zero_ids = (int32_t*)calloc((size_t)m, sizeof(int32_t));
    int bad = -1;
    if (!eo || !so || !hm || !wt || !sg || !zero_ids) goto done;
    bad = q4o_expert_ffn(w_gate, w_up, w_down, num_experts, h_post, ids, m, top_k, hidden, inter, eo);
    if (shared_mode != 0)
        q4o_expert_ffn(ws_gate, ws_up, ws_down, 1, h_post, zero_ids, m, 1, hidden, shared_inter, so);
    for (int64_t i = 0; i < mh; ++i) hm[i] = h_mid[i];
    for (int64_t p = 0; p < n_pairs; ++p) wt[p] = weights[p];
    if (shared_gate)
        for (int t = 0; t < m; ++t) sg[t] = shared_gate[t];
    q4o_moe_combine(hm, eo, wt, so, sg, shared_mode, m, top_k, hidden, y);
done:
    free(eo); free(so); free(hm); free(wt); free(sg); free(zero_ids);
    return bad;
}

/* ---- pair bucketing --------------------------------------------------------------------------- */

int q4o_bucket(const int32_t* ids, int n_pairs, int num_experts, int32_t* counts,
               int32_t* offsets, int32_t* perm) {
    for (int e = 0; e < num_experts; ++e) counts[e] = 0;
    int bad = 0;
    for (int p = 0; p < n_pairs; ++p) {
        if (ids[p] < 0 || ids[p] >= num_experts) ++bad;
        else ++counts[ids[p]];
    }
    offsets[0] = 0;
    for (int e = 0; e < num_experts; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)(num_experts > 0 ? num_experts : 1));
    if (!cursor) return -1;
    for (int e = 0; e < num_experts; ++e) cursor[e] = offsets[e];
    int tail = offsets[num_experts];
    for (int p = 0; p < n_pairs; ++p) { /* increasing p keeps each bucket sorted */
        if (ids[p] < 0 || ids[p] >= num_experts) perm[tail++] = p;
        else perm[cursor[ids[p]]++] = p;
    }
    free(cursor);
    return bad;
}

/* ---- threading --------------------------------------------------------------------------------- */

int q4o_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

int q4o_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

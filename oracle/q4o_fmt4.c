/*
 * q4o_fmt4.c -- CPU oracle for two other 4-bit weight formats run through the same MoE
 * id-GEMV walk as Q4_K. TEST INFRASTRUCTURE, like the rest of this directory.
 *
 * Sources (page titles of the studied material):
 *   [P2] moeflux 0.1.0-pre.3, src/riir/moe/expert_forward.rs -- the MLX-style affine 4-bit
 *        expert blob: `gpu_expert_forward` (an expert is [gate | up | down] blocks, each bound
 *        to the matvec at three offsets: weights, scales, biases), `encode_matvec` (group
 *        size GROUP_SIZE), `synth::expert_data_seeded` (bf16 scales 0x3C00, biases 0).
 *   [P3] cortiq-engine 0.7.7, examples/mv_lab.rs -- the q4tp matrix as its production kernel
 *        `cur` reads it: per row gpr = k/32 groups of 16 bytes (32 codes, nibble - 8), a
 *        half2 (base, step) per row, a 5-bit code per group, group scale exp2(base + code*step).
 * Readings where the pages leave the layout open (stated at each function): the affine value
 * is MLX's w = scale*q + bias with q the unsigned nibble; in both formats the codes of 8
 * consecutive weights fill one little-endian 32-bit word, weight 8j+i in bits 4i..4i+3 of
 * word j (the q4tp kernel's unpacking; for the affine blob the MLX packing); an expert of a
 * stacked slab starts expert_stride bytes after the previous one.
 *
 * All arithmetic is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include "q4k_oracle.h"

/* code of weight c of a row whose codes start at p: nibble c%2 of byte c/2, low nibble first
 * (the same as bits 4*(c%8) of little-endian word c/8) */
static int nibble_at(const uint8_t* p, int64_t c) {
    const uint8_t byte = p[c / 2];
    return (c % 2) ? (byte >> 4) : (byte & 0x0F);
}

static uint16_t u16_at(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* MLX affine 4-bit [n, k], group size gs: codes at mat (row r: k/2 bytes from r*k/2), scales
 * bf16 [n, k/gs] at mat + s_off, biases bf16 [n, k/gs] at mat + b_off.
 *   w[r][c] = scale[r][c/gs] * q[r][c] + bias[r][c/gs]. */
void q4o_affine4_dequant(const uint8_t* mat, uint64_t s_off, uint64_t b_off, int64_t n, int64_t k,
                         int gs, double* out) {
    const int64_t groups = k / gs;
    for (int64_t r = 0; r < n; ++r)
        for (int64_t c = 0; c < k; ++c) {
            const int q = nibble_at(mat + r * (k / 2), c);
            const int64_t g = r * groups + c / gs;
            const double scale = q4o_bf16_to_double(u16_at(mat + s_off + 2 * g));
            const double bias = q4o_bf16_to_double(u16_at(mat + b_off + 2 * g));
            out[r * k + c] = scale * q + bias;
        }
}

/* q4tp [n, k], gpr = k/32: codes of row r group g at mat + (r*gpr + g)*16 (weight 32g + i is
 * nibble i of those 16 bytes); (base, step) binary16 at mat + n*gpr*16 + 4r; 5-bit group codes
 * from mat + n*gpr*16 + 4n, row stride ceil(5*gpr/8) bytes, code of group g in bits
 * 5g .. 5g+4 of the row's bytes read as one little-endian bit string.
 *   w[r][32g + i] = (nibble - 8) * 2^(base + code*step). */
void q4o_q4tp_dequant(const uint8_t* mat, int64_t n, int64_t k, double* out) {
    const int64_t gpr = k / 32;
    const uint8_t* params = mat + n * gpr * 16;
    const uint8_t* codes = params + 4 * n;
    const int64_t cstride = (gpr * 5 + 7) / 8;
    for (int64_t r = 0; r < n; ++r) {
        const double base = (double)q4o_half_to_float(u16_at(params + 4 * r));
        const double step = (double)q4o_half_to_float(u16_at(params + 4 * r + 2));
        for (int64_t g = 0; g < gpr; ++g) {
            int code = 0;
            for (int b = 0; b < 5; ++b) {  /* bit 5g+b of the row's code string */
                const int64_t bit = 5 * g + b;
                code |= ((codes[r * cstride + bit / 8] >> (bit % 8)) & 1) << b;
            }
            const double scale = exp2(base + code * step);
            for (int i = 0; i < 32; ++i)
                out[r * k + 32 * g + i] = (nibble_at(mat + (r * gpr + g) * 16, i) - 8) * scale;
        }
    }
}

/* Bytes of one [n, k] matrix in each format (without the stacking stride). */
uint64_t q4o_fmt4_matrix_bytes(int fmt, int64_t n, int64_t k, int gs) {
    if (fmt == Q4O_FMT_AFFINE) return (uint64_t)(n * k / 2 + 2 * 2 * n * (k / gs));
    return (uint64_t)(n * (k / 32) * 16 + 4 * n + n * (((k / 32) * 5 + 7) / 8));
}

/* The id-GEMV walk of q4o_moe_id_gemv over a slab of either format: expert e's matrix at
 * w + e*expert_stride (affine: scales and biases at s_off / b_off from it). */
int q4o_moe_id_gemv_fmt4(int fmt, const uint8_t* w, uint64_t expert_stride, uint64_t s_off,
                         uint64_t b_off, int gs, int num_experts, const float* a, int64_t outer,
                         int64_t inner, const int32_t* ids, int m, int top_k, int n, int k,
                         double* out) {
    double* dense = (double*)malloc(sizeof(double) * (size_t)n * (size_t)k);
    if (!dense) return -1;
    int bad = 0;
    for (int e = -1; e < num_experts; ++e) {
        /* e = -1: the pairs with an out-of-range id get zero rows */
        int used = 0;
        for (int64_t p = 0; p < (int64_t)m * top_k; ++p) {
            const int valid = ids[p] >= 0 && ids[p] < num_experts;
            if ((e < 0 && valid) || (e >= 0 && ids[p] != e)) continue;
            if (e < 0) {
                ++bad;
                for (int r = 0; r < n; ++r) out[p * n + r] = 0.0;
                continue;
            }
            if (!used) {
                const uint8_t* mat = w + (uint64_t)e * expert_stride;
                if (fmt == Q4O_FMT_AFFINE) q4o_affine4_dequant(mat, s_off, b_off, n, k, gs, dense);
                else q4o_q4tp_dequant(mat, n, k, dense);
                used = 1;
            }
            const float* x = a + (p / top_k) * outer + (p % top_k) * inner;
            for (int r = 0; r < n; ++r) {
                double acc = 0.0;
                for (int c = 0; c < k; ++c) acc += dense[(int64_t)r * k + c] * (double)x[c];
                out[p * n + r] = acc;
            }
        }
    }
    free(dense);
    return bad;
}

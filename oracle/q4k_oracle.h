/*
 * q4k_oracle.h -- CPU oracle for the Q4_K mixture-of-experts id-GEMV layer.
 *
 * TEST INFRASTRUCTURE. This library is the slow, plain reference that the CUDA
 * path is checked against. Only the test suite, the package smoke check and
 * the CPU-baseline / reference leg of the benchmark may load it. It shares no
 * code, header, table or helper with the CUDA library, and neither includes
 * the other.
 *
 * Sources of each definition (page titles of the studied material):
 *   [P1] ferrum-kernels 0.7.7, src/backend/metal/q4_k_moe_id_gemv_batched.rs
 *        -- module doc (the src1 outer/inner stride walk), the doc comment of
 *        `dispatch_gemv_q4k_moe_id_batched_on_encoder` (slab layout
 *        [num_experts, n, k/256], expert stride nb02 = n*(k/256)*144 bytes,
 *        ids flat with pair = token*top_k + slot, out [m*top_k, n]) and the
 *        test module (the batched call equals m per-token calls).
 *   [P2] moeflux 0.1.0-pre.3, src/riir/moe/expert_forward.rs -- module doc
 *        (gate, up, SwiGLU, down), `combine_kernel_name` (sigmoid-gated vs
 *        unscaled shared expert), `encode_moe_combine_residual_n_tokens` doc
 *        (hidden_out = h_mid + moe_sum + sigmoid(gate) * shared_out),
 *        `encode_moe_gather_id_fuse` doc (map0 buckets pairs by expert, then
 *        gate/up with a broadcast row, down with a per-pair row).
 *   [Q4K] The Q4_K super-block: 256 weights in 144 bytes -- fp16 d, fp16
 *        dmin, 12 bytes holding eight 6-bit scales and eight 6-bit mins,
 *        128 bytes of 4-bit codes; w = d*sc*q - dmin*m. The bit placement is
 *        the GGML Q4_K layout that [P1] names through candle's
 *        GgmlDType::Q4K (a reading; the pages do not print it).
 *
 * Conventions: all integers are little-endian; arrays are row-major; sizes in
 * elements unless named *_bytes. Every function is single-call, synchronous,
 * allocates only what it frees before returning, and never touches a GPU.
 */
#ifndef Q4K_ORACLE_H
#define Q4K_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define Q4O_QK 256          /* weights per super-block                    */
#define Q4O_BLOCK_BYTES 144 /* bytes per super-block                      */

/* ---- IEEE binary16 -------------------------------------------------------- */
/* Exact decode of one binary16 value (denormals, inf and NaN included). */
float q4o_half_to_float(uint16_t h);
/* Round-to-nearest-even encode of one binary32 value into binary16. */
uint16_t q4o_float_to_half_rne(float f);
void q4o_half_to_float_n(const uint16_t* h, float* f, int64_t n);
void q4o_float_to_half_rne_n(const float* f, uint16_t* h, int64_t n);

/* ---- Q4_K decode [Q4K] ------------------------------------------------------ */
/* Sub-block j (0..7) scale and min of one 144-byte block, masked-byte form. */
void q4o_block_scale_min(const uint8_t* block, int j, int* sc, int* mn);
/* Block-wise unpacker: 256 weights of one block, w = fp32(fp32(d)*sc)*q - fp32(fp32(dmin)*m). */
void q4o_dequant_block(const uint8_t* block, float* w256);
/* Element-at-a-time unpacker, written independently of the block-wise one:
 * every field is read by absolute bit position in the row's byte string. */
float q4o_weight_at(const uint8_t* row, int64_t k);
/* rows x k weights of a Q4_K matrix (row stride k/256*144 bytes). elementwise!=0
 * selects q4o_weight_at, else the block-wise unpacker. */
void q4o_dequant_rows(const uint8_t* w, int64_t rows, int64_t k, float* out, int elementwise);

/* ---- quantizer (test-data generator) ---------------------------------------- */
/* Per 32-weight sub-block: lo = min(0, min x), hi = max x, scale = (hi-lo)/15,
 * mn = -lo; d = fp16(max scale / 63), dmin = fp16(max mn / 63);
 * sc = min(63, rint(scale/d)), m = min(63, rint(mn/dmin)) (0 when the divisor
 * is 0); q = clamp(rint((x + dmin*m)/(d*sc)), 0, 15) (0 when d*sc is 0).
 * Every step is one IEEE binary32 operation, rounded to nearest even.
 * k must be a multiple of 256. */
void q4o_quantize_rows(const float* x, int64_t rows, int64_t k, uint8_t* out);

/* ---- MoE id-GEMV [P1] ---------------------------------------------------------
 * For every pair p in [0, m*top_k): t = p / top_k, s = p % top_k,
 *   row(p) = t*outer + s*inner                    (floats into a)
 *   out[p, r] = sum_c W[ids[p]][r][c] * a[row(p) + c]   (products and sums fp64)
 * w: stacked slab [num_experts][n][k/256] blocks. A pair whose id lies outside
 * [0, num_experts) gets an all-zero output row. Returns the number of such
 * pairs. */
int q4o_moe_id_gemv(const uint8_t* w, int num_experts, const float* a, int64_t outer,
                    int64_t inner, const int32_t* ids, int m, int top_k, int n, int k,
                    double* out);
/* Same walk over fp64 activations (used for the down projection of the FFN). */
int q4o_moe_id_gemv_f64(const uint8_t* w, int num_experts, const double* a, int64_t outer,
                        int64_t inner, const int32_t* ids, int m, int top_k, int n, int k,
                        double* out);

/* ---- expert FFN [P2] ------------------------------------------------------------
 * g = gemv(w_gate, h_post; outer=hidden, inner=0), u = gemv(w_up, ...),
 * act[p, i] = silu(g) * u with silu(x) = x / (1 + exp(-x)),
 * expert_out = gemv(w_down, act; outer=top_k*inter, inner=inter).
 * Returns the number of out-of-range ids (their rows are zero). */
double q4o_silu(double x);
int q4o_expert_ffn(const uint8_t* w_gate, const uint8_t* w_up, const uint8_t* w_down,
                   int num_experts, const float* h_post, const int32_t* ids, int m, int top_k,
                   int hidden, int inter, double* expert_out);

/* ---- combine [P2] -----------------------------------------------------------------
 * y[t, h] = h_mid[t, h] + sum_{s<top_k} weights[t*top_k+s] * expert_out[t*top_k+s, h]
 *           + g_t * shared_out[t, h]
 * shared_mode 0: no shared term; 1: g_t = 1/(1+exp(-shared_gate[t])); 2: g_t = 1. */
void q4o_moe_combine(const double* h_mid, const double* expert_out, const double* weights,
                     const double* shared_out, const double* shared_gate, int shared_mode,
                     int m, int top_k, int hidden, double* y);

/* ---- whole layer: routed FFN + shared-expert FFN + combine ----------------------
 * The shared expert is a dense FFN with intermediate size shared_inter applied to
 * every token (num_experts=1, top_k=1, ids all 0); pass NULL slabs and
 * shared_mode 0 when there is none. Returns the number of out-of-range ids. */
int q4o_moe_layer(const uint8_t* w_gate, const uint8_t* w_up, const uint8_t* w_down,
                  int num_experts, const uint8_t* ws_gate, const uint8_t* ws_up,
                  const uint8_t* ws_down, int shared_inter, int shared_mode,
                  const float* h_post, const float* h_mid, const int32_t* ids,
                  const float* weights, const float* shared_gate, int m, int top_k,
                  int hidden, int inter, double* y);

/* ---- pair bucketing [P2 map0] -------------------------------------------------------
 * Counting sort of the pairs by expert id, stable in pair index:
 * counts[e] = #{p : ids[p] == e}, offsets = exclusive prefix sum (E+1 entries),
 * perm[offsets[e] .. offsets[e+1]) = those pairs in increasing order; pairs with
 * an out-of-range id follow in perm[offsets[E] .. P) in increasing order.
 * Returns the number of out-of-range ids. */
int q4o_bucket(const int32_t* ids, int n_pairs, int num_experts, int32_t* counts,
               int32_t* offsets, int32_t* perm);

/* ---- router and chained norm (q4o_route.c) [P2] -------------------------------------
 * bf16 decode: the upper 16 bits of a binary32. */
double q4o_bf16_to_double(uint16_t b);
/* logits[t, e] = sum_h bf16(w[e, h]) * x[t, h]   (w [num_experts, hidden] bf16 bits). */
void q4o_router_logits(const float* x, const uint16_t* w, int m, int num_experts, int hidden,
                       double* logits);
/* Softmax over all experts; the top_k largest logits are chosen, larger first, equal logits
 * by lower id; weight = the expert's softmax probability, divided by the chosen experts' sum
 * when normalize. ids/weights [m, top_k]. Returns 0, or -1 on bad arguments. */
int q4o_route_softmax(const double* logits, int m, int num_experts, int top_k, int normalize,
                      int32_t* ids, double* weights);
/* noaux_tc: s = sigmoid(logit), choice on s + bias within the topk_group best of n_group
 * groups (group score: sum of its max(1, top_k/topk_group) best s + bias), weight = s
 * (normalised over the chosen when normalize) * scale. Returns 0, or -1 on bad arguments. */
int q4o_route_sigmoid_grouped(const double* logits, const float* bias, int m, int num_experts,
                              int top_k, int n_group, int topk_group, int normalize, double scale,
                              int32_t* ids, double* weights);
/* out[t, h] = x[t, h] / sqrt(mean_h x[t, h]^2 + eps) * bf16(w[h]). */
void q4o_rms_norm(const double* x, const uint16_t* w, int m, int hidden, double eps, double* out);

/* ---- other 4-bit formats (q4o_fmt4.c) [P2 MLX-affine blob, P3 q4tp] ----------------- */
#define Q4O_FMT_AFFINE 0 /* w = scale*q + bias, bf16 scale/bias per gs weights of a row   */
#define Q4O_FMT_Q4TP 1   /* w = (q - 8) * 2^(base + code*step), 5-bit code per 32 weights  */
void q4o_affine4_dequant(const uint8_t* mat, uint64_t s_off, uint64_t b_off, int64_t n, int64_t k,
                         int gs, double* out);
void q4o_q4tp_dequant(const uint8_t* mat, int64_t n, int64_t k, double* out);
uint64_t q4o_fmt4_matrix_bytes(int fmt, int64_t n, int64_t k, int gs);
/* The q4o_moe_id_gemv walk over a slab of either format (expert e at w + e*expert_stride).
 * Returns the number of out-of-range ids (zero rows), or -1 if allocation failed. */
int q4o_moe_id_gemv_fmt4(int fmt, const uint8_t* w, uint64_t expert_stride, uint64_t s_off,
                         uint64_t b_off, int gs, int num_experts, const float* a, int64_t outer,
                         int64_t inner, const int32_t* ids, int m, int top_k, int n, int k,
                         double* out);

/* ---- threading ---------------------------------------------------------------- */
/* Threads used by the parallel loops (0 = OpenMP default). Returns the count in effect. */
int q4o_set_threads(int n);
int q4o_get_threads(void);

#ifdef __cplusplus
}
#endif
#endif

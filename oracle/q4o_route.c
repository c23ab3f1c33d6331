/*
 * q4o_route.c -- CPU oracle for the router (gate logits, top-k selection, routing weights)
 * that produces a MoE layer's expert ids and weights, and for the RMSNorm chained after the
 * layer's combine. TEST INFRASTRUCTURE, like the rest of this directory: only the tests, the
 * package smoke check and the benchmark's CPU legs load it.
 *
 * Sources (page titles of the studied material):
 *   [P2] moeflux 0.1.0-pre.3, src/riir/moe/expert_forward.rs
 *        - `MoeBuffers::gate_logits`: the router's gate logits, one f32 per expert, written by
 *          a bf16 matvec on the GPU and read by the `noaux_tc` routing;
 *        - `synth::expert_weights_seeded`: the routing weights are what the router emits after
 *          softmax, top-K and normalisation (they sum to 1);
 *        - `ChainToNormed` and the "chain appendix" of the K-expert encoder: after the combine,
 *          `rms_norm_sum_sq` then `rms_norm_apply_bf16` with the next layer's input-norm weight
 *          (bf16) and `eps` turn the combine's output into the next layer's normed input.
 * Where these leave a step open the plainest reading is taken (each is stated below at its
 * function): the softmax runs over all experts and the selection is on the logits; the
 * `noaux_tc` scoring is the aux-loss-free DeepSeek-V3 rule (sigmoid affinities, a per-expert
 * correction bias used only to choose, groups limited by the sum of their best affinities,
 * weights from the unbiased affinities); RMSNorm is x / sqrt(mean(x^2) + eps) * w.
 *
 * All arithmetic is fp64. Ties in a selection go to the lower index.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include "q4k_oracle.h"

/* bf16 is the upper half of an IEEE binary32: the value is exact in binary32 and fp64. */
double q4o_bf16_to_double(uint16_t b) {
    union { uint32_t u; float f; } v;
    v.u = (uint32_t)b << 16;
    return (double)v.f;
}

void q4o_router_logits(const float* x, const uint16_t* w, int m, int num_experts, int hidden,
                       double* logits) {
    for (int t = 0; t < m; ++t)
        for (int e = 0; e < num_experts; ++e) {
            double acc = 0.0;
            for (int h = 0; h < hidden; ++h)
                acc += q4o_bf16_to_double(w[(int64_t)e * hidden + h]) * (double)x[(int64_t)t * hidden + h];
            logits[(int64_t)t * num_experts + e] = acc;
        }
}

/* ---- selection: the k largest scores, larger first, equal scores by lower index ---------- */

typedef struct {
    double score;
    int idx;
} scored;

static int by_score_desc(const void* pa, const void* pb) {
    const scored* a = (const scored*)pa;
    const scored* b = (const scored*)pb;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return a->idx < b->idx ? -1 : (a->idx > b->idx ? 1 : 0);
}

/* The top_k entries of score[0..n) among those with allowed[i] != 0 (allowed NULL: all), in
 * selection order, into sel[0..top_k). Returns 0, or -1 if fewer than top_k are allowed. */
static int select_top(const double* score, const unsigned char* allowed, int n, int top_k, int* sel) {
    scored* s = (scored*)malloc(sizeof(scored) * (size_t)(n > 0 ? n : 1));
    if (!s) return -1;
    int cnt = 0;
    for (int i = 0; i < n; ++i)
        if (!allowed || allowed[i]) { s[cnt].score = score[i]; s[cnt].idx = i; ++cnt; }
    if (cnt < top_k) { free(s); return -1; }
    qsort(s, (size_t)cnt, sizeof(scored), by_score_desc);
    for (int j = 0; j < top_k; ++j) sel[j] = s[j].idx;
    free(s);
    return 0;
}

/* ---- softmax routing ---------------------------------------------------------------------- */

int q4o_route_softmax(const double* logits, int m, int num_experts, int top_k, int normalize,
                      int32_t* ids, double* weights) {
    if (m < 0 || num_experts < 1 || top_k < 1 || top_k > num_experts) return -1;
    double* p = (double*)malloc(sizeof(double) * (size_t)num_experts);
    int* sel = (int*)malloc(sizeof(int) * (size_t)top_k);
    if (!p || !sel) { free(p); free(sel); return -1; }
    int rc = 0;
    for (int t = 0; t < m && rc == 0; ++t) {
        const double* l = logits + (int64_t)t * num_experts;
        /* p = softmax(l) over all experts */
        double mx = l[0];
        for (int e = 1; e < num_experts; ++e) mx = l[e] > mx ? l[e] : mx;
        double z = 0.0;
        for (int e = 0; e < num_experts; ++e) { p[e] = exp(l[e] - mx); z += p[e]; }
        for (int e = 0; e < num_experts; ++e) p[e] /= z;
        /* choose on the logits (softmax keeps their order; equal logits stay equal) */
        rc = select_top(l, NULL, num_experts, top_k, sel);
        double zs = 0.0;
        for (int j = 0; j < top_k; ++j) zs += p[sel[j]];
        for (int j = 0; j < top_k; ++j) {
            ids[(int64_t)t * top_k + j] = sel[j];
            weights[(int64_t)t * top_k + j] = normalize ? p[sel[j]] / zs : p[sel[j]];
        }
    }
    free(p);
    free(sel);
    return rc;
}

/* ---- sigmoid routing with a correction bias and group limit (noaux_tc) --------------------
 * s_e = sigmoid(l_e); c_e = s_e + bias_e (bias NULL: 0) decides the choice only.
 * The experts form n_group groups of num_experts/n_group consecutive ids. A group's score is
 * the sum of its per = max(1, top_k / topk_group) largest c; the topk_group best groups are
 * kept; the top_k largest c among their experts are chosen. Weights are the chosen s,
 * divided by their sum when normalize, then multiplied by scale. n_group = 1 is plain top-k
 * on c. */
int q4o_route_sigmoid_grouped(const double* logits, const float* bias, int m, int num_experts,
                              int top_k, int n_group, int topk_group, int normalize, double scale,
                              int32_t* ids, double* weights) {
    if (m < 0 || num_experts < 1 || top_k < 1 || n_group < 1 || num_experts % n_group != 0 ||
        topk_group < 1 || topk_group > n_group)
        return -1;
    const int gsize = num_experts / n_group;
    int per = top_k / topk_group;
    if (per < 1) per = 1;
    if (per > gsize || top_k > topk_group * gsize) return -1;
    double* s = (double*)malloc(sizeof(double) * (size_t)num_experts);
    double* c = (double*)malloc(sizeof(double) * (size_t)num_experts);
    double* gscore = (double*)malloc(sizeof(double) * (size_t)n_group);
    unsigned char* allowed = (unsigned char*)malloc((size_t)num_experts);
    int* gsel = (int*)malloc(sizeof(int) * (size_t)n_group);
    int* best = (int*)malloc(sizeof(int) * (size_t)per);
    int* sel = (int*)malloc(sizeof(int) * (size_t)top_k);
    int rc = (s && c && gscore && allowed && gsel && best && sel) ? 0 : -1;
    for (int t = 0; t < m && rc == 0; ++t) {
        const double* l = logits + (int64_t)t * num_experts;
        for (int e = 0; e < num_experts; ++e) {
            s[e] = 1.0 / (1.0 + exp(-l[e]));
            c[e] = s[e] + (bias ? (double)bias[e] : 0.0);
        }
        for (int g = 0; g < n_group && rc == 0; ++g) {
            rc = select_top(c + (int64_t)g * gsize, NULL, gsize, per, best);
            double sum = 0.0;
            for (int j = 0; j < per; ++j) sum += c[(int64_t)g * gsize + best[j]];
            gscore[g] = sum;
        }
        if (rc == 0) rc = select_top(gscore, NULL, n_group, topk_group, gsel);
        if (rc != 0) break;
        for (int e = 0; e < num_experts; ++e) allowed[e] = 0;
        for (int j = 0; j < topk_group; ++j)
            for (int i = 0; i < gsize; ++i) allowed[gsel[j] * gsize + i] = 1;
        rc = select_top(c, allowed, num_experts, top_k, sel);
        double zs = 0.0;
        for (int j = 0; j < top_k; ++j) zs += s[sel[j]];
        for (int j = 0; j < top_k; ++j) {
            ids[(int64_t)t * top_k + j] = sel[j];
            weights[(int64_t)t * top_k + j] = (normalize ? s[sel[j]] / zs : s[sel[j]]) * scale;
        }
    }
    free(s); free(c); free(gscore); free(allowed); free(gsel); free(best); free(sel);
    return rc;
}

/* ---- RMSNorm -------------------------------------------------------------------------------
 * out[t, h] = x[t, h] / sqrt(sum_h x[t, h]^2 / hidden + eps) * bf16(w[h]). */
void q4o_rms_norm(const double* x, const uint16_t* w, int m, int hidden, double eps, double* out) {
    for (int t = 0; t < m; ++t) {
        const double* xr = x + (int64_t)t * hidden;
        double ss = 0.0;
        for (int h = 0; h < hidden; ++h) ss += xr[h] * xr[h];
        const double r = 1.0 / sqrt(ss / hidden + eps);
        for (int h = 0; h < hidden; ++h) out[(int64_t)t * hidden + h] = xr[h] * r * q4o_bf16_to_double(w[h]);
    }
}

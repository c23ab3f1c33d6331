// q4k_route.cuh -- the router's choice (q4k_router.cu): the top-k of a token's scores and its
// routing weights.
//
// moeflux expert_forward.rs (MoeBuffers::gate_logits, the noaux_tc routing,
// synth::expert_weights_seeded): fp32 gate logits of a bf16 matvec of the layer input, then
// the top-k choice and the routing weights. Choice: the larger score first, equal scores by the
// lower expert id, NaN below every number; see route_token.
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "q4kmoe.h"

namespace q4k {

__device__ __forceinline__ float route_bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float route_bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Ranking key: NaN below every number.
__device__ __forceinline__ float rank_key(float v) { return v != v ? -INFINITY : v; }

// One 64-bit key per candidate, larger first: the value's bits made monotone (NaN lowest, -0 as
// +0) in the high word, the complement of the index in the low word (equal values: the lower index is the
// larger key). 0 is "no candidate"; every candidate's key is above it.
__device__ __forceinline__ unsigned long long choice_key(float v, int i) {
    const uint32_t b = v == 0.0f ? 0u : __float_as_uint(v);  // -0 ranks as +0
    const uint32_t hv = (v != v) ? 0u : ((b & 0x80000000u) ? ~b : (b | 0x80000000u));
    return ((unsigned long long)hv << 32) | (uint32_t)(~(uint32_t)i);
}

// The warp's largest key (every lane gets it): the largest high word, then among the lanes that
// hold it the largest low word.
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long k) {
    const uint32_t hv = (uint32_t)(k >> 32);
    const uint32_t mv = __reduce_max_sync(0xffffffffu, hv);
    const uint32_t ml = __reduce_max_sync(0xffffffffu, hv == mv ? (uint32_t)k : 0u);
    return ((unsigned long long)mv << 32) | ml;
}

// Choose the top_k (<= N) best entries of key[0..E) (warp-wide; with gsize > 0 only experts
// whose group g = e / gsize has bit g of `kept` set). Each lane keeps its own best N
// candidates' keys, sorted, in registers (one pass over e = lane, lane + 32, ...: a max/min per
// slot); then top_k rounds of a warp-wide largest key over the lanes' heads, the owner dropping
// its head. Lane j < top_k gets the j-th choice (-1: none).
template <int N>
__device__ __forceinline__ void choose(const float* key, int E, int top_k, uint32_t kept, int gsize, int lane,
                                       int& my_i) {
    unsigned long long L[N];
#pragma unroll
    for (int j = 0; j < N; ++j) L[j] = 0ull;
    for (int e = lane; e < E; e += 32) {
        if (gsize > 0 && !((kept >> (e / gsize)) & 1u)) continue;
        unsigned long long x = choice_key(key[e], e);
#pragma unroll
        for (int j = 0; j < N; ++j) {  // insertion into the sorted list
            const unsigned long long hi = L[j] > x ? L[j] : x;
            x = L[j] > x ? x : L[j];
            L[j] = j < top_k ? hi : L[j];
        }
    }
    my_i = -1;
    for (int j = 0; j < top_k; ++j) {
        const unsigned long long b = warp_max_key(L[0]);
        if (lane == j) my_i = b ? (int)~(uint32_t)b : -1;
        if (b != 0ull && L[0] == b) {  // this lane's head was chosen: drop it
#pragma unroll
            for (int q = 0; q + 1 < N; ++q) L[q] = L[q + 1];
            L[N - 1] = 0ull;
        }
    }
}

// Sum, largest first, of the `per` (<= N) largest values of v[0..n) (rank keys).
template <int N>
__device__ __forceinline__ float top_sum(const float* v, int n, int per) {
    float top[N];
#pragma unroll
    for (int j = 0; j < N; ++j) top[j] = -INFINITY;
    for (int e0 = 0; e0 < n; e0 += 8) {
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = e0 + u < n ? rank_key(v[e0 + u]) : -INFINITY;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            float y = x[u];
#pragma unroll
            for (int j = 0; j < N; ++j) {  // insertion into a descending list
                const float hi = fmaxf(top[j], y);
                y = fminf(top[j], y);
                top[j] = j < per ? hi : top[j];
            }
        }
    }
    float s = top[0];
#pragma unroll
    for (int j = 1; j < N; ++j)
        if (j < per) s = __fadd_rn(s, top[j]);
    return rank_key(s);
}

struct RouteRule {
    int E, K, scoring, normalize, n_group, topk_group, per;
    float scale;
};

// One token's choice (warp-wide) from its logits lg[0..E) (shared memory): cs[0..E) scratch
// for the corrected scores, bias[0..E) the correction bias (grouped scoring; may be null).
// Lane j < K gets the j-th chosen expert (my_i) and its weight (my_w).
__device__ __forceinline__ void route_token(const float* lg, float* cs, const float* bias, const RouteRule& R,
                                            int lane, int& my_i, float& my_w) {
    const int E = R.E, K = R.K;
    my_i = -1;
    my_w = 0.0f;
    if (R.scoring == Q4K_ROUTE_SOFTMAX) {
        if (K <= 8) choose<8>(lg, E, K, 0u, 0, lane, my_i);
        else choose<16>(lg, E, K, 0u, 0, lane, my_i);
        const float lmax = __shfl_sync(0xffffffffu, my_i >= 0 ? lg[my_i] : 0.0f, 0);
        const float p = (lane < K && my_i >= 0) ? expf(lg[my_i] - lmax) : 0.0f;
        float z = 0.0f;
        if (R.normalize) {  // over the chosen, in choice order
            for (int j = 0; j < K; ++j) z = __fadd_rn(z, __shfl_sync(0xffffffffu, p, j));
        } else {  // over all experts: each lane's in index order, then xor shuffles
            for (int e = lane; e < E; e += 32) z = __fadd_rn(z, expf(lg[e] - lmax));
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) z = __fadd_rn(z, __shfl_xor_sync(0xffffffffu, z, off));
        }
        my_w = p / z;
        return;
    }
    const int gsize = E / R.n_group;
    for (int e = lane; e < E; e += 32) cs[e] = __fadd_rn(1.0f / (1.0f + expf(-lg[e])), bias ? bias[e] : 0.0f);
    __syncwarp();
    uint32_t kept = 0xffffffffu;
    if (R.n_group > 1) {
        // lane g scores group g; the topk_group best groups are kept
        unsigned long long gk = 0ull;  // lane g's group key (score, g)
        if (lane < R.n_group) {
            const float gs =
                R.per <= 4 ? top_sum<4>(cs + lane * gsize, gsize, R.per) : top_sum<16>(cs + lane * gsize, gsize, R.per);
            gk = choice_key(gs, lane);
        }
        kept = 0u;
        for (int j = 0; j < R.topk_group; ++j) {
            const unsigned long long b = warp_max_key(gk);
            if (b != 0ull) kept |= 1u << (~(uint32_t)b);
            if (gk == b) gk = 0ull;
        }
    }
    const int gs_arg = R.n_group > 1 ? gsize : 0;
    if (K <= 8) choose<8>(cs, E, K, kept, gs_arg, lane, my_i);
    else choose<16>(cs, E, K, kept, gs_arg, lane, my_i);
    const float s = (lane < K && my_i >= 0) ? 1.0f / (1.0f + expf(-lg[my_i])) : 0.0f;
    if (R.normalize) {
        float z = 0.0f;
        for (int j = 0; j < K; ++j) z = __fadd_rn(z, __shfl_sync(0xffffffffu, s, j));
        my_w = __fmul_rn(s / z, R.scale);
    } else {
        my_w = __fmul_rn(s, R.scale);
    }
}

}  // namespace q4k

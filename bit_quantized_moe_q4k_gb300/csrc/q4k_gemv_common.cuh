// q4k_gemv_common.cuh -- device building blocks of the id-GEMV kernel (q4k_gemv.cu).
//
// Staged activations (both kernels): per 32-element sub-block j of a row, 16-bit fixed point
// X = rint(x / delta), delta = max|x| / 32767, as a low byte plane (unsigned) and a high byte
// plane (signed) at xs + (j/2)*144 + (j%2)*64 (32 B each), and (delta, sum X) at meta[j].
// A lane's Q4_K sub-block dot product is then the exact integer S_j = sum_i q_i X_i (dp4a on
// both planes), and (ferrum-kernels q4_k_moe_id_gemv_batched.rs: Q4_K weight
// w = d*sc_j*q - dmin*m_j) sum_i w_i x_i = delta_j * (d*sc_j * S_j - dmin*m_j * sum_i X_i).
#pragma once

#include <cuda_fp16.h>

#include "q4k_bucket.cuh"
#include "q4k_internal.cuh"

namespace q4k {

constexpr int kThreads = 128;               // 4 warps
constexpr int kWarps = kThreads / 32;
constexpr int kTB = 4;                      // max tokens of one bucket per work item
constexpr int kPairBytes = 144;             // staged planes of 2 sub-blocks + 16 B pad
constexpr int kMaxGroups = 2;

constexpr int kStageUnroll = 8;            // float4 loads in flight per thread while staging

__device__ __forceinline__ uint4 ldg16(const uint8_t* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Start [p, p + bytes) into L2 (TMA engine; no registers, no load slots). p and bytes are
// multiples of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

__device__ __forceinline__ int warp_id_of_thread() { return threadIdx.x >> 5; }

// Programmatic dependent launch: let the next kernel in the stream start its prologue, and
// wait for the previous kernel's results before reading them (no-ops without the launch
// attribute).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// (scale, min) of sub-blocks ja = 2c and jb = 2c + 1 from the 16-byte block header
// (d, dmin, 12 scale bytes; GGML Q4_K placement), multiplied by d and dmin.
// The two 6-bit values of a kind are gathered side by side in one word (bytes 0 and 1):
//   c < 2:  sc = bytes 2c, 2c+1 of scales[0..3] & 63,  m = bytes of scales[4..7] & 63;
//   c >= 2: sc = low nibbles of scales[8 + 2c-4 ..] | top two bits of scales[2c-4 ..] << 4,
//           m  = high nibbles of scales[8 + 2c-4 ..] | top two bits of scales[4 + 2c-4 ..] << 4.
// A byte v becomes the float 2^23 + v by placing it under the exponent bits of 2^23, and
// fma(2^23 + v, d, -2^23 d) = v*d with one rounding: the same value as d * (float)v.
__device__ __forceinline__ void block_scales(uint4 h, int c, float& sa, float& ma, float& sb, float& mb) {
    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&h.x));  // (d, dmin)
    const unsigned sh = (unsigned)(c & 1) * 16u;
    const unsigned y = h.y >> sh, z = h.z >> sh, w = h.w >> sh;
    const bool hi = c >= 2;
    const unsigned scw = hi ? ((w & 0x0F0Fu) | ((y >> 2) & 0x3030u)) : (y & 0x3F3Fu);
    const unsigned mw = hi ? (((w >> 4) & 0x0F0Fu) | ((z >> 2) & 0x3030u)) : (z & 0x3F3Fu);
    const float od = -8388608.0f * dd.x, om = -8388608.0f * dd.y;
    sa = fmaf(__uint_as_float(__byte_perm(scw, 0x4B000000u, 0x7650)), dd.x, od);
    sb = fmaf(__uint_as_float(__byte_perm(scw, 0x4B000000u, 0x7651)), dd.x, od);
    ma = fmaf(__uint_as_float(__byte_perm(mw, 0x4B000000u, 0x7650)), dd.y, om);
    mb = fmaf(__uint_as_float(__byte_perm(mw, 0x4B000000u, 0x7651)), dd.y, om);
}

// Exact integer dot products of one lane's 64 codes with one token's staged planes.
// q0, q1: the lane's 32 code bytes; L*/H*: low / high planes of sub-blocks a and b.
// The same from staged planes held in registers: x[0..7] low plane of sub-block a, x[8..15]
// its high plane, x[16..23] / x[24..31] those of sub-block b.
__device__ __forceinline__ int dp4a_us(unsigned a, int b, int c) {  // unsigned bytes of a, signed bytes of b
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// The high nibbles are used in place (masked, i.e. times 16): both of their sums are then
// multiples of 16 and the shift at the end is exact.
__device__ __forceinline__ void dot64_regs(const uint4& q0, const uint4& q1, const uint32_t (&x)[32], int& Sa,
                                           int& Sb) {
    const unsigned qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    unsigned sal = 0, sbl = 0;
    int sah = 0, sbh = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const unsigned lo = qw[i] & 0x0F0F0F0Fu;
        const unsigned hi = qw[i] & 0xF0F0F0F0u;
        sal = __dp4a(lo, x[i], sal);
        sah = __dp4a((int)lo, (int)x[8 + i], sah);
        sbl = __dp4a(hi, x[16 + i], sbl);
        sbh = dp4a_us(hi, (int)x[24 + i], sbh);
    }
    Sa = (int)sal + sah * 256;
    Sb = ((int)sbl + sbh * 256) >> 4;
}

__device__ __forceinline__ void dot64(const uint4& q0, const uint4& q1, const uint4* xp, int& Sa, int& Sb) {
    uint32_t x[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 v = xp[i];
        x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
    }
    dot64_regs(q0, q1, x, Sa, Sb);
}

// Quantize one float4 (elements 4*fi .. 4*fi+3 of a row) as part of its 32-element sub-block:
// the 8 consecutive lanes holding fi = 8j .. 8j+7 reduce max|x| and sum(X) with shuffles.
// All 32 lanes of the warp must call it together (v = 0 where a lane has nothing); lanes with
// `store` write their part of the planes of row `xs_row` and, for the first lane of a
// sub-block, (delta, sum X) to meta_row[j].
__device__ __forceinline__ void stage_quad(float4 v, int fi, bool store, uint8_t* xs_row, float2* meta_row) {
    float mx = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    int X[4] = {0, 0, 0, 0};
    if (mx > 0.0f) {
        const float inv = 32767.0f / mx;
        X[0] = max(-32767, min(32767, __float2int_rn(v.x * inv)));
        X[1] = max(-32767, min(32767, __float2int_rn(v.y * inv)));
        X[2] = max(-32767, min(32767, __float2int_rn(v.z * inv)));
        X[3] = max(-32767, min(32767, __float2int_rn(v.w * inv)));
    }
    int sx = X[0] + X[1] + X[2] + X[3];
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) sx += __shfl_xor_sync(0xffffffffu, sx, off);
    if (store) {
        const int j = fi >> 3, wi = fi & 7;
        const uint32_t lo = (uint32_t)(X[0] & 0xFF) | ((uint32_t)(X[1] & 0xFF) << 8) |
                            ((uint32_t)(X[2] & 0xFF) << 16) | ((uint32_t)(X[3] & 0xFF) << 24);
        const uint32_t hi = (uint32_t)((X[0] >> 8) & 0xFF) | ((uint32_t)((X[1] >> 8) & 0xFF) << 8) |
                            ((uint32_t)((X[2] >> 8) & 0xFF) << 16) | ((uint32_t)((X[3] >> 8) & 0xFF) << 24);
        uint32_t* planes = reinterpret_cast<uint32_t*>(xs_row + (j >> 1) * kPairBytes + (j & 1) * 64);
        planes[wi] = lo;
        planes[8 + wi] = hi;
        if (wi == 0) meta_row[j] = make_float2(mx / 32767.0f, (float)sx);
    }
}

constexpr int kDepth = 4;  // blocks of the weight stream in flight per lane

// Small-batch bucketing, one warp per group (at most 32 pairs): lane p holds pair p's expert;
// __match_any_sync groups the pairs of one expert (the member mask, in increasing pair order,
// is the bucket); the distinct experts are ranked by id over the leaders' ballot; a warp scan
// turns their item counts into item offsets. By rank r < U: e[r] expert, mask[r] members,
// start[r] first item; start[U] is the group's item total.
struct FastGroup {
    int e[32];
    unsigned mask[32];
    int start[33];
    int U;
};

// ids == null: every pair uses expert 0. An expert's items: ceil(pairs / TB_) chunks times
// `tiles` row tiles (none when tc_min > 0 and it has at least tc_min pairs).
__device__ __forceinline__ void fast_bucket(const int32_t* ids, int n_pairs, int num_experts, int tiles, int TB_,
                                            int tc_min, FastGroup& F, int* s_bad) {
    const int lane = threadIdx.x & 31;
    int key = -1;
    if (lane < n_pairs) {
        const int32_t e = ids ? ids[lane] : 0;
        key = id_valid(e, num_experts) ? e : -1;
    }
    const unsigned bad = __ballot_sync(0xffffffffu, lane < n_pairs && key < 0);
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const bool leader = key >= 0 && (__ffs(peers) - 1) == lane;
    const int cnt = __popc(peers);
    const unsigned leaders = __ballot_sync(0xffffffffu, leader);
    const int U = __popc(leaders);
    int rank = 0;
    for (unsigned rest = leaders; rest; rest &= rest - 1u) {  // uniform over the warp
        const int kj = __shfl_sync(0xffffffffu, key, __ffs(rest) - 1);
        rank += kj < key ? 1 : 0;
    }
    int items = 0;
    if (leader) {
        items = (tc_min > 0 && cnt >= tc_min) ? 0 : ((cnt + TB_ - 1) / TB_) * tiles;
        F.e[rank] = key;
        F.mask[rank] = peers;
        F.start[rank] = items;  // item count, turned into an offset below
    }
    __syncwarp();
    int v = lane < U ? F.start[lane] : 0;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane < U) F.start[lane] = incl - v;
    if (lane == 31) F.start[U] = incl;  // U <= 32
    if (lane == 0) { F.U = U; *s_bad = __popc(bad); }
    __syncwarp();
}


// Combine of rows [r0, r1) of every token (moeflux expert_forward.rs, the batched combine):
//   y = h_mid + sum_s w[t*T+s] * out0[t*T+s] + g_t * out1[t],
// g_t = sigmoid(shared_gate[t]) or 1 (out1 null: no shared term), slots in order. Expert
// rows were written by other CTAs: read them from L2. A pair whose id is out of range
// contributes nothing (its row is zero by definition). Thread tid of nthr.
__device__ __forceinline__ void combine_span(const CombineSpec& cb, const float* out0, const int32_t* ids,
                                             int num_experts, int n_pairs, int T, int H, const float* out1, int r0,
                                             int r1, int tid, int nthr) {
    const int m = n_pairs / T;
    const int span = r1 - r0;
    for (int idx = tid; idx < m * span; idx += nthr) {
        const int t = idx / span, r = r0 + idx % span;
        const int64_t o = (int64_t)t * H + r;
        float acc = cb.h_mid[o];
        for (int s = 0; s < T; ++s) {
            const int p = t * T + s;
            if (id_valid(ids ? ids[p] : 0, num_experts)) acc = fmaf(cb.weights[p], __ldcg(out0 + (int64_t)p * H + r), acc);
        }
        if (out1) {
            const float g = cb.shared_mode == Q4K_SHARED_SIGMOID ? 1.0f / (1.0f + expf(-cb.shared_gate[t])) : 1.0f;
            acc = fmaf(g, __ldcg(out1 + o), acc);
        }
        cb.y[o] = acc;
    }
}

}  // namespace q4k

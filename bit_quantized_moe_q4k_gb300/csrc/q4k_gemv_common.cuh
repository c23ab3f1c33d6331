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

// 16 bytes of a weight row: from global memory, or (SMEM) from a copy in shared memory.
template <bool SMEM>
__device__ __forceinline__ uint4 ldw16(const uint8_t* p) {
    if (!SMEM) return ldg16(p);
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
    return v;
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

// One lane's term of a block for one token, its sub-blocks a and b:
//   delta_a * (d*sc_a * S_a - dmin*m_a * sum X_a) + delta_b * (d*sc_b * S_b - dmin*m_b * sum X_b)
// (mt = (delta_a, sum X_a, delta_b, sum X_b)). Every rounding is spelled out (no contraction
// choices left to the compiler).
//
// The order in which a row's terms are summed is fixed for every kernel, whatever lanes it
// gives the row: with the row's blocks split over S lanes (block b to lane sl = b % S, in the
// order i = b / S), each (c, sl) first folds its terms left to right, T_0 + T_1 + T_2 + ...,
// then the partial sums of the 4*S lanes (c, sl) are added by xor shuffles over c (1, 2) and
// then over sl (4, 8, ...). So every kernel gets the same bits for a row (fold_term and the
// lane shuffles of item_compute, used by the id-GEMV, the single-launch layer and the other
// 4-bit formats' kernel).
__device__ __forceinline__ float block_term(const float4& mt, float sa, float ma, float sb, float mb, int Sa, int Sb) {
    const float ua = __fmaf_rn(sa, (float)Sa, -__fmul_rn(ma, mt.y));
    const float ub = __fmaf_rn(sb, (float)Sb, -__fmul_rn(mb, mt.w));
    return __fmaf_rn(mt.z, ub, __fmul_rn(mt.x, ua));
}

// The fold of a lane's terms: the first term as it is, every later one added on.
__device__ __forceinline__ float fold_term(float acc, float term, bool first) {
    return first ? term : __fadd_rn(acc, term);
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


// One projection group of a launch as the kernels see it.
struct GroupDev {
    const uint8_t* w;
    const uint8_t* w2;
    const int32_t* ids;
    const float* a;
    float* out;
    int64_t outer, inner;
    int64_t nb01;  // bytes per row
    int64_t nb02;  // bytes per expert
    int num_experts, n_pairs, top_k, n, k, tiles;
    int lg_split;  // log2 of the lanes splitting one row's blocks (rows per warp = 8 >> lg_split)
};

// What a lane streams for one work item: one row of one slab (kOne), the same row of two
// slabs (kFused: gate and up, out = silu(g) * u), or two rows of one slab half a tile apart
// (kPair: a tile of twice the rows for the same registers).
constexpr int kOne = 0, kFused = 1, kPair = 2;

// Rows of a work item's tile for a split lg and kind.
__host__ __device__ __forceinline__ int item_tile_rows(int lg_split, int kind) {
    return kWarps * (8 >> lg_split) * (kind == kPair ? 2 : 1);
}

// Host: log2 of the lanes that split one row's blocks for a given k, so that a lane's share
// fits the kDepth-deep ring where possible (k = 2048: 2 lanes x 4 blocks; k = 4096: 4 x 4;
// k = 768: 1 x 3).
inline int lg_split_for(int k) {
    const int nb = k / kQK;
    return nb >= 4 * kDepth ? 2 : (nb >= 2 * kDepth ? 1 : 0);
}

// Host: the kernels' view of a group with the given split and item kind (row tiles of
// item_tile_rows(lg_split, kind) rows).
inline GroupDev group_dev(const GemvGroup& S, int lg_split, int kind = kOne) {
    GroupDev G{};
    G.w = S.w; G.w2 = S.w2; G.ids = S.ids; G.a = S.a; G.out = S.out;
    G.outer = S.outer; G.inner = S.inner;
    G.nb01 = (int64_t)(S.k / kQK) * kBlockBytes;
    G.nb02 = (int64_t)S.n * G.nb01;
    G.num_experts = S.num_experts; G.n_pairs = S.m * S.top_k; G.top_k = S.top_k;
    G.n = S.n; G.k = S.k;
    G.lg_split = lg_split;
    const int tile_rows = item_tile_rows(lg_split, kind);
    G.tiles = (S.n + tile_rows - 1) / tile_rows;
    return G;
}

// Quantize one activation row of k floats into its planes (xs_row) and (delta, sum X) pairs
// (meta_row). Thread f handles float4 f of the row; all loads of a pass are issued before any
// is used. SRC: 0 global (read-only path), 1 global written by other CTAs of this launch (read
// from L2), 2 shared memory. NTHR threads (whole warps) take part, tid = 0 .. NTHR-1.
template <int SRC, int NTHR = kThreads>
__device__ __forceinline__ void stage_row(const float* row, int k, uint8_t* xs_row, float2* meta_row,
                                          int tid = threadIdx.x) {
    const int nf = k / 4;
    for (int f0 = 0; f0 < nf; f0 += NTHR * kStageUnroll) {
        float4 v[kStageUnroll];
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            const int f = f0 + u * NTHR + tid;
            const float4* src = reinterpret_cast<const float4*>(row) + f;
            v[u] = f < nf ? (SRC == 0 ? __ldg(src) : (SRC == 1 ? __ldcg(src) : *src)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            const int f = f0 + u * NTHR + tid;  // groups of 8 threads are all in or all out
            if (f0 + u * NTHR >= nf) break;
            stage_quad(v[u], f, f < nf, xs_row, meta_row);
        }
    }
}

// The activation row of pair p.
__device__ __forceinline__ const float* act_row(const GroupDev& G, int p) {
    return G.a + (int64_t)(p / G.top_k) * G.outer + (int64_t)(p % G.top_k) * G.inner;
}

// Stage the activation rows of the item's pairs (token t at xs + t*tok_bytes, meta + t*(k/32)).
// COHERENT: the rows were written by other CTAs of the same launch (read them from L2).
template <bool COHERENT = false>
__device__ __forceinline__ void stage_rows(const GroupDev& G, const int* s_pairs, int nt, uint8_t* xs,
                                           float2* meta) {
    const int64_t tok_bytes = (int64_t)(G.k / 64) * kPairBytes;
    for (int t = 0; t < nt; ++t)
        stage_row<COHERENT ? 1 : 0>(act_row(G, s_pairs[t]), G.k, xs + t * tok_bytes, meta + t * (G.k / 32));
}

// The same from rows already copied into shared memory (token t at raw + t*k).
__device__ __forceinline__ void stage_rows_smem(const float* raw, int nt, int k, uint8_t* xs, float2* meta) {
    const int64_t tok_bytes = (int64_t)(k / 64) * kPairBytes;
    for (int t = 0; t < nt; ++t) stage_row<2>(raw + (int64_t)t * k, k, xs + t * tok_bytes, meta + t * (k / 32));
}

// A lane's share of one work item (a row tile of one expert's slab) and its kDepth-deep ring
// of weight loads: H the block header, Q0/Q1 the lane's 32 code bytes of the first stream;
// H2/R0/R1 the same of the second (kFused: the up slab's row; kPair: the row half a tile on).
// Lane layout: lane = c | s << 2 | r << (2 + lg_split). c (0..3) picks the 64-weight group of
// a block (code bytes 32c..32c+31 = sub-blocks 2c, 2c+1); s picks which blocks of the row the
// lane streams (b = s, s + S, ...; S = 1 << lg_split lanes share a row's blocks); r is the row
// within the warp (8 / S rows per warp). Splitting the row's blocks over more lanes keeps
// each lane's share within the ring, so all of an item's weight loads are in flight at once.
template <int KIND, bool SMEM = false>
struct ItemLane {
    const uint8_t* wr;
    const uint8_t* wr2;
    int c, S, sl, row, row2, nbl;
    bool row_ok, row2_ok;
    uint4 H[kDepth], Q0[kDepth], Q1[kDepth], H2[kDepth], R0[kDepth], R1[kDepth];
};

// Start the item's weight stream: the first kDepth blocks of the lane's share. SMEM: the
// tile's rows (from its first row, consecutive, nb01 bytes each) are in shared memory at
// smem_tile (kFused: the up slab's at smem_tile2).
template <int KIND, bool SMEM = false>
__device__ __forceinline__ void item_issue(const GroupDev& G, int e, int tile, int lane, int warp,
                                           ItemLane<KIND, SMEM>& L, const uint8_t* smem_tile = nullptr,
                                           const uint8_t* smem_tile2 = nullptr) {
    const int lgS = G.lg_split;
    const int rpw = 8 >> lgS;  // rows per warp
    L.c = lane & 3;
    L.S = 1 << lgS;
    L.sl = (lane >> 2) & (L.S - 1);
    L.row = tile * item_tile_rows(lgS, KIND) + warp * rpw + (lane >> (2 + lgS));
    L.row_ok = L.row < G.n;
    L.row2 = L.row + kWarps * rpw;
    L.row2_ok = KIND == kFused ? L.row_ok : (KIND == kPair && L.row2 < G.n);
    const int nb = G.k / kQK;
    L.nbl = L.sl < nb ? (nb - L.sl + L.S - 1) / L.S : 0;  // blocks b = sl + S*i of this lane
    const int64_t tile_off = (int64_t)tile * item_tile_rows(lgS, KIND) * G.nb01;
    const uint8_t* slab = SMEM ? smem_tile - tile_off : G.w + (int64_t)e * G.nb02;
    const uint8_t* slab2 = KIND != kFused ? nullptr : (SMEM ? smem_tile2 - tile_off : G.w2 + (int64_t)e * G.nb02);
    L.wr = slab + (int64_t)(L.row_ok ? L.row : 0) * G.nb01;
    L.wr2 = KIND == kFused ? slab2 + (int64_t)(L.row_ok ? L.row : 0) * G.nb01
                           : (KIND == kPair ? slab + (int64_t)(L.row2_ok ? L.row2 : 0) * G.nb01 : nullptr);
#pragma unroll
    for (int i = 0; i < kDepth; ++i) {
        L.H[i] = L.Q0[i] = L.Q1[i] = L.H2[i] = L.R0[i] = L.R1[i] = make_uint4(0, 0, 0, 0);
        if (i < L.nbl) {
            if (L.row_ok) {
                const uint8_t* p = L.wr + (int64_t)(L.sl + L.S * i) * kBlockBytes;
                L.H[i] = ldw16<SMEM>(p); L.Q0[i] = ldw16<SMEM>(p + 16 + 32 * L.c);
                L.Q1[i] = ldw16<SMEM>(p + 32 + 32 * L.c);
            }
            if (KIND != kOne && L.row2_ok) {
                const uint8_t* p2 = L.wr2 + (int64_t)(L.sl + L.S * i) * kBlockBytes;
                L.H2[i] = ldw16<SMEM>(p2); L.R0[i] = ldw16<SMEM>(p2 + 16 + 32 * L.c);
                L.R1[i] = ldw16<SMEM>(p2 + 32 + 32 * L.c);
            }
        }
    }
}

// A result word of the single-launch layer: the float's bits under the launch's 32-bit tag, so
// a reader knows from the word alone whether this launch has written it. One relaxed 64-bit
// store (single-copy atomic).
__device__ __forceinline__ void st_tagged(uint64_t* p, float v, uint32_t tag32) {
    const uint64_t w = ((uint64_t)tag32 << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

// The item's dot products against the nt staged tokens (pairs s_pairs[0..nt)), the reduction
// over the lanes of a row, and the write of out[pair, row] (kFused: silu(g) * u; kPair: both
// rows). out64 != null: the results go as tagged words to out64[pair, row] instead.
template <int KIND, int TB, bool SMEM = false>
__device__ __forceinline__ void item_compute(const GroupDev& G, ItemLane<KIND, SMEM>& L, const int* s_pairs, int nt,
                                             const uint8_t* xs, const float2* meta, int lane,
                                             uint64_t* out64 = nullptr, uint32_t tag32 = 0) {
    constexpr bool TWO = KIND != kOne;
    const int S = L.S, c = L.c;
    const int nsb = G.k / 32;
    const int64_t tok_bytes = (int64_t)(G.k / 64) * kPairBytes;
    float acc[TB], acc2[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) { acc[t] = 0.0f; acc2[t] = 0.0f; }
    for (int i0 = 0; i0 < L.nbl; i0 += kDepth) {
#pragma unroll
        for (int j = 0; j < kDepth; ++j) {
            const int i = i0 + j;
            if (i < L.nbl) {
                const int b = L.sl + S * i;
                float sa, ma, sb, mb, sa2 = 0.f, ma2 = 0.f, sb2 = 0.f, mb2 = 0.f;
                block_scales(L.H[j], c, sa, ma, sb, mb);
                if (TWO) block_scales(L.H2[j], c, sa2, ma2, sb2, mb2);
#pragma unroll
                for (int t = 0; t < TB; ++t) {
                    if (t < nt) {
                        const uint4* xp = reinterpret_cast<const uint4*>(xs + t * tok_bytes + (4 * b + c) * kPairBytes);
                        const float4 mt = *reinterpret_cast<const float4*>(meta + t * nsb + 8 * b + 2 * c);
                        int Sa, Sb;
                        dot64(L.Q0[j], L.Q1[j], xp, Sa, Sb);
                        acc[t] = fold_term(acc[t], block_term(mt, sa, ma, sb, mb, Sa, Sb), i == 0);
                        if (TWO) {
                            dot64(L.R0[j], L.R1[j], xp, Sa, Sb);
                            acc2[t] = fold_term(acc2[t], block_term(mt, sa2, ma2, sb2, mb2, Sa, Sb), i == 0);
                        }
                    }
                }
                if (i + kDepth < L.nbl) {  // refill this slot with block b + S*kDepth
                    if (L.row_ok) {
                        const uint8_t* p = L.wr + (int64_t)(b + S * kDepth) * kBlockBytes;
                        L.H[j] = ldw16<SMEM>(p); L.Q0[j] = ldw16<SMEM>(p + 16 + 32 * c);
                        L.Q1[j] = ldw16<SMEM>(p + 32 + 32 * c);
                    }
                    if (TWO && L.row2_ok) {
                        const uint8_t* p2 = L.wr2 + (int64_t)(b + S * kDepth) * kBlockBytes;
                        L.H2[j] = ldw16<SMEM>(p2); L.R0[j] = ldw16<SMEM>(p2 + 16 + 32 * c);
                        L.R1[j] = ldw16<SMEM>(p2 + 32 + 32 * c);
                    }
                }
            }
        }
    }
    // reduce over the 4*S lanes of the row (c bits, then s bits) and write
#pragma unroll
    for (int t = 0; t < TB; ++t) {
        for (int off = 1; off < 4 * S; off <<= 1) {
            acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
            if (TWO) acc2[t] += __shfl_xor_sync(0xffffffffu, acc2[t], off);
        }
    }
    if ((lane & (4 * S - 1)) == 0) {
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            if (t < nt && out64) {
                uint64_t* o = out64 + (int64_t)s_pairs[t] * G.n;
                if (KIND == kFused) {
                    if (L.row_ok) st_tagged(o + L.row, silu(acc[t]) * acc2[t], tag32);
                } else {
                    if (L.row_ok) st_tagged(o + L.row, acc[t], tag32);
                    if (KIND == kPair && L.row2_ok) st_tagged(o + L.row2, acc2[t], tag32);
                }
            } else if (t < nt) {
                float* o = G.out + (int64_t)s_pairs[t] * G.n;
                if (KIND == kFused) {
                    if (L.row_ok) o[L.row] = silu(acc[t]) * acc2[t];
                } else {
                    if (L.row_ok) o[L.row] = acc[t];
                    if (KIND == kPair && L.row2_ok) o[L.row2] = acc2[t];
                }
            }
        }
    }
}

// A work item of a launch whose groups were bucketed by fast_bucket: group gi, bucket rank r
// (expert e), row tile, chunk of the bucket and its nt <= TB_ tokens.
struct FastLoc {
    int gi, r, e, tile, nt, chunk;
};

// Warp-wide (all 32 lanes; the result is the same in every lane). items[gi]: first item of
// group gi. pairs != null: the chunk's pairs, in increasing order, go to pairs[0..nt).
__device__ __forceinline__ FastLoc fast_locate(const FastGroup* F, const int* items, const GroupDev* g, int n_groups,
                                               int TB_, int item, int* pairs) {
    const int lane = threadIdx.x & 31;
    int gi = 0;
    while (gi + 1 < n_groups && item >= items[gi + 1]) ++gi;
    const FastGroup& Fg = F[gi];
    const int local = item - items[gi];
    const bool mine = lane < Fg.U && Fg.start[lane] <= local && local < Fg.start[lane + 1];
    const int r = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
    const unsigned mask = Fg.mask[r];
    const int in_e = local - Fg.start[r];
    const int tiles = g[gi].tiles;
    FastLoc L;
    L.gi = gi;
    L.r = r;
    L.e = Fg.e[r];
    L.chunk = in_e / tiles;  // tiles of one chunk run together (no restaging)
    L.tile = in_e % tiles;
    L.nt = min(TB_, __popc(mask) - L.chunk * TB_);
    if (pairs) {  // pair `lane` is a member: its place in the bucket is the members below it
        const int q = __popc(mask & ((1u << lane) - 1u)) - L.chunk * TB_;
        if (((mask >> lane) & 1u) && q >= 0 && q < L.nt) pairs[q] = lane;
    }
    return L;
}

// Combine of rows [r0, r1) of every token (moeflux expert_forward.rs, the batched combine):
//   y = h_mid + sum_s w[t*T+s] * out0[t*T+s] + g_t * out1[t],
// g_t = sigmoid(shared_gate[t]) or 1 (out1 null: no shared term), slots in order. Expert
// rows were written by other CTAs: read them from L2. A pair whose id is out of range
// contributes nothing (its row is zero by definition). Thread tid of nthr. All of an
// element's loads are issued before the sums (one round trip), which run in slot order.
__device__ __forceinline__ void combine_span(const CombineSpec& cb, const float* out0, const int32_t* ids,
                                             int num_experts, int n_pairs, int T, int H, const float* out1, int r0,
                                             int r1, int tid, int nthr) {
    const int m = n_pairs / T;
    const int span = r1 - r0;
    for (int idx = tid; idx < m * span; idx += nthr) {
        const int t = idx / span, r = r0 + idx % span;
        const int64_t o = (int64_t)t * H + r;
        float v[Q4K_MAX_TOP_K], w[Q4K_MAX_TOP_K];
        bool ok[Q4K_MAX_TOP_K];
#pragma unroll
        for (int s = 0; s < Q4K_MAX_TOP_K; ++s) {  // independent loads (rows of bad ids unused)
            const int p = t * T + s;
            ok[s] = s < T && id_valid(ids ? ids[p] : 0, num_experts);
            w[s] = s < T ? cb.weights[p] : 0.0f;
            v[s] = s < T ? __ldcg(out0 + (int64_t)p * H + r) : 0.0f;
        }
        const float sh = out1 ? __ldcg(out1 + o) : 0.0f;
        float acc = cb.h_mid[o];
#pragma unroll
        for (int s = 0; s < Q4K_MAX_TOP_K; ++s)
            if (ok[s]) acc = fmaf(w[s], v[s], acc);
        if (out1) {
            const float g = cb.shared_mode == Q4K_SHARED_SIGMOID ? 1.0f / (1.0f + expf(-cb.shared_gate[t])) : 1.0f;
            acc = fmaf(g, sh, acc);
        }
        cb.y[o] = acc;
    }
}

}  // namespace q4k

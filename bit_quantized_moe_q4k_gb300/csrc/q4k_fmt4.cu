// q4k_fmt4.cu -- the MoE id-GEMV over two other 4-bit weight formats, on the Q4_K kernel's
// skeleton: the same pair bucketing (fast_bucket / block histogram), the same activation
// staging (16-bit fixed point per 32-element sub-block, exact dp4a sums), the same lane
// layout (a lane owns 64 weights = sub-blocks 2c, 2c+1 of a 256-weight block; S lanes split a
// row's blocks; kDepth blocks in flight), the same fold order of a row's terms and the same
// fused gate|up + SwiGLU epilogue. Only the decoder differs:
//
//  * MLX-style affine 4-bit (moeflux expert_forward.rs: the expert blob's weights | scales |
//    biases bound at three offsets, GROUP_SIZE): w = scale * q + bias per group of gs weights
//    of a row, bf16 scale and bias. Per sub-block j (32 weights, one group or half of one):
//      sum_i w_i x_i = delta_j * (scale * S_j + bias * sum_i X_i).
//  * q4tp (cortiq-engine mv_lab.rs, the production kernel `cur`): w = (q - 8) * 2^(base +
//    code*step), a 5-bit code per 32-weight group, (base, step) binary16 per row:
//      sum_i w_i x_i = delta_j * (scale_j * S_j - 8 * scale_j * sum_i X_i).
// Both formats keep the 4-bit codes in weight order (weight 8i+h in bits 4h of little-endian
// word i), so a word's nibbles are spread to two byte vectors (weights 8i..8i+3, 8i+4..8i+7)
// that line up with the staged planes.
#include <algorithm>

#include "q4k_gemv_common.cuh"

namespace q4k {
namespace {

struct Fmt4Params {
    GroupDev g;              // a, ids, out, walk, n, k, tiles, lg_split (w / w2: the slabs)
    int64_t expert_stride;   // bytes from one expert's matrix to the next
    int64_t s_off, b_off;    // affine: scales, biases from a matrix's start; q4tp: params, codes
    int gs;                  // affine group size (32, 64, 128)
    int cstride;             // q4tp code bytes per row
    int tb;
    int fast;
    int x_off, meta_off;
    int* err_flag;
};

// Nibbles of weights 8i..8i+7 (one little-endian word) as bytes: lo = weights 8i..8i+3,
// hi = weights 8i+4..8i+7.
__device__ __forceinline__ void spread_nibbles(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t t = w & 0x0F0F0F0Fu;          // weights 0, 2, 4, 6
    const uint32_t u = (w >> 4) & 0x0F0F0F0Fu;   // weights 1, 3, 5, 7
    lo = __byte_perm(t, u, 0x5140);
    hi = __byte_perm(t, u, 0x7362);
}

// Exact integer dot products of a lane's 64 codes (weight order) with one token's staged
// planes of sub-blocks a and b (xp: low / high plane of a, then of b).
__device__ __forceinline__ void dot64_seq(const uint4& q0, const uint4& q1, const uint4* xp, int& Sa, int& Sb) {
    uint32_t x[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 v = xp[i];
        x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
    }
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    unsigned sal = 0, sbl = 0;
    int sah = 0, sbh = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t lo, hi;
        spread_nibbles(qw[i], lo, hi);  // sub-block a: weights 8i .. 8i+7
        sal = __dp4a(lo, x[2 * i], sal);
        sal = __dp4a(hi, x[2 * i + 1], sal);
        sah = __dp4a((int)lo, (int)x[8 + 2 * i], sah);
        sah = __dp4a((int)hi, (int)x[8 + 2 * i + 1], sah);
        spread_nibbles(qw[4 + i], lo, hi);  // sub-block b
        sbl = __dp4a(lo, x[16 + 2 * i], sbl);
        sbl = __dp4a(hi, x[16 + 2 * i + 1], sbl);
        sbh = __dp4a((int)lo, (int)x[24 + 2 * i], sbh);
        sbh = __dp4a((int)hi, (int)x[24 + 2 * i + 1], sbh);
    }
    Sa = (int)sal + sah * 256;
    Sb = (int)sbl + sbh * 256;
}

__device__ __forceinline__ float bf16_at(const uint8_t* p) {
    return __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t*>(p)) << 16);
}

// One lane's share of an item for a format, two slabs when TWO (gate and up).
template <bool TWO>
struct FmtLane {
    const uint8_t* m1;  // the expert's matrix (codes at row * k/2)
    const uint8_t* m2;
    int c, S, sl, row, nbl;
    bool row_ok;
    float base1, step1, base2, step2;  // q4tp row parameters
    uint4 Q0[kDepth], Q1[kDepth], R0[kDepth], R1[kDepth];
    uint32_t A[kDepth], B[kDepth], A2[kDepth], B2[kDepth];  // affine: scale, bias bits; q4tp: codes
};

// The per-block side data of (row, block b, lane c): affine: the bf16 scales of sub-blocks a
// and b (lo / hi halves of A) and their biases (B); q4tp: the two 5-bit codes (A).
template <int FMT>
__device__ __forceinline__ void side_load(const Fmt4Params& P, const uint8_t* mat, int row, int b, int c, uint32_t& A,
                                          uint32_t& B) {
    const int k = P.g.k;
    if (FMT == Q4K_FMT_AFFINE4) {
        const int ja = 8 * b + 2 * c;  // first sub-block of the lane
        const int64_t rowg = (int64_t)row * (k / P.gs);
        if (P.gs == 32) {  // two groups, adjacent bf16 pairs (4-byte aligned: ja even)
            A = *reinterpret_cast<const uint32_t*>(mat + P.s_off + 2 * (rowg + ja));
            B = *reinterpret_cast<const uint32_t*>(mat + P.b_off + 2 * (rowg + ja));
        } else {
            const int g = (32 * ja) / P.gs;  // one group for both sub-blocks
            const uint32_t s = *reinterpret_cast<const uint16_t*>(mat + P.s_off + 2 * (rowg + g));
            const uint32_t t = *reinterpret_cast<const uint16_t*>(mat + P.b_off + 2 * (rowg + g));
            A = s | (s << 16);
            B = t | (t << 16);
        }
    } else {
        const int bit = 5 * (8 * b + 2 * c);  // codes of groups 8b+2c and 8b+2c+1: 10 bits
        const uint8_t* cp = mat + P.b_off + (int64_t)row * P.cstride + (bit >> 3);
        A = (((uint32_t)cp[0] | ((uint32_t)cp[1] << 8)) >> (bit & 7)) & 0x3FFu;
        B = 0;
    }
}

// (scale, min) pairs of sub-blocks a and b in block_term's convention:
// term_j = scale_j * S_j - min_j * sum X_j.
template <int FMT>
__device__ __forceinline__ void side_scales(uint32_t A, uint32_t B, float base, float step, float& sa, float& ma,
                                            float& sb, float& mb) {
    if (FMT == Q4K_FMT_AFFINE4) {
        sa = __uint_as_float(A << 16);
        sb = __uint_as_float(A & 0xFFFF0000u);
        ma = -__uint_as_float(B << 16);
        mb = -__uint_as_float(B & 0xFFFF0000u);
    } else {
        sa = exp2f(__fmaf_rn((float)(A & 31u), step, base));
        sb = exp2f(__fmaf_rn((float)(A >> 5), step, base));
        ma = 8.0f * sa;
        mb = 8.0f * sb;
    }
}

template <int FMT, bool TWO>
__device__ __forceinline__ void fmt_issue(const Fmt4Params& P, int e, int tile, int lane, int warp, FmtLane<TWO>& L) {
    const GroupDev& G = P.g;
    const int lgS = G.lg_split;
    const int rpw = 8 >> lgS;
    L.c = lane & 3;
    L.S = 1 << lgS;
    L.sl = (lane >> 2) & (L.S - 1);
    L.row = tile * item_tile_rows(lgS, kOne) + warp * rpw + (lane >> (2 + lgS));
    L.row_ok = L.row < G.n;
    const int nb = G.k / kQK;
    L.nbl = L.sl < nb ? (nb - L.sl + L.S - 1) / L.S : 0;
    const int row = L.row_ok ? L.row : 0;
    L.m1 = G.w + (int64_t)e * P.expert_stride;
    L.m2 = TWO ? G.w2 + (int64_t)e * P.expert_stride : nullptr;
    L.base1 = L.step1 = L.base2 = L.step2 = 0.0f;
    if (FMT == Q4K_FMT_Q4TP && L.row_ok) {
        const float2 p1 = __half22float2(*reinterpret_cast<const __half2*>(L.m1 + P.s_off + 4 * (int64_t)row));
        L.base1 = p1.x; L.step1 = p1.y;
        if (TWO) {
            const float2 p2 = __half22float2(*reinterpret_cast<const __half2*>(L.m2 + P.s_off + 4 * (int64_t)row));
            L.base2 = p2.x; L.step2 = p2.y;
        }
    }
    const int64_t rb = (int64_t)row * (G.k / 2);
#pragma unroll
    for (int i = 0; i < kDepth; ++i) {
        L.Q0[i] = L.Q1[i] = L.R0[i] = L.R1[i] = make_uint4(0, 0, 0, 0);
        L.A[i] = L.B[i] = L.A2[i] = L.B2[i] = 0u;
        if (i < L.nbl && L.row_ok) {
            const int b = L.sl + L.S * i;
            const uint8_t* p = L.m1 + rb + 128 * b + 32 * L.c;
            L.Q0[i] = ldg16(p); L.Q1[i] = ldg16(p + 16);
            side_load<FMT>(P, L.m1, row, b, L.c, L.A[i], L.B[i]);
            if (TWO) {
                const uint8_t* p2 = L.m2 + rb + 128 * b + 32 * L.c;
                L.R0[i] = ldg16(p2); L.R1[i] = ldg16(p2 + 16);
                side_load<FMT>(P, L.m2, row, b, L.c, L.A2[i], L.B2[i]);
            }
        }
    }
}

template <int FMT, bool TWO, int TB>
__device__ __forceinline__ void fmt_compute(const Fmt4Params& P, FmtLane<TWO>& L, const int* s_pairs, int nt,
                                            const uint8_t* xs, const float2* meta, int lane) {
    const GroupDev& G = P.g;
    const int S = L.S, c = L.c;
    const int nsb = G.k / 32;
    const int64_t tok_bytes = (int64_t)(G.k / 64) * kPairBytes;
    const int row = L.row_ok ? L.row : 0;
    const int64_t rb = (int64_t)row * (G.k / 2);
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
                side_scales<FMT>(L.A[j], L.B[j], L.base1, L.step1, sa, ma, sb, mb);
                if (TWO) side_scales<FMT>(L.A2[j], L.B2[j], L.base2, L.step2, sa2, ma2, sb2, mb2);
#pragma unroll
                for (int t = 0; t < TB; ++t) {
                    if (t < nt) {
                        const uint4* xp = reinterpret_cast<const uint4*>(xs + t * tok_bytes + (4 * b + c) * kPairBytes);
                        const float4 mt = *reinterpret_cast<const float4*>(meta + t * nsb + 8 * b + 2 * c);
                        int Sa, Sb;
                        dot64_seq(L.Q0[j], L.Q1[j], xp, Sa, Sb);
                        acc[t] = fold_term(acc[t], block_term(mt, sa, ma, sb, mb, Sa, Sb), i == 0);
                        if (TWO) {
                            dot64_seq(L.R0[j], L.R1[j], xp, Sa, Sb);
                            acc2[t] = fold_term(acc2[t], block_term(mt, sa2, ma2, sb2, mb2, Sa, Sb), i == 0);
                        }
                    }
                }
                if (i + kDepth < L.nbl && L.row_ok) {  // refill this slot with block b + S*kDepth
                    const int bn = b + S * kDepth;
                    const uint8_t* p = L.m1 + rb + 128 * bn + 32 * c;
                    L.Q0[j] = ldg16(p); L.Q1[j] = ldg16(p + 16);
                    side_load<FMT>(P, L.m1, row, bn, c, L.A[j], L.B[j]);
                    if (TWO) {
                        const uint8_t* p2 = L.m2 + rb + 128 * bn + 32 * c;
                        L.R0[j] = ldg16(p2); L.R1[j] = ldg16(p2 + 16);
                        side_load<FMT>(P, L.m2, row, bn, c, L.A2[j], L.B2[j]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < TB; ++t) {
        for (int off = 1; off < 4 * S; off <<= 1) {
            acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
            if (TWO) acc2[t] += __shfl_xor_sync(0xffffffffu, acc2[t], off);
        }
    }
    if ((lane & (4 * S - 1)) == 0 && L.row_ok) {
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            if (t < nt) {
                float* o = G.out + (int64_t)s_pairs[t] * G.n;
                o[L.row] = TWO ? silu(acc[t]) * acc2[t] : acc[t];
            }
        }
    }
}

template <int FMT, bool TWO, int TB>
__global__ void __launch_bounds__(kThreads, 3) fmt4_kernel(const __grid_constant__ Fmt4Params P) {
    extern __shared__ __align__(16) uint8_t smem[];
    int* cnt = reinterpret_cast<int*>(smem);  // [E] counts then [E] item starts (general path)
    __shared__ int s_warp[33];
    __shared__ int s_bad;
    __shared__ int s_pairs[kTB];
    __shared__ int s_info[4];  // expert, tile, tokens, chunk
    __shared__ int s_pairs_key[2];
    __shared__ int s_staged_key[2];
    __shared__ FastGroup s_fast;
    __shared__ int s_items[2];
    const GroupDev& G = P.g;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0) { s_items[0] = 0; s_pairs_key[0] = -1; s_staged_key[0] = -1; }
    int* start = cnt + G.num_experts;
    if (P.fast) {
        if (warp == 0) fast_bucket(G.ids, G.n_pairs, G.num_experts, G.tiles, TB, 0, s_fast, &s_bad);
        __syncthreads();
        if (threadIdx.x == 0) s_items[1] = s_fast.start[s_fast.U];
    } else {
        block_histogram(G.ids, G.n_pairs, G.num_experts, cnt, &s_bad);
        for (int e = threadIdx.x; e < G.num_experts; e += kThreads) start[e] = ((cnt[e] + TB - 1) / TB) * G.tiles;
        __syncthreads();
        const int total = block_exclusive_scan(start, G.num_experts, s_warp);
        if (threadIdx.x == 0) s_items[1] = total;
    }
    __syncthreads();
    const int total_items = s_items[1];
    uint8_t* xs = smem + P.x_off;
    float2* meta = reinterpret_cast<float2*>(smem + P.meta_off);
    const int per_cta = (total_items + gridDim.x - 1) / gridDim.x;
    const int item_begin = blockIdx.x * per_cta;
    const int item_end = min(total_items, item_begin + per_cta);
    for (int item = item_begin; item < item_end; ++item) {
        if (P.fast) {
            if (warp == 0) {
                const FastLoc F = fast_locate(&s_fast, s_items, &G, 1, TB, item, s_pairs);
                if (lane == 0) {
                    s_info[0] = F.e; s_info[1] = F.tile; s_info[2] = F.nt; s_info[3] = F.chunk;
                    s_pairs_key[0] = F.e; s_pairs_key[1] = F.chunk;
                }
            }
        } else if (threadIdx.x == 0) {
            const int local = item;
            int lo = 0, hi = G.num_experts - 1;  // last e with start[e] <= local
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (start[mid] <= local) lo = mid; else hi = mid - 1;
            }
            const int in_e = local - start[lo];
            const int chunk = in_e / G.tiles;
            s_info[0] = lo; s_info[1] = in_e % G.tiles; s_info[2] = min(TB, cnt[lo] - chunk * TB); s_info[3] = chunk;
        }
        __syncthreads();
        const int e = s_info[0], tile = s_info[1], nt = s_info[2], chunk = s_info[3];
        FmtLane<TWO> L;
        fmt_issue<FMT, TWO>(P, e, tile, lane, warp, L);
        if (!P.fast && warp == 0 && !(s_pairs_key[0] == e && s_pairs_key[1] == chunk)) {
            warp_gather_bucket(G.ids, G.n_pairs, e, chunk * TB, nt, s_pairs);
            __syncwarp();
            if (lane == 0) { s_pairs_key[0] = e; s_pairs_key[1] = chunk; }
        }
        __syncthreads();
        // the staged rows belong to (expert, chunk): restage only when that changes
        const bool restage = !(s_staged_key[0] == e && s_staged_key[1] == chunk);
        __syncthreads();
        if (restage) {
            stage_rows(G, s_pairs, nt, xs, meta);
            if (threadIdx.x == 0) { s_staged_key[0] = e; s_staged_key[1] = chunk; }
        }
        __syncthreads();
        fmt_compute<FMT, TWO, TB>(P, L, s_pairs, nt, xs, meta, lane);
        __syncthreads();
    }
    if (blockIdx.x == 0 && s_bad > 0) {  // out-of-range ids: flag and zero their rows
        if (threadIdx.x == 0) raise_flag(P.err_flag, Q4K_ERR_EXPERT_ID);
        for (int p = 0; p < G.n_pairs; ++p) {
            if (id_valid(G.ids[p], G.num_experts)) continue;
            for (int r = threadIdx.x; r < G.n; r += kThreads) G.out[(int64_t)p * G.n + r] = 0.0f;
        }
    }
}

using Fmt4Kernel = void (*)(Fmt4Params);

template <int FMT>
Fmt4Kernel pick(bool two, int tb) {
    if (two) return tb == 1 ? fmt4_kernel<FMT, true, 1> : fmt4_kernel<FMT, true, kTB>;
    return tb == 1 ? fmt4_kernel<FMT, false, 1> : fmt4_kernel<FMT, false, kTB>;
}

}  // namespace

int num_sms();

cudaError_t launch_fmt4(int fmt, const uint8_t* w, const uint8_t* w2, uint64_t expert_stride, uint64_t s_off,
                        uint64_t b_off, int gs, int num_experts, const float* a, int64_t outer, int64_t inner,
                        const int32_t* ids, int m, int top_k, int n, int k, float* out, int* err_flag,
                        cudaStream_t stream) {
    GemvGroup S{};
    S.w = w; S.w2 = w2; S.ids = ids; S.a = a; S.outer = outer; S.inner = inner; S.out = out;
    S.num_experts = num_experts; S.m = m; S.top_k = top_k; S.n = n; S.k = k;
    Fmt4Params P{};
    P.g = group_dev(S, lg_split_for(k), kOne);
    if (P.g.n_pairs == 0) return cudaSuccess;
    P.expert_stride = (int64_t)expert_stride;
    P.gs = gs;
    if (fmt == Q4K_FMT_AFFINE4) {
        P.s_off = (int64_t)s_off;
        P.b_off = (int64_t)b_off;
    } else {  // q4tp: params after the n*k/2 code bytes, 5-bit group codes after the params
        P.s_off = (int64_t)n * (k / 2);
        P.b_off = P.s_off + 4 * (int64_t)n;
        P.cstride = (k / 32) * 5 / 8;
    }
    P.err_flag = err_flag;
    const int64_t pairs = P.g.n_pairs;
    const int tb = pairs > num_experts ? kTB : 1;
    P.tb = tb;
    P.fast = pairs <= 32 ? 1 : 0;
    const int ints = P.fast ? 0 : 2 * num_experts;
    const int64_t per_tok = (int64_t)(k / 64) * kPairBytes + (int64_t)(k / 32) * 8;
    int off = ((ints * 4) + 15) & ~15;
    P.x_off = off;
    off += (int)((int64_t)(k / 64) * kPairBytes * tb);
    off = (off + 15) & ~15;
    P.meta_off = off;
    off += (k / 32) * 8 * tb;
    const size_t smem = (size_t)off;
    if (per_tok * tb > 200 * 1024) return cudaErrorInvalidValue;
    Fmt4Kernel kern = fmt == Q4K_FMT_AFFINE4 ? pick<Q4K_FMT_AFFINE4>(w2 != nullptr, tb) : pick<Q4K_FMT_Q4TP>(w2 != nullptr, tb);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
    int64_t max_items = pairs * P.g.tiles;
    int64_t grid = (int64_t)num_sms() * per_sm;
    if (grid > max_items) grid = max_items;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

}  // namespace q4k

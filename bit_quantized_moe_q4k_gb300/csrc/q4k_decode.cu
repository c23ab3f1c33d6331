// q4k_decode.cu -- a decode-size MoE layer (a few tokens) in ONE launch, with every weight
// byte the layer touches on its way into shared memory before any arithmetic starts.
//
// What it computes (moeflux expert_forward.rs: gate, up, SwiGLU, down, then the batched
// combine y = h_mid + sum_s w_s * expert_out_s + g * shared_out; ferrum-kernels
// q4_k_moe_id_gemv_batched.rs for each projection): the same as the two-launch layer of
// q4k_gemv.cu, bit for bit. Every output row is summed in the order all kernels use (each
// lane's block terms folded left to right, then the xor shuffles over its lanes; see
// block_term), the down input is staged with the same arithmetic (per 32-element sub-block:
// max|x|, X = rint(x * 32767 / max), sum X), and the combine adds the slots in order.
//
// How (GB300 design). One CTA per SM, 16 warps, up to ~220 KB of shared memory each, so a
// decode layer's touched weights (Qwen3-MoE-like m = 1: 24 MB) fit in the grid's shared
// memory at once and all of them are requested from HBM within the first microsecond:
//  1. Every CTA buckets the ids (one warp), stages the tokens' h_post rows, and one thread
//     issues bulk copies (cp.async.bulk, mbarrier completion) of ALL the CTA's weight bytes:
//     its gate|up items (32 rows of one expert's gate and up slabs, in 8-row slices with an
//     mbarrier each), then its down rows (one contiguous range of hidden rows of every expert
//     of the batch and of the shared expert). Before waiting for the previous kernel it
//     already starts its share of the shared expert's slabs into L2.
//  2. Gate|up: rows stream through the warps as their slices land. A lane owns one 64-weight
//     group of one block of every row it sees and keeps that block's activations in
//     registers, so shared memory only delivers the weights (the activation planes are 2.2x
//     the bytes of the weights they meet, and re-reading them per row left the kernel bound
//     by shared-memory bandwidth). The warp that completes an item forms silu(g) * u for its
//     32 rows -- one 32-element sub-block of the down input -- quantizes that sub-block to the
//     staged 16-bit form, stores it to the workspace and publishes the item's flag.
//  3. Down: each CTA waits for every item's flag (the one hand-off between CTAs), copies the
//     staged down inputs of all pairs from L2, and streams its hidden rows of every expert
//     through the warps the same way.
//  4. Combine: the CTA holds those rows of every expert, so it forms y for them itself: no
//     second hand-off, no counters, no atomics.
// CTA 0 advances the generation word of the tagged flags (q4k_sync.cuh) while it waits for
// the items. Every wait is bounded; the grid is one CTA per SM, all resident at once.
#include <algorithm>
#include <cstdlib>

#include "q4k_gemv_common.cuh"
#include "q4k_sm100.cuh"
#include "q4k_sync.cuh"

namespace q4k {

namespace {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecItemRows = 32;                        // gate|up rows per item: one down-input sub-block
constexpr int kDecSliceRows = 8;                        // rows per bulk copy (one mbarrier each)
constexpr int kDecSlices = kDecItemRows / kDecSliceRows;
constexpr int kDecMaxItems = 8;                         // gate|up items per CTA
constexpr int kDecMaxTokens = 4;                        // m
constexpr int kDecMaxPairs = 32;                        // routed pairs (one warp buckets them)
constexpr int kDecRowTile = 8;                          // hidden rows per down tile
constexpr int kDecBarB = kDecMaxItems * kDecSlices;     // the down rows' mbarrier
constexpr int kDecMaxCtas = 1024;                       // start-tag words

struct DecodeParams {
    GroupDev a[kMaxGroups];   // gate|up + SwiGLU: routed experts, shared expert (same k = hidden)
    GroupDev b[kMaxGroups];   // down: routed, shared (both with the routed group's lane split)
    int n_groups, m, has_shared;
    uint8_t* stg_planes[kMaxGroups];  // staged down inputs in the workspace: row r's planes at
    float2* stg_meta[kMaxGroups];     // + r * (k/64)*144, its (delta, sum X) at + r * (k/32)
    // dynamic shared memory layout (byte offsets)
    int off_x, off_xmeta;             // staged h_post rows of the m tokens
    int off_gu;                       // g and u of the items: [item][pair][gate|up][32] floats
    int gu_pairs;
    int off_eout;                     // down rows: [routed pairs, then shared tokens][rows_max]
    int off_hmid;                     // h_mid of the CTA's rows: [token][rows_max]
    int off_a, item_bytes;            // gate|up tiles: item j at off_a + j*item_bytes (gate, then up)
    int off_act[kMaxGroups], off_actmeta[kMaxGroups];  // staged down inputs (over the gate|up tiles)
    int off_b;                        // down rows of the CTA
    int rows_max, n_row_tiles;
    CombineSpec cb;
    uint64_t* gen;                    // generation word
    uint64_t* cta_tag;                // [kDecMaxCtas] the tag each CTA read
    uint64_t* flags;                  // [cap_flags] one per gate|up item
    int cap_flags;
    const uint8_t* pf[3];             // shared expert slabs started into L2 before the wait
    uint64_t pf_bytes[3];
    int* err_flag;
    uint64_t wait_ns;
};

__device__ __forceinline__ uint4 lds16(const uint8_t* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

// Lanes of a row stream. A row of k weights has nb = k/256 blocks, which item_compute splits
// over S = 1 << lg lanes (block b to lane sl = b % S, i = b / S) times 4 (the 64-weight group
// c). Here they are laid out side by side: a slot of L = 4*S*NI lanes, NI = ceil(nb / S), in
// which lane c | sl << 2 | i << (2 + lg) owns group c of block b = sl + S*i of every row that
// passes (lanes with b >= nb hold nothing), with that block's staged activations in
// registers. A row's sum is then formed in the fixed order of block_term: the fold over i by
// NI - 1 shuffles up the slot, then the xor shuffles over c and sl.
struct RowLanes {
    int S, nb, NI, L, NS, slot, c, sl, i, b;
    bool live;  // the lane belongs to a slot
};

__host__ __device__ __forceinline__ int row_slot_lanes(int k, int lg) {
    const int S = 1 << lg, nb = k / kQK;
    return 4 * S * ((nb + S - 1) / S);
}

__device__ __forceinline__ RowLanes row_lanes_of(int k, int lg, int lane) {
    RowLanes R;
    R.S = 1 << lg;
    R.nb = k / kQK;
    R.NI = (R.nb + R.S - 1) / R.S;
    R.L = 4 * R.S * R.NI;
    R.NS = 32 / R.L;
    R.slot = lane / R.L;
    const int w = lane - R.slot * R.L;
    R.c = w & 3;
    R.sl = (w >> 2) & (R.S - 1);
    R.i = w >> (2 + lg);
    R.b = R.sl + R.S * R.i;
    R.live = R.slot < R.NS;
    return R;
}

// The lane's block of a staged token row (planes and (delta, sum X) pairs in shared memory).
__device__ __forceinline__ void load_x(const uint8_t* xrow, const float2* xmeta, const RowLanes& R, uint32_t (&x)[32],
                                       float4& mt) {
    const uint8_t* xp = xrow + (4 * R.b + R.c) * kPairBytes;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const uint4 v = lds16(xp + 16 * u);
        x[4 * u] = v.x; x[4 * u + 1] = v.y; x[4 * u + 2] = v.z; x[4 * u + 3] = v.w;
    }
    const uint4 m4 = lds16(reinterpret_cast<const uint8_t*>(xmeta + 8 * R.b + 2 * R.c));
    mt = make_float4(__uint_as_float(m4.x), __uint_as_float(m4.y), __uint_as_float(m4.z), __uint_as_float(m4.w));
}

// The row's sum from every lane's term T: valid in the slot's lanes of the last stage
// (i == NI - 1); lanes outside every slot pass junk that no slot reads.
__device__ __forceinline__ float row_sum(float T, const RowLanes& R) {
    float F = T;
    for (int d = 1; d < R.NI; ++d) {
        const float prev = __shfl_up_sync(0xffffffffu, F, 4 * R.S);
        if (R.i == d) F = R.b < R.nb ? __fadd_rn(prev, T) : prev;
    }
    for (int off = 1; off < 4 * R.S; off <<= 1) F += __shfl_xor_sync(0xffffffffu, F, off);
    return F;
}

// Lane (c = 0, sl = 0) of the last stage of a live slot: the one that holds the row's sum.
__device__ __forceinline__ bool row_owner(const RowLanes& R) {
    return R.live && R.i == R.NI - 1 && R.c == 0 && R.sl == 0;
}

// Block-wide: wait until f1[j] == tag for j < n1 and f2[j] == tag for j < n2 (acquire loads;
// the closing barrier passes the acquisitions on to every thread). False once limit_ns has
// passed. Uniform over the block.
__device__ bool dec_wait_tags(const uint64_t* f1, int n1, const uint64_t* f2, int n2, uint64_t tag,
                              uint64_t limit_ns) {
    const int n = n1 + n2;
    int j = threadIdx.x;
    const uint64_t t0 = sm100::global_timer_ns();
    for (;;) {
        uint64_t v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int jj = j + u * kDecThreads;
            v[u] = jj < n ? ld_acquire_u64(jj < n1 ? f1 + jj : f2 + (jj - n1)) : tag;
        }
        int seen = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (v[u] != tag) break;
            ++seen;
        }
        j += seen * kDecThreads;
        if (__syncthreads_and(j >= n)) return true;
        const bool late = sm100::global_timer_ns() - t0 > limit_ns;
        if (__syncthreads_or(late)) return false;
    }
}

// The bucketing of the routed pairs (one warp; lane p holds pair p): buckets by increasing
// expert id, members in increasing pair order.
struct DecBuckets {
    int U;                      // buckets
    int e[kDecMaxPairs];        // expert of bucket r
    int cnt[kDecMaxPairs];      // its pairs
    uint8_t plist[kDecMaxPairs][kDecMaxPairs];  // its pairs, increasing
    unsigned valid;             // pairs with an id in [0, num_experts)
    int bad;                    // pairs with an id outside
};

__device__ __forceinline__ void dec_bucket(const int32_t* ids, int n_pairs, int num_experts, DecBuckets& B) {
    const int lane = threadIdx.x & 31;
    int key = -1;
    if (lane < n_pairs) {
        const int32_t e = ids[lane];
        key = id_valid(e, num_experts) ? e : -1;
    }
    const bool valid = key >= 0;
    const unsigned vmask = __ballot_sync(0xffffffffu, valid);
    const unsigned badm = __ballot_sync(0xffffffffu, lane < n_pairs && !valid);
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const bool leader = valid && (__ffs(peers) - 1) == lane;
    const unsigned leaders = __ballot_sync(0xffffffffu, leader);
    int rank = 0;
    for (unsigned rest = leaders; rest; rest &= rest - 1u) {  // uniform over the warp
        const int kj = __shfl_sync(0xffffffffu, key, __ffs(rest) - 1);
        rank += kj < key ? 1 : 0;
    }
    if (leader) {
        B.e[rank] = key;
        B.cnt[rank] = __popc(peers);
    }
    if (valid) B.plist[rank][__popc(peers & ((1u << lane) - 1u))] = (uint8_t)lane;
    if (lane == 0) {
        B.U = __popc(leaders);
        B.valid = vmask;
        B.bad = __popc(badm);
    }
    __syncwarp();
}

__global__ void __launch_bounds__(kDecThreads, 1) decode_layer_kernel(const __grid_constant__ DecodeParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ DecBuckets s_b;
    __shared__ __align__(8) uint64_t s_bar[kDecBarB + 1];
    __shared__ int s_done[kDecMaxItems];   // rows of each gate|up item finished (per pair)
    __shared__ int s_icnt[kDecMaxItems];   // pairs of each gate|up item of the CTA
    __shared__ uint8_t s_itok[kDecMaxItems][kDecMaxPairs];  // token of each pair slot
    __shared__ int s_pmax;
    __shared__ float s_w[kDecMaxPairs];    // routing weights
    __shared__ float s_g[kDecMaxTokens];   // shared-expert gate factor per token
    __shared__ uint64_t s_tag;
    __shared__ volatile int s_abort, s_never;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = gridDim.x, cta = blockIdx.x;
    const GroupDev& A0 = P.a[0];
    const GroupDev& B0 = P.b[0];
    const int H = B0.n, T = A0.top_k, m = P.m, n_pairs = A0.n_pairs;

    // the shared expert's slabs do not depend on the previous kernel: start this CTA's share
    // of them into L2 before waiting for it (L2 is the coherence point, so this cannot stale)
    if (tid < 3 && P.pf[tid]) {
        const uint64_t units = P.pf_bytes[tid] / 16;
        const uint64_t u0 = units * cta / G, u1 = units * (cta + 1) / G;
        for (uint64_t u = u0; u < u1; u += 4096) {
            const uint64_t n = u1 - u < 4096 ? u1 - u : 4096;
            bulk_prefetch_l2(P.pf[tid] + u * 16, (uint32_t)(n * 16));
        }
    }
    if (tid == 0) {
        for (int i = 0; i <= kDecBarB; ++i) sm100::mbar_init(&s_bar[i], 1);
        sm100::fence_mbar_init();
        s_abort = 0;
        s_never = 0;
    }
    if (tid < kDecMaxItems) s_done[tid] = 0;

    // ids, h_post, h_mid and the generation word may come from earlier kernels of the stream
    pdl_wait();
    pdl_launch_dependents();

    // hidden rows of this CTA in the down phase (independent of the ids)
    const int rt0 = (int)((int64_t)cta * P.n_row_tiles / G), rt1 = (int)((int64_t)(cta + 1) * P.n_row_tiles / G);
    const int row_lo = rt0 * kDecRowTile, row_hi = min(H, rt1 * kDecRowTile);
    const int rows_c = max(0, row_hi - row_lo);
    uint8_t* xs0 = smem + P.off_x;
    float2* xm0 = reinterpret_cast<float2*>(smem + P.off_xmeta);
    const int ka = A0.k;
    const int64_t xrow = (int64_t)(ka / 64) * kPairBytes;
    float* hmid_s = reinterpret_cast<float*>(smem + P.off_hmid);

    if (warp == 0) {
        dec_bucket(A0.ids, n_pairs, A0.num_experts, s_b);
    } else if (warp == 1) {
        if (lane == 0) {
            const uint64_t tag = next_tag(ld_relaxed_u64(P.gen));
            s_tag = tag;
            st_relaxed_u64(P.cta_tag + cta, tag);  // this CTA has read the generation
        }
        if (lane < n_pairs) s_w[lane] = P.cb.weights[lane];
        if (lane < m && P.has_shared)
            s_g[lane] = P.cb.shared_mode == Q4K_SHARED_SIGMOID ? 1.0f / (1.0f + expf(-P.cb.shared_gate[lane])) : 1.0f;
        for (int i = lane; i < m * rows_c; i += 32) {
            const int t = i / rows_c, rl = i % rows_c;
            hmid_s[t * P.rows_max + rl] = P.cb.h_mid[(int64_t)t * H + row_lo + rl];
        }
    } else {
        // the m tokens' h_post rows, staged once for every gate|up item of the CTA
        for (int t = 0; t < m; ++t)
            stage_row<0, kDecThreads - 64>(A0.a + (int64_t)t * A0.outer, ka, xs0 + t * xrow, xm0 + t * (ka / 32),
                                           tid - 64);
    }
    __syncthreads();

    // ---- the gate|up items of this CTA: routed buckets (tiles of 32 rows), then the shared expert
    const int U = s_b.U;
    const int ta0 = A0.n / kDecItemRows, ta1 = P.has_shared ? P.a[1].n / kDecItemRows : 0;
    const int na = U * ta0 + ta1;
    const int a0 = (int)((int64_t)cta * na / G), a1 = (int)((int64_t)(cta + 1) * na / G);
    const int nitems = a1 - a0;
    const bool fits = nitems <= kDecMaxItems && na <= P.cap_flags;
    const uint64_t tag = s_tag;
    // locate an item: group, bucket (routed) , expert, row tile
    auto locate = [&](int item, int& g, int& r, int& e, int& tile) {
        if (item < U * ta0) {
            g = 0; r = item / ta0; tile = item % ta0; e = s_b.e[r];
        } else {
            g = 1; r = 0; tile = item - U * ta0; e = 0;
        }
    };
    const int units_b = U + (P.has_shared ? 1 : 0);
    // the CTA's items: pairs, and the token of each pair slot
    if (warp == 1 && fits) {
        int pm = 0;
        for (int j = 0; j < nitems; ++j) {
            int g, r, e, tile;
            locate(a0 + j, g, r, e, tile);
            const int cnt = g == 0 ? s_b.cnt[r] : m;
            if (lane < cnt) s_itok[j][lane] = (uint8_t)(g == 0 ? s_b.plist[r][lane] / T : lane);
            if (lane == 0) s_icnt[j] = cnt;
            pm = max(pm, cnt);
        }
        if (lane == 0) s_pmax = pm;
    }
    int64_t boff_sh = 0;  // byte offset of the shared expert's down rows in region B
    if (tid == 0 && fits) {
        // every weight byte of the CTA, in the order it is needed
        for (int j = 0; j < nitems; ++j) {
            int g, r, e, tile;
            locate(a0 + j, g, r, e, tile);
            const GroupDev& A = P.a[g];
            const uint32_t bytes = (uint32_t)(kDecSliceRows * A.nb01);
            uint8_t* dst = smem + P.off_a + (int64_t)j * P.item_bytes;
            for (int s = 0; s < kDecSlices; ++s) {
                const int64_t row0 = (int64_t)tile * kDecItemRows + s * kDecSliceRows;
                const int64_t src = (int64_t)e * A.nb02 + row0 * A.nb01;
                uint64_t* bar = &s_bar[j * kDecSlices + s];
                sm100::mbar_arrive_expect_tx(bar, 2 * bytes);
                sm100::bulk_g2s(dst + (s * kDecSliceRows) * A.nb01, A.w + src, bytes, bar);
                sm100::bulk_g2s(dst + (kDecItemRows + s * kDecSliceRows) * A.nb01, A.w2 + src, bytes, bar);
            }
        }
        if (rows_c > 0) {
            uint32_t total = 0;
            for (int u = 0; u < units_b; ++u) total += (uint32_t)(rows_c * P.b[u < U ? 0 : 1].nb01);
            sm100::mbar_arrive_expect_tx(&s_bar[kDecBarB], total);
            int64_t off = 0;
            for (int u = 0; u < units_b; ++u) {
                const int g = u < U ? 0 : 1;
                const GroupDev& B = P.b[g];
                const int e = g == 0 ? s_b.e[u] : 0;
                const uint32_t bytes = (uint32_t)(rows_c * B.nb01);
                sm100::bulk_g2s(smem + P.off_b + off, B.w + (int64_t)e * B.nb02 + (int64_t)row_lo * B.nb01, bytes,
                                &s_bar[kDecBarB]);
                off += bytes;
            }
        }
    }
    boff_sh = (int64_t)U * rows_c * B0.nb01;
    __syncthreads();  // the item tables (and the issue, which runs before any wait in its warp)

    // ---- gate|up rows, streamed through the warps' slots: stream sigma takes the rows
    // rho = sigma, sigma + ns, ... of the CTA's items in (item, slice, gate|up, row) order, so all
    // streams move through the slices in the order they land; each row once per pair slot
    // pi < pmax (slots beyond the item's pairs do nothing)
    {
        const RowLanes R = row_lanes_of(ka, A0.lg_split, lane);
        const int ns = kDecWarps * R.NS;
        const int sigma = warp * R.NS + R.slot;
        const int NR = fits ? nitems * 2 * kDecItemRows : 0;
        const int nrho = (R.live && sigma < NR) ? (NR - sigma + ns - 1) / ns : 0;
        const int nrho_max = __reduce_max_sync(0xffffffffu, nrho);
        const int pmax = s_pmax;
        float* gu = reinterpret_cast<float*>(smem + P.off_gu);
        uint32_t x[32];
        float4 mt = make_float4(0.f, 0.f, 0.f, 0.f);
        int xkey = -1, last_bar = -1;
        for (int t = 0; t < nrho_max; ++t) {
            const int rho = sigma + t * ns;
            const bool rvalid = t < nrho;
            const int j = rho >> 6, s = (rho >> 4) & 3, slab = (rho >> 3) & 1, rin = (rho & 7) + 8 * s;
            bool landed = true;
            if (rvalid && j * kDecSlices + s != last_bar) {
                last_bar = j * kDecSlices + s;
                landed = mbar_wait_for(&s_bar[last_bar], 0, &s_abort, P.wait_ns);
            }
            if (!__all_sync(0xffffffffu, landed)) {
                s_abort = 1;
                break;
            }
            const int cnt = rvalid ? s_icnt[j] : 0;
            uint4 H = make_uint4(0, 0, 0, 0), Q0 = H, Q1 = H;
            if (rvalid && R.b < R.nb) {
                const uint8_t* p = smem + P.off_a + (int64_t)j * P.item_bytes +
                                   (int64_t)(slab * kDecItemRows + rin) * A0.nb01 + R.b * kBlockBytes;
                H = lds16(p);
                Q0 = lds16(p + 16 + 32 * R.c);
                Q1 = lds16(p + 32 + 32 * R.c);
            }
            float sa, ma, sb, mb;
            block_scales(H, R.c, sa, ma, sb, mb);
            int trig = -1;
            for (int pi = 0; pi < pmax; ++pi) {
                const bool work = pi < cnt;
                float T = 0.0f;
                if (work && R.b < R.nb) {
                    const int tok = s_itok[j][pi];
                    if (tok != xkey) {
                        load_x(xs0 + tok * xrow, xm0 + tok * (ka / 32), R, x, mt);
                        xkey = tok;
                    }
                    int Sa, Sb;
                    dot64_regs(Q0, Q1, x, Sa, Sb);
                    T = block_term(mt, sa, ma, sb, mb, Sa, Sb);
                }
                const float v = row_sum(T, R);
                if (work && row_owner(R)) {
                    gu[((j * P.gu_pairs + pi) * 2 + slab) * kDecItemRows + rin] = v;
                    __threadfence_block();
                    if (atomicAdd(&s_done[j], 1) == 2 * kDecItemRows * cnt - 1) trig = j;
                }
            }
            // an item whose rows are all done: the warp stages its 32 rows of the down input
            for (unsigned tm = __ballot_sync(0xffffffffu, trig >= 0); tm; tm &= tm - 1u) {
                const int jj = __shfl_sync(0xffffffffu, trig, __ffs(tm) - 1);
                __syncwarp();
                __threadfence_block();
                int gg, rr, ee, tt;
                locate(a0 + jj, gg, rr, ee, tt);
                const int cc = s_icnt[jj];
                const GroupDev& B = P.b[gg];
                const int kb = B.k;
                const int64_t pb = (int64_t)(kb / 64) * kPairBytes;
                for (int pp = 0; pp < cc; ++pp) {
                    const int p = gg == 0 ? s_b.plist[rr][pp] : pp;
                    const float gv = gu[((jj * P.gu_pairs + pp) * 2 + 0) * kDecItemRows + lane];
                    const float uv = gu[((jj * P.gu_pairs + pp) * 2 + 1) * kDecItemRows + lane];
                    const float a = silu(gv) * uv;
                    float mx = fabsf(a);
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                    int X = 0;
                    if (mx > 0.0f) {
                        const float inv = 32767.0f / mx;
                        X = max(-32767, min(32767, __float2int_rn(a * inv)));
                    }
                    int sx = X;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) sx += __shfl_xor_sync(0xffffffffu, sx, off);
                    uint8_t* planes = P.stg_planes[gg] + (int64_t)p * pb + (tt >> 1) * kPairBytes + (tt & 1) * 64;
                    planes[lane] = (uint8_t)(X & 0xFF);
                    planes[32 + lane] = (uint8_t)((X >> 8) & 0xFF);
                    if (lane == 0) P.stg_meta[gg][(int64_t)p * (kb / 32) + tt] = make_float2(mx / 32767.0f, (float)sx);
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) st_release_u64(P.flags + a0 + jj, tag);
            }
        }
    }
    __syncthreads();  // the gate|up tiles' space is free for the staged down inputs

    // ---- one hand-off: every gate|up item of the launch (CTA 0 also confirms that every CTA
    // read the generation word, then advances it)
    bool ok = fits && !s_abort;
    if (ok) ok = dec_wait_tags(P.flags, na, P.cta_tag, cta == 0 ? G : 0, tag, P.wait_ns);
    if (ok && cta == 0 && tid == 0) st_relaxed_u64(P.gen, tag);
    if (ok) {
        // staged down inputs of every pair (routed, then the shared expert's tokens), from L2:
        // both groups' rows (planes, then (delta, sum X) pairs, contiguous per group in the
        // workspace and in shared memory) in one pass of loads
        const int64_t n0 = (int64_t)n_pairs * ((B0.k / 64) * kPairBytes + (B0.k / 32) * 8) / 16;
        const int64_t n1 = P.has_shared ? (int64_t)m * ((P.b[1].k / 64) * kPairBytes + (P.b[1].k / 32) * 8) / 16 : 0;
        const uint4* s0 = reinterpret_cast<const uint4*>(P.stg_planes[0]);
        const uint4* s1 = reinterpret_cast<const uint4*>(P.stg_planes[1]);
        uint4* d0 = reinterpret_cast<uint4*>(smem + P.off_act[0]);
        uint4* d1 = reinterpret_cast<uint4*>(smem + P.off_act[1]);
        for (int64_t i0 = 0; i0 < n0 + n1; i0 += 8 * kDecThreads) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t i = i0 + u * kDecThreads + tid;
                if (i < n0 + n1) v[u] = __ldcg(i < n0 ? s0 + i : s1 + (i - n0));
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t i = i0 + u * kDecThreads + tid;
                if (i < n0) d0[i] = v[u];
                else if (i < n0 + n1) d1[i - n0] = v[u];
            }
        }
        ok = __syncthreads_and(rows_c == 0 || mbar_wait_for(&s_bar[kDecBarB], 0, &s_abort, P.wait_ns));
    }

    // ---- down rows of every expert (and the shared expert) for the CTA's rows of hidden,
    // streamed through the warps' slots: a pass over the routed units (and the shared expert
    // when its rows have the same length), then one over the shared expert otherwise. Stream
    // sigma takes a contiguous range of the pass's (unit, pair slot, row) items, so its lanes
    // reload their activations only when the pair changes.
    float* eout = reinterpret_cast<float*>(smem + P.off_eout);
    if (ok && rows_c > 0) {
        const bool same_k = !P.has_shared || P.b[1].k == B0.k;
        for (int pass = 0; pass < (same_k ? 1 : 2); ++pass) {
            const int u_lo = pass == 0 ? 0 : U;
            const int u_hi = pass == 0 ? (same_k ? units_b : U) : units_b;
            const int kb = pass == 0 ? B0.k : P.b[1].k;
            const RowLanes R = row_lanes_of(kb, B0.lg_split, lane);
            const int ns = kDecWarps * R.NS;
            const int sigma = warp * R.NS + R.slot;
            int pmax = 1;
            for (int u = u_lo; u < u_hi; ++u) pmax = max(pmax, u < U ? s_b.cnt[u] : m);
            const int NQ = (u_hi - u_lo) * pmax * rows_c;
            const int q0 = R.live ? (int)((int64_t)sigma * NQ / ns) : 0;
            const int nq = R.live ? (int)((int64_t)(sigma + 1) * NQ / ns) - q0 : 0;
            const int nq_max = __reduce_max_sync(0xffffffffu, nq);
            uint32_t x[32];
            float4 mt = make_float4(0.f, 0.f, 0.f, 0.f);
            int xkey = -1;
            // the lane's item: unit, pair slot, row (advanced one by one)
            int rl = q0 % rows_c, pi = (q0 / rows_c) % pmax, u = u_lo + q0 / rows_c / pmax;
            for (int t = 0; t < nq_max; ++t) {
                const bool valid = t < nq;
                const int g = u < U ? 0 : 1;
                const int cnt = g == 0 ? s_b.cnt[u] : m;
                const bool work = valid && pi < cnt;
                const int p = work ? (g == 0 ? s_b.plist[u][pi] : pi) : 0;
                float T = 0.0f;
                if (work && R.b < R.nb) {
                    const int key = u * kDecMaxPairs + pi;
                    if (key != xkey) {
                        load_x(smem + P.off_act[g] + (int64_t)p * (kb / 64) * kPairBytes,
                               reinterpret_cast<const float2*>(smem + P.off_actmeta[g]) + (int64_t)p * (kb / 32), R, x, mt);
                        xkey = key;
                    }
                    const GroupDev& B = P.b[g];
                    const int64_t boff = g == 0 ? (int64_t)u * rows_c * B.nb01 : boff_sh;
                    const uint8_t* w = smem + P.off_b + boff + (int64_t)rl * B.nb01 + R.b * kBlockBytes;
                    const uint4 H = lds16(w), Q0 = lds16(w + 16 + 32 * R.c), Q1 = lds16(w + 32 + 32 * R.c);
                    float sa, ma, sb, mb;
                    block_scales(H, R.c, sa, ma, sb, mb);
                    int Sa, Sb;
                    dot64_regs(Q0, Q1, x, Sa, Sb);
                    T = block_term(mt, sa, ma, sb, mb, Sa, Sb);
                }
                const float v = row_sum(T, R);
                if (work && row_owner(R)) eout[(g == 0 ? p : n_pairs + p) * P.rows_max + rl] = v;
                if (valid) {
                    if (++rl == rows_c) {
                        rl = 0;
                        if (++pi == pmax) { pi = 0; ++u; }
                    }
                }
            }
        }
    }
    __syncthreads();

    // ---- combine of the CTA's rows: y = h_mid + sum_s w_s * eout_s (slot order) + g * shared
    if (ok) {
        for (int i = tid; i < m * rows_c; i += kDecThreads) {
            const int t = i / rows_c, rl = i % rows_c;
            float acc = hmid_s[t * P.rows_max + rl];
            for (int s = 0; s < T; ++s) {
                const int p = t * T + s;
                if ((s_b.valid >> p) & 1u) acc = fmaf(s_w[p], eout[p * P.rows_max + rl], acc);
            }
            if (P.has_shared) acc = fmaf(s_g[t], eout[(n_pairs + t) * P.rows_max + rl], acc);
            P.cb.y[(int64_t)t * H + row_lo + rl] = acc;
        }
    }

    // every bulk copy this CTA started lands before it leaves (also after a wait gave up)
    if (tid == 0 && fits) {
        for (int j = 0; j < nitems; ++j)
            for (int s = 0; s < kDecSlices; ++s) mbar_wait_for(&s_bar[j * kDecSlices + s], 0, &s_never, sm100::kWaitNs);
        if (rows_c > 0) mbar_wait_for(&s_bar[kDecBarB], 0, &s_never, sm100::kWaitNs);
    }
    if (tid == 0) {
        if (!fits) raise_flag(P.err_flag, Q4K_ERR_LIMIT);
        else if (!ok) raise_flag(P.err_flag, Q4K_ERR_TIMEOUT);
        if (cta == 0 && s_b.bad) raise_flag(P.err_flag, Q4K_ERR_EXPERT_ID);
    }
}

// ------------------------------------------------------------------------------------------
struct DecPlan {
    bool ok;
    int max_items, rows_max, n_row_tiles, na_max, gu_pairs, item_bytes;
    int off_x, off_xmeta, off_gu, off_eout, off_hmid, off_a, off_b, off_act[2], off_actmeta[2];
    size_t smem;
};

int64_t align_to(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// The shared-memory plan for these sizes on a grid of `grid` CTAs, for the most buckets the
// ids can make (every routed pair a different expert).
DecPlan dec_plan(int m, int top_k, int num_experts, int hidden, int inter, int shared_inter, int grid,
                 size_t smem_cap) {
    DecPlan D{};
    const int P = m * top_k;
    if (m < 1 || m > kDecMaxTokens || P > kDecMaxPairs || grid < 1 || grid > kDecMaxCtas) return D;
    if (hidden % kQK || inter % kQK || shared_inter % kQK) return D;
    // every row must fit one warp's slot of lanes (the row streams)
    const int lg_b = lg_split_for(inter);
    if (row_slot_lanes(hidden, lg_split_for(hidden)) > 32 || row_slot_lanes(inter, lg_b) > 32 ||
        (shared_inter > 0 && row_slot_lanes(shared_inter, lg_b) > 32))
        return D;
    const int umax = std::min(P, num_experts);
    const bool sh = shared_inter > 0;
    D.na_max = umax * (inter / kDecItemRows) + (sh ? shared_inter / kDecItemRows : 0);
    D.max_items = (D.na_max + grid - 1) / grid;
    if (D.max_items > kDecMaxItems) return D;
    D.n_row_tiles = (hidden + kDecRowTile - 1) / kDecRowTile;
    D.rows_max = (D.n_row_tiles + grid - 1) / grid * kDecRowTile;
    const int64_t nb01_a = (int64_t)(hidden / kQK) * kBlockBytes;
    const int64_t nb01_b0 = (int64_t)(inter / kQK) * kBlockBytes;
    const int64_t nb01_b1 = sh ? (int64_t)(shared_inter / kQK) * kBlockBytes : 0;
    D.item_bytes = (int)(2 * kDecItemRows * nb01_a);
    D.gu_pairs = P;
    int64_t off = 0;
    D.off_x = (int)off;      off += (int64_t)m * (hidden / 64) * kPairBytes;
    off = align_to(off, 16);
    D.off_xmeta = (int)off;  off += (int64_t)m * (hidden / 32) * 8;
    off = align_to(off, 16);
    D.off_gu = (int)off;     off += (int64_t)D.max_items * D.gu_pairs * 2 * kDecItemRows * 4;
    off = align_to(off, 16);
    D.off_eout = (int)off;   off += (int64_t)(P + (sh ? m : 0)) * D.rows_max * 4;
    off = align_to(off, 16);
    D.off_hmid = (int)off;   off += (int64_t)m * D.rows_max * 4;
    off = align_to(off, 128);
    D.off_a = (int)off;
    // staged down inputs (after the gate|up tiles are done with, in their space)
    int64_t so = off;
    D.off_act[0] = (int)so;     so += (int64_t)P * (inter / 64) * kPairBytes;
    D.off_actmeta[0] = (int)so; so += (int64_t)P * (inter / 32) * 8;
    D.off_act[1] = (int)so;     so += sh ? (int64_t)m * (shared_inter / 64) * kPairBytes : 0;
    D.off_actmeta[1] = (int)so; so += sh ? (int64_t)m * (shared_inter / 32) * 8 : 0;
    off = std::max<int64_t>(off + (int64_t)D.max_items * D.item_bytes, so);
    off = align_to(off, 128);
    D.off_b = (int)off;
    off += (int64_t)D.rows_max * (umax * nb01_b0 + nb01_b1);
    D.smem = (size_t)off;
    D.ok = D.smem <= smem_cap;
    return D;
}

bool g_dec_attr_set[64] = {};
size_t g_dec_cap[64] = {};

// Dynamic shared memory a CTA of the kernel may use on the current device (0 on error).
size_t dec_smem_cap(int dev) {
    if (dev < 0 || dev >= 64) return 0;
    if (!g_dec_attr_set[dev]) {
        int optin = 0;
        if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
        cudaFuncAttributes fa{};
        if (cudaFuncGetAttributes(&fa, decode_layer_kernel) != cudaSuccess) return 0;
        const size_t cap = optin > (int)fa.sharedSizeBytes ? (size_t)optin - fa.sharedSizeBytes : 0;
        if (cudaFuncSetAttribute(decode_layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cap) !=
            cudaSuccess)
            return 0;
        g_dec_cap[dev] = cap;
        g_dec_attr_set[dev] = true;
    }
    return g_dec_cap[dev];
}

}  // namespace

// Words of the sync area the kernel uses: after the single-launch layer's head (generation word,
// counter-set headers and counters, which this kernel leaves alone), kDecMaxCtas start tags and
// one flag per gate|up item (at most one bucket per routed pair).
size_t layer_decode_sync_words(int m, int top_k, int hidden, int inter, int shared_inter) {
    const int64_t na = (int64_t)m * top_k * (inter / kDecItemRows) + shared_inter / kDecItemRows;
    return layer_sync_head_words(hidden) + (size_t)kDecMaxCtas + (size_t)na;
}

bool layer_decode_fits(int m, int top_k, int num_experts, int hidden, int inter, int shared_inter) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const size_t cap = dec_smem_cap(dev);
    if (cap == 0) {
        cudaGetLastError();
        return false;
    }
    return dec_plan(m, top_k, num_experts, hidden, inter, shared_inter, num_sms(), cap).ok;
}

cudaError_t launch_layer_decode(const GemvGroup* gu, const GemvGroup* dn, int n_groups, const CombineSpec& cb,
                                uint64_t* sync, size_t sync_words, uint8_t* const* stage, int* err_flag,
                                cudaStream_t stream) {
    if (n_groups < 1 || n_groups > kMaxGroups || !sync || !stage[0] || (n_groups > 1 && !stage[1]))
        return cudaErrorNotSupported;
    const int m = gu[0].m, top_k = gu[0].top_k, E = gu[0].num_experts;
    const int hidden = gu[0].k, inter = gu[0].n, sinter = n_groups > 1 ? gu[1].n : 0;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const size_t cap = dec_smem_cap(dev);
    if (cap == 0) return cudaErrorNotSupported;
    const int grid = std::min(num_sms(), kDecMaxCtas);
    const DecPlan D = dec_plan(m, top_k, E, hidden, inter, sinter, grid, cap);
    if (!D.ok) return cudaErrorNotSupported;
    const size_t head = layer_sync_head_words(hidden);
    if (sync_words < head + (size_t)kDecMaxCtas + (size_t)D.na_max) return cudaErrorNotSupported;

    DecodeParams P{};
    P.n_groups = n_groups;
    P.m = m;
    P.has_shared = n_groups > 1 ? 1 : 0;
    const int lg_a = lg_split_for(hidden), lg_b = lg_split_for(inter);
    for (int g = 0; g < n_groups; ++g) {
        P.a[g] = group_dev(gu[g], lg_a, kFused);
        P.b[g] = group_dev(dn[g], lg_b, kOne);  // the shared expert's down rows with the routed split
        const int rows = g == 0 ? m * top_k : m;
        const int kb = dn[g].k;
        P.stg_planes[g] = stage[g];
        P.stg_meta[g] = reinterpret_cast<float2*>(stage[g] + (int64_t)rows * (kb / 64) * kPairBytes);
    }
    P.off_x = D.off_x; P.off_xmeta = D.off_xmeta; P.off_gu = D.off_gu; P.gu_pairs = D.gu_pairs;
    P.off_eout = D.off_eout; P.off_hmid = D.off_hmid; P.off_a = D.off_a; P.item_bytes = D.item_bytes;
    for (int g = 0; g < 2; ++g) { P.off_act[g] = D.off_act[g]; P.off_actmeta[g] = D.off_actmeta[g]; }
    P.off_b = D.off_b;
    P.rows_max = D.rows_max;
    P.n_row_tiles = D.n_row_tiles;
    P.cb = cb;
    P.gen = sync;
    P.cta_tag = sync + head;
    P.flags = P.cta_tag + kDecMaxCtas;
    P.cap_flags = (int)std::min<size_t>(sync_words - head - kDecMaxCtas, 1u << 30);
    if (P.has_shared) {
        P.pf[0] = gu[1].w;  P.pf_bytes[0] = (uint64_t)gu[1].n * (gu[1].k / kQK) * kBlockBytes;
        P.pf[1] = gu[1].w2; P.pf_bytes[1] = P.pf_bytes[0];
        P.pf[2] = dn[1].w;  P.pf_bytes[2] = (uint64_t)dn[1].n * (dn[1].k / kQK) * kBlockBytes;
    }
    P.err_flag = err_flag;
    P.wait_ns = wait_limit_ns();

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = D.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_layer_kernel, P);
}

}  // namespace q4k

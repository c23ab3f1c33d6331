// q4k_stream.cu -- the id-GEMV for small batches (every group holds at most 32 pairs), with
// the weight rows moved by the TMA engine.
//
// Same result as the bucketed kernel of q4k_gemv.cu (ferrum-kernels
// q4_k_moe_id_gemv_batched.rs: out[p, r] = W_{ids[p]}[r, :] . a[t*outer + s*inner, :];
// with a second slab, silu(gate) * up as in moeflux expert_forward.rs), organised for decode:
//  * Work item = (pair, tile of R rows of the pair's expert). The R rows of one expert are
//    contiguous in the slab, so one bulk copy (cp.async.bulk, completing on an mbarrier)
//    per slab moves the item's weights into a shared-memory stage: no per-thread load
//    slots, no partially used cache lines, and the copies of the next stages run while the
//    current one is computed.
//  * A thread owns a fixed set of 64-weight groups of a row (group g = block g/4, weights
//    64*(g%4) .. +63) and holds the staged activation planes of those groups in registers;
//    it walks the item's rows, reading each row's block header and its 32 code bytes from
//    shared memory (conflict-free 16-byte reads), and keeps one partial sum per row.
//    tpr threads (a power of two >= k/64, at most 128) share a row; 128/tpr rows are
//    walked side by side. Partial sums are reduced with shuffles (and across warps through
//    shared memory when tpr > 32).
//  * Items of one expert's tile run back to back for its pairs (the repeated copy then
//    comes from L2); each CTA takes a balanced contiguous range of items.
//  * A launch that may overlap the previous kernel (programmatic dependent launch) issues its
//    weight copies before waiting for that kernel; activations are read after the wait.
//  * With the combine fused (the down launch of a layer), the last CTA to finish a row tile
//    forms y for those rows.
#include <algorithm>

#include "q4k_gemv_common.cuh"
#include "q4k_sm100.cuh"

namespace q4k {

namespace {
using namespace sm100;

constexpr int kSThreads = 128;
constexpr int kSWarps = kSThreads / 32;
constexpr int kSStages = 2;
constexpr int kSRpt = 4;     // rows per thread per item (R = kSRpt * 128 / tpr) ...
constexpr int kSMaxRpt = 8;  // ... or twice that for the second group of a fused combine
constexpr int kSMaxGpt = 2;  // 64-weight groups per thread (k <= 128 * 64 * 2)
constexpr size_t kSSmemMax = 200 * 1024;

struct SGroup {
    const uint8_t* w;
    const uint8_t* w2;
    const int32_t* ids;
    const float* a;
    float* out;
    int64_t outer, inner;
    int64_t nb01, nb02;
    int num_experts, n_pairs, top_k, n, k;
    int R, tiles;      // rows per item, ceil(n / R)
    int tpr, gpt;      // threads per row (power of two), 64-weight groups per thread
    int64_t a_bytes;   // span of the activation rows the group reads (L2 prefetch; 0: none)
};

struct SParams {
    SGroup g[kMaxGroups];
    int n_groups;
    int tc_min;
    int pdl;
    int* err_flag;
    int has_combine;
    CombineSpec cb;
    unsigned* zero;
    int n_zero;
    int stage_bytes;        // bytes per stage (both slabs)
    int xs_off, meta_off;   // staged activation planes and (delta, sumX) pairs
    int wait_first;         // wait for the previous kernel before reading anything (first launch of a layer)
};

struct SItem {
    int gi, e, tile, p;
};

// Item -> (group, expert, tile, pair); warp-collective. Items of expert e: its pairs times
// its tiles, pairs fastest.
__device__ __forceinline__ SItem s_locate(const FastGroup* s_fast, const int* s_items, int n_groups, int item) {
    const int lane = threadIdx.x & 31;
    SItem it;
    it.gi = (n_groups > 1 && item >= s_items[1]) ? 1 : 0;
    const FastGroup& F = s_fast[it.gi];
    const int local = item - s_items[it.gi];
    const bool mine = lane < F.U && F.start[lane] <= local && local < F.start[lane + 1];
    const int r = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
    const unsigned mask = F.mask[r];
    const int cnt = __popc(mask);
    const int in_e = local - F.start[r];
    const int q = in_e % cnt;  // the q-th member of the bucket, members in pair order
    it.e = F.e[r];
    it.tile = in_e / cnt;
    const bool member = (mask >> lane) & 1u;
    const unsigned b = __ballot_sync(0xffffffffu, member && __popc(mask & ((1u << lane) - 1u)) == q);
    it.p = __ffs(b) - 1;
    return it;
}

// Stage one activation row (all threads): planes of group g at xs + g*144, meta[j] per
// 32-element sub-block j. pre (when given) holds this thread's loads of the first pass.
__device__ __forceinline__ void load_pass(const float* row, int nf, int f0, float4 (&v)[kStageUnroll]) {
#pragma unroll
    for (int u = 0; u < kStageUnroll; ++u) {
        const int f = f0 + u * kSThreads + (int)threadIdx.x;
        v[u] = f < nf ? __ldg(reinterpret_cast<const float4*>(row) + f) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

__device__ __forceinline__ void stage_row(const float* row, int k, uint8_t* xs, float2* meta,
                                          const float4 (*pre)[kStageUnroll]) {
    const int nf = k / 4;
    for (int f0 = 0; f0 < nf; f0 += kSThreads * kStageUnroll) {
        float4 v[kStageUnroll];
        if (pre && f0 == 0) {
#pragma unroll
            for (int u = 0; u < kStageUnroll; ++u) v[u] = (*pre)[u];
        } else {
            load_pass(row, nf, f0, v);
        }
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            if (f0 + u * kSThreads >= nf) break;  // uniform over the block
            const int f = f0 + u * kSThreads + (int)threadIdx.x;
            stage_quad(v[u], f, f < nf, xs, meta);
        }
    }
}

__device__ __forceinline__ uint4 lds16(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

template <bool FUSED>
__global__ void __launch_bounds__(kSThreads, 2)
idgemv_stream_kernel(const __grid_constant__ SParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bar_full[kSStages];
    __shared__ FastGroup s_fast[kMaxGroups];
    __shared__ int s_bad[kMaxGroups];
    __shared__ int s_items[kMaxGroups + 1];
    __shared__ float s_red[2][kSWarps][kSMaxRpt];
    __shared__ volatile int s_abort;
    __shared__ int s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the ids and activations may come from the previous kernel: with wait_first, wait, then
    // let the next launch (which reads the ids before its own wait) start
    if (P.wait_first) pdl_wait();
    pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < kSStages; ++s) mbar_init(&bar_full[s], 1);
        fence_mbar_init();
        s_abort = 0;
    }
    if (P.zero && blockIdx.x == 0)
        for (int i = tid; i < P.n_zero; i += kSThreads) P.zero[i] = 0u;
    // the activation rows go towards L2 now, ahead of the weight copies in the memory queues
    // (only without a previous kernel still writing them)
    const bool acts_ready = !P.pdl || P.wait_first;
    if (acts_ready && blockIdx.x < 4 && tid < P.n_groups && P.g[tid].a_bytes > 0) {
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(P.g[tid].a) & ~uintptr_t(15);
        const uintptr_t a1 = (reinterpret_cast<uintptr_t>(P.g[tid].a) + (uintptr_t)P.g[tid].a_bytes + 15) & ~uintptr_t(15);
        bulk_prefetch_l2(reinterpret_cast<const void*>(a0), (uint32_t)(a1 - a0));
    }
    // ---- bucketing: one warp per group (ids are inputs of the layer)
    if (warp < P.n_groups) {
        const SGroup& G = P.g[warp];
        fast_bucket(G.ids, G.n_pairs, G.num_experts, G.tiles, 1, P.tc_min, s_fast[warp], &s_bad[warp]);
    }
    __syncthreads();
    if (tid == 0) {
        s_items[0] = 0;
        for (int gi = 0; gi < P.n_groups; ++gi) s_items[gi + 1] = s_items[gi] + s_fast[gi].start[s_fast[gi].U];
    }
    __syncthreads();
    const int total = s_items[P.n_groups];
    const int ib = (int)(((int64_t)blockIdx.x * total) / gridDim.x);
    const int ie = (int)(((int64_t)(blockIdx.x + 1) * total) / gridDim.x);

    // ---- weight copies of the first stages (the slabs are not written by any kernel)
    auto issue = [&](int item, int s) {  // all lanes of warp 0
        const SItem it = s_locate(s_fast, s_items, P.n_groups, item);
        if (lane == 0) {
            const SGroup& G = P.g[it.gi];
            const int r0 = it.tile * G.R;
            const uint32_t bytes = (uint32_t)(min(G.R, G.n - r0) * G.nb01);
            uint8_t* dst = smem + s * P.stage_bytes;
            const int64_t off = (int64_t)it.e * G.nb02 + (int64_t)r0 * G.nb01;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bar_full[s], FUSED ? 2 * bytes : bytes);
            bulk_g2s(dst, G.w + off, bytes, &bar_full[s]);
            if (FUSED) bulk_g2s(dst + (int64_t)G.R * G.nb01, G.w2 + off, bytes, &bar_full[s]);
        }
    };
    // The first item's activation loads leave before the weight copies (responses come back
    // in about the order of the requests), unless the previous kernel may still write them.
    float4 xpre[kStageUnroll];
    const bool have_pre = acts_ready && ib < ie;
    if (have_pre) {
        const SItem it0 = s_locate(s_fast, s_items, P.n_groups, ib);
        const SGroup& G0 = P.g[it0.gi];
        load_pass(G0.a + (int64_t)(it0.p / G0.top_k) * G0.outer + (int64_t)(it0.p % G0.top_k) * G0.inner, G0.k / 4, 0,
                  xpre);
    }
    if (warp == 0)
        for (int j = 0; j < kSStages && ib + j < ie; ++j) issue(ib + j, j);

    uint8_t* xs = smem + P.xs_off;
    float2* meta = reinterpret_cast<float2*>(smem + P.meta_off);
    uint32_t xr[kSMaxGpt][32];
    float4 xm[kSMaxGpt];
    int x_gi = -1;
    int64_t x_row = -1;
    bool waited = !P.pdl;
    const unsigned expected = P.has_combine && P.g[0].tiles > 0 ? (unsigned)(total / P.g[0].tiles) : 0u;

    for (int item = ib; item < ie; ++item) {
        const int j = item - ib, s = j % kSStages;
        const uint32_t ph = (uint32_t)(j / kSStages) & 1u;
        const SItem it = s_locate(s_fast, s_items, P.n_groups, item);
        const SGroup& G = P.g[it.gi];
        const int tpr = G.tpr, RP = kSThreads / tpr;
        const int tir = tid & (tpr - 1), rpi = tid / tpr;
        const int ngr = G.k / 64;

        // ---- the pair's activation row, staged and moved to registers when it changes
        const int64_t arow = (int64_t)(it.p / G.top_k) * G.outer + (int64_t)(it.p % G.top_k) * G.inner;
        if (it.gi != x_gi || arow != x_row) {  // uniform over the block
            if (!waited) {
                pdl_wait();  // the activations may come from the previous kernel
                waited = true;
            }
            stage_row(G.a + arow, G.k, xs, meta, (have_pre && item == ib) ? &xpre : nullptr);
            __syncthreads();
#pragma unroll
            for (int q = 0; q < kSMaxGpt; ++q) {
                const int g = tir + q * tpr;
                if (q < G.gpt && g < ngr) {
                    const uint4* xp = reinterpret_cast<const uint4*>(xs + g * kPairBytes);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint4 v = xp[i];
                        xr[q][4 * i] = v.x; xr[q][4 * i + 1] = v.y; xr[q][4 * i + 2] = v.z; xr[q][4 * i + 3] = v.w;
                    }
                    xm[q] = *reinterpret_cast<const float4*>(meta + 2 * g);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) xr[q][i] = 0u;
                    xm[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            x_gi = it.gi;
            x_row = arow;
        }

        // ---- the item's rows
        if (!mbar_wait(&bar_full[s], ph, &s_abort)) {
            s_abort = 1;
            raise_flag(P.err_flag, Q4K_ERR_TIMEOUT);
        }
        const int r0 = it.tile * G.R;
        const int rows_valid = min(G.R, G.n - r0);
        const int rpt = G.R / RP;  // kSRpt or 2 * kSRpt (uniform)
        const uint8_t* st = smem + s * P.stage_bytes;
        const uint8_t* st2 = st + (int64_t)G.R * G.nb01;
        // Rows past the tile's end and groups past the row's end are clamped to valid ones
        // (their results are not used; a clamped group meets zero activations), so the row
        // bodies have no branches and the loads and dot products of all rows interleave.
        float acc[kSMaxRpt], acc2[kSMaxRpt];
        auto row_dot = [&](int i) {
            acc[i] = 0.f;
            acc2[i] = 0.f;
            const int r = min(rpi + i * RP, rows_valid - 1);
#pragma unroll
            for (int q = 0; q < kSMaxGpt; ++q) {
                if (q < G.gpt) {  // uniform
                    const int g = min(tir + q * tpr, ngr - 1);
                    const int b = g >> 2, c = g & 3;
                    const uint8_t* pb = st + (int64_t)r * G.nb01 + b * kBlockBytes;
                    float sa, ma, sb, mb;
                    int Sa, Sb;
                    block_scales(lds16(pb), c, sa, ma, sb, mb);
                    dot64_regs(lds16(pb + 16 + 32 * c), lds16(pb + 32 + 32 * c), xr[q], Sa, Sb);
                    acc[i] += xm[q].x * (sa * (float)Sa - ma * xm[q].y) + xm[q].z * (sb * (float)Sb - mb * xm[q].w);
                    if (FUSED) {
                        const uint8_t* pb2 = st2 + (int64_t)r * G.nb01 + b * kBlockBytes;
                        block_scales(lds16(pb2), c, sa, ma, sb, mb);
                        dot64_regs(lds16(pb2 + 16 + 32 * c), lds16(pb2 + 32 + 32 * c), xr[q], Sa, Sb);
                        acc2[i] += xm[q].x * (sa * (float)Sa - ma * xm[q].y) + xm[q].z * (sb * (float)Sb - mb * xm[q].w);
                    }
                }
            }
        };
#pragma unroll
        for (int i = 0; i < kSRpt; ++i) row_dot(i);
        if (rpt > kSRpt) {
#pragma unroll
            for (int i = kSRpt; i < kSMaxRpt; ++i) row_dot(i);
        } else {
#pragma unroll
            for (int i = kSRpt; i < kSMaxRpt; ++i) { acc[i] = 0.f; acc2[i] = 0.f; }
        }
        // ---- reduce over the tpr threads of a row and write
        const int wl = tpr < 32 ? tpr : 32;
#pragma unroll
        for (int i = 0; i < kSMaxRpt; ++i) {
            if (i < rpt) {
                for (int off = 1; off < wl; off <<= 1) {
                    acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], off);
                    if (FUSED) acc2[i] += __shfl_xor_sync(0xffffffffu, acc2[i], off);
                }
            }
        }
        float* out = G.out + (int64_t)it.p * G.n + r0;
        if (tpr <= 32) {
            if (tir == 0) {
#pragma unroll
                for (int i = 0; i < kSMaxRpt; ++i) {
                    const int r = rpi + i * RP;
                    if (i < rpt && r < rows_valid) out[r] = FUSED ? silu(acc[i]) * acc2[i] : acc[i];
                }
            }
            __syncthreads();  // stage s is read by everyone
        } else {
            if (lane == 0) {
#pragma unroll
                for (int i = 0; i < kSMaxRpt; ++i) {
                    s_red[0][warp][i] = acc[i];
                    s_red[1][warp][i] = acc2[i];
                }
            }
            __syncthreads();  // stage s is read by everyone; partials are in s_red
            if (tid < rows_valid) {
                const int r = tid, rp_r = r % RP, i_r = r / RP, wpr = tpr / 32;
                float g = 0.f, u = 0.f;
                for (int w = rp_r * wpr; w < (rp_r + 1) * wpr; ++w) {
                    g += s_red[0][w][i_r];
                    u += s_red[1][w][i_r];
                }
                out[r] = FUSED ? silu(g) * u : g;
            }
            __syncthreads();  // s_red is rewritten by the next item
        }
        // ---- refill stage s
        if (warp == 0 && item + kSStages < ie) issue(item + kSStages, s);
        if (P.has_combine) {
            // every item of this row tile, from either group, counts once; the last one combines
            if (tid == 0) {
                __threadfence();
                s_last = atomicAdd(&P.cb.counters[it.tile], 1u) + 1u == expected;
            }
            __syncthreads();
            if (s_last) {
                __threadfence();
                const SGroup& R = P.g[0];
                const bool shared = P.cb.shared_mode != Q4K_SHARED_NONE && P.n_groups > 1;
                combine_span(P.cb, R.out, R.ids, R.num_experts, R.n_pairs, R.top_k, R.n, shared ? P.g[1].out : nullptr,
                             it.tile * R.R, min(R.n, (it.tile + 1) * R.R), tid, kSThreads);
                if (tid == 0) P.cb.counters[it.tile] = 0u;
            }
            __syncthreads();
        }
    }
    // every expert went to the tensor-core path: no item counts, so combine every tile
    if (P.has_combine && total == 0) {
        pdl_wait();
        const SGroup& R = P.g[0];
        const bool shared = P.cb.shared_mode != Q4K_SHARED_NONE && P.n_groups > 1;
        for (int tile = blockIdx.x; tile < R.tiles; tile += gridDim.x)
            combine_span(P.cb, R.out, R.ids, R.num_experts, R.n_pairs, R.top_k, R.n, shared ? P.g[1].out : nullptr,
                         tile * R.R, min(R.n, (tile + 1) * R.R), tid, kSThreads);
    }
    // out-of-range ids: flag and zero their rows (CTA 0, after the previous kernel is done)
    if (blockIdx.x == 0) {
        pdl_wait();
        for (int gi = 0; gi < P.n_groups; ++gi) {
            const SGroup& G = P.g[gi];
            if (!G.ids || s_bad[gi] == 0) continue;
            if (tid == 0) raise_flag(P.err_flag, Q4K_ERR_EXPERT_ID);
            for (int p = 0; p < G.n_pairs; ++p) {
                if (id_valid(G.ids[p], G.num_experts)) continue;
                for (int r = tid; r < G.n; r += kSThreads) G.out[(int64_t)p * G.n + r] = 0.0f;
            }
        }
    }
    // after a timeout, let the copies still in flight land before the CTA leaves (bounded)
    if (s_abort && tid == 0) {
        volatile int never = 0;
        for (int item = max(ib, ie - kSStages); item < ie; ++item) {
            const int j = item - ib;
            mbar_wait(&bar_full[j % kSStages], (uint32_t)(j / kSStages) & 1u, &never);
        }
    }
}

constexpr int kMaxDevicesS = 64;
bool g_s_attr_set[2][kMaxDevicesS] = {};

int pow2_at_least(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

}  // namespace

cudaError_t launch_idgemv_stream(const GemvGroup* groups, int n_groups, bool fused_swiglu, bool pdl, int* err_flag,
                                 cudaStream_t stream, int tc_min, const CombineSpec* combine, unsigned* zero,
                                 int n_zero, bool pdl_wait_first) {
    if (n_groups < 1 || n_groups > kMaxGroups) return cudaErrorNotSupported;
    SParams P{};
    P.n_groups = n_groups;
    P.err_flag = err_flag;
    P.tc_min = tc_min;
    P.pdl = pdl ? 1 : 0;
    P.wait_first = (pdl && pdl_wait_first) ? 1 : 0;
    P.zero = zero;
    P.n_zero = zero ? n_zero : 0;
    if (combine) {
        P.has_combine = 1;
        P.cb = *combine;
    }
    const int slabs = fused_swiglu ? 2 : 1;
    int rp[kMaxGroups] = {};
    int64_t max_items = 0;
    int kmax = 0;
    for (int gi = 0; gi < n_groups; ++gi) {
        const GemvGroup& S = groups[gi];
        if ((int64_t)S.m * S.top_k > 32) return cudaErrorNotSupported;
        SGroup& G = P.g[gi];
        G.w = S.w; G.w2 = S.w2; G.ids = S.ids; G.a = S.a; G.out = S.out;
        G.outer = S.outer; G.inner = S.inner;
        G.nb01 = (int64_t)(S.k / kQK) * kBlockBytes;
        G.nb02 = (int64_t)S.n * G.nb01;
        G.num_experts = S.num_experts; G.n_pairs = S.m * S.top_k; G.top_k = S.top_k;
        G.n = S.n; G.k = S.k;
        const int ngr = S.k / 64;
        G.tpr = std::min(kSThreads, pow2_at_least(ngr));
        G.gpt = (ngr + G.tpr - 1) / G.tpr;
        if (G.gpt > kSMaxGpt) return cudaErrorNotSupported;
        rp[gi] = kSThreads / G.tpr;
        G.R = kSRpt * rp[gi];
        const int64_t span = S.m > 0 ? ((int64_t)(S.m - 1) * S.outer + (int64_t)(S.top_k - 1) * S.inner + S.k) * 4 : 0;
        G.a_bytes = span <= (1 << 20) ? span : 0;
        kmax = std::max(kmax, S.k);
    }
    // with the combine fused, every group uses group 0's row tiles (one counter per tile)
    if (combine && n_groups > 1) {
        const int rmax = std::max(rp[0], rp[1]), rmin = std::min(rp[0], rp[1]);
        if (kSRpt * rmax > kSMaxRpt * rmin) return cudaErrorNotSupported;
        P.g[0].R = P.g[1].R = kSRpt * rmax;
    }
    int64_t stage = 0;
    for (int gi = 0; gi < n_groups; ++gi) {
        SGroup& G = P.g[gi];
        G.tiles = (G.n + G.R - 1) / G.R;
        stage = std::max<int64_t>(stage, (int64_t)slabs * G.R * G.nb01);
        max_items += (int64_t)G.n_pairs * G.tiles;
    }
    if (combine && P.g[0].tiles > combine->n_counters) return cudaErrorInvalidValue;
    if (max_items == 0 && !combine) return cudaSuccess;
    if (max_items == 0) max_items = 1;
    stage = (stage + 127) & ~int64_t(127);
    P.stage_bytes = (int)stage;
    P.xs_off = (int)(kSStages * stage);
    P.meta_off = P.xs_off + ((kmax / 64) * kPairBytes + 15) / 16 * 16;
    const size_t smem = (size_t)P.meta_off + (size_t)(kmax / 32) * 8;
    if (smem > kSSmemMax) return cudaErrorNotSupported;
    void (*kern)(SParams) = fused_swiglu ? idgemv_stream_kernel<true> : idgemv_stream_kernel<false>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevicesS) return cudaErrorInvalidDevice;
    const int kind = fused_swiglu ? 1 : 0;
    if (!g_s_attr_set[kind][dev]) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSSmemMax);
        if (err != cudaSuccess) return err;
        g_s_attr_set[kind][dev] = true;
    }
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSThreads, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)num_sms() * per_sm;
    if (grid > max_items) grid = max_items;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

}  // namespace q4k

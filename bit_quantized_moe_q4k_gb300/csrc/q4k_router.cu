// q4k_router.cu -- the router of a MoE layer: gate logits, top-k choice and routing weights,
// producing the ids and weights the layer's bucketing and combine read.
//
// moeflux expert_forward.rs (MoeBuffers::gate_logits): the router's gate logits are one fp32
// per expert from a bf16 matvec of the layer input; its `noaux_tc` routing and the
// softmax + top-K + normalise routing (synth::expert_weights_seeded) turn them into the
// chosen experts and their weights.
//
// One launch. A token tile's logits are computed by one thread-block cluster: the experts'
// rows are dealt round robin to the cluster's CTAs, each CTA spreads every row over all its
// threads (a thread holds 8-column chunks of the tile's activations in registers, reused for
// every row), and the CTAs store the logits into the shared memory of the cluster's first
// CTA through distributed shared memory. After the cluster barrier that CTA chooses, one warp
// per token. No global scratch, no flags, no second launch.
//
// Arithmetic (fixed order, so every launch gives the same bits): a logit is the fp32 sum of
// bf16(w) * x with each thread folding its chunks left to right (fma), the 32 lanes of a warp
// added by xor shuffles (1, 2, 4, 8, 16) and the 8 warps added in warp order. Choice: the
// larger score first, equal scores by the lower expert id; NaN ranks below every number.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "q4k_internal.cuh"

namespace q4k {
namespace {

constexpr int kRThreads = 256;
constexpr int kRWarps = kRThreads / 32;
// rows in flight per CTA: as many as keep a thread's weight registers at 32
__host__ __device__ constexpr int rows_in_flight(int nch) { return nch <= 2 ? 4 : (nch <= 4 ? 2 : 1); }
// the first CTA's tables (logits, corrected scores, taken flags: 9 bytes per expert and token)
constexpr size_t kRouterSmemBudget = 160 * 1024;
constexpr size_t kRouterSmemMax = kRouterSmemBudget + 16;

struct RouterParams {
    const float* x;         // [m, hidden]
    const uint16_t* w;      // [num_experts, hidden] bf16
    const float* bias;      // [num_experts] or null
    const uint16_t* w_sg;   // [hidden] bf16 shared-expert gate row, or null
    int32_t* ids;           // [m, top_k]
    float* weights;         // [m, top_k]
    float* logits;          // [m, num_experts] or null
    float* shared_gate;     // [m] (with w_sg)
    int m, E, H, top_k;
    int scoring, normalize;
    float scale;
    int n_group, topk_group, per;
    int tile;               // tokens per cluster (<= the kernel's TT)
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nrank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_arrive_release() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Store v at the same shared-memory offset as `local` in CTA `rank` of the cluster.
__device__ __forceinline__ void st_cluster_f32(const float* local, uint32_t rank, float v) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(r), "f"(v) : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Ranking key: NaN below every number.
__device__ __forceinline__ float rank_key(float v) { return v != v ? -INFINITY : v; }

// (v, i) beats (u, j): a candidate (i >= 0) beats none; a larger key wins; equal keys go to
// the lower index.
__device__ __forceinline__ bool beats(float v, int i, float u, int j) {
    if (i < 0) return false;
    if (j < 0) return true;
    return v > u || (v == u && i < j);
}

// Warp-wide best of the lanes' (v, i); every lane gets the winner.
__device__ __forceinline__ void warp_best(float& v, int& i) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float u = __shfl_xor_sync(0xffffffffu, v, off);
        const int j = __shfl_xor_sync(0xffffffffu, i, off);
        if (beats(u, j, v, i)) { v = u; i = j; }
    }
}

// The lane's best untaken, allowed entry among e = lane, lane + 32, ... (key[e]).
__device__ __forceinline__ void lane_best(const float* key, const uint8_t* taken, const uint32_t* allowed_groups,
                                          int gsize, int E, int lane, float& v, int& i) {
    v = -INFINITY;
    i = -1;
    for (int e = lane; e < E; e += 32) {
        if (taken[e]) continue;
        if (allowed_groups && !((allowed_groups[0] >> (e / gsize)) & 1u)) continue;
        const float k = rank_key(key[e]);
        if (beats(k, e, v, i)) { v = k; i = e; }
    }
}

// Choose top_k of key[0..E) (warp-wide). Lane j < top_k gets the j-th choice in (my_i).
__device__ __forceinline__ void choose(const float* key, uint8_t* taken, const uint32_t* allowed_groups, int gsize,
                                       int E, int top_k, int lane, int& my_i) {
    float v;
    int i;
    lane_best(key, taken, allowed_groups, gsize, E, lane, v, i);
    my_i = -1;
    for (int j = 0; j < top_k; ++j) {
        float bv = v;
        int bi = i;
        warp_best(bv, bi);
        if (lane == j) my_i = bi;
        if (bi >= 0 && (bi & 31) == lane) {  // the owner marks it and looks again
            taken[bi] = 1;
            lane_best(key, taken, allowed_groups, gsize, E, lane, v, i);
        }
        __syncwarp();
    }
}

template <int NCH, int TT>
__global__ void __launch_bounds__(kRThreads, 1) router_kernel(const RouterParams P) {
    constexpr int kRB = rows_in_flight(NCH);
    extern __shared__ __align__(16) unsigned char smem[];
    // leader's arrays: logits [tile][E], corrected scores [tile][E], taken flags [tile][E]
    float* s_logit = reinterpret_cast<float*>(smem);
    float* s_c = s_logit + (size_t)P.tile * P.E;
    uint8_t* s_taken = reinterpret_cast<uint8_t*>(s_c + (size_t)P.tile * P.E);
    __shared__ float s_red[2][kRWarps][kRB * TT];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cluster_rank(), CS = cluster_nrank();
    const int t0 = blockIdx.y * P.tile;
    const int nt = min(P.tile, P.m - t0);
    cluster_arrive_relaxed();  // every CTA of the cluster has started before any remote store
    // programmatic dependent launch: the layer launched next may start its prologue now (it
    // waits for this grid before reading ids or weights); this grid waits for the previous
    // kernel (which may have written x) before reading
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // this thread's activation chunks (8 columns each) of the tile's tokens
    float xr[TT][NCH][8];
    const int nchunk = P.H / 8;
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int q = tid + c * kRThreads;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (t < nt && q < nchunk) {
                const float4* src = reinterpret_cast<const float4*>(P.x + (int64_t)(t0 + t) * P.H) + 2 * q;
                a = __ldg(src);
                b = __ldg(src + 1);
            }
            xr[t][c][0] = a.x; xr[t][c][1] = a.y; xr[t][c][2] = a.z; xr[t][c][3] = a.w;
            xr[t][c][4] = b.x; xr[t][c][5] = b.y; xr[t][c][6] = b.z; xr[t][c][7] = b.w;
        }

    const int rows = P.E + (P.w_sg ? 1 : 0);
    bool waited = false;
    int batch = 0;
    for (int r0 = (int)rank; r0 < rows; r0 += kRB * (int)CS, ++batch) {
        // issue every load of the batch's rows first
        uint4 wv[kRB][NCH];
#pragma unroll
        for (int b = 0; b < kRB; ++b) {
            const int row = r0 + b * (int)CS;
            const uint16_t* wr = row < P.E ? P.w + (int64_t)row * P.H : P.w_sg;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                const int q = tid + c * kRThreads;
                wv[b][c] = (row < rows && q < nchunk) ? __ldg(reinterpret_cast<const uint4*>(wr) + q) : make_uint4(0, 0, 0, 0);
            }
        }
        float acc[kRB][TT];
#pragma unroll
        for (int b = 0; b < kRB; ++b)
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                float s = 0.0f;
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    const uint32_t u[4] = {wv[b][c].x, wv[b][c].y, wv[b][c].z, wv[b][c].w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        s = __fmaf_rn(bf16_lo(u[h]), xr[t][c][2 * h], s);
                        s = __fmaf_rn(bf16_hi(u[h]), xr[t][c][2 * h + 1], s);
                    }
                }
                acc[b][t] = s;
            }
        float* red = &s_red[batch & 1][0][0];
#pragma unroll
        for (int b = 0; b < kRB; ++b)
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                float s = acc[b][t];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
                if (lane == 0) red[warp * (kRB * TT) + b * TT + t] = s;
            }
        __syncthreads();
        if (!waited) { cluster_wait(); waited = true; }
        if (tid < kRB * TT) {
            const int b = tid / TT, t = tid % TT;
            const int row = r0 + b * (int)CS;
            if (row < rows && t < nt) {
                float s = red[b * TT + t];
#pragma unroll
                for (int w = 1; w < kRWarps; ++w) s = __fadd_rn(s, red[w * (kRB * TT) + b * TT + t]);
                if (row < P.E) {
                    st_cluster_f32(s_logit + (size_t)t * P.E + row, 0, s);
                    if (P.logits) P.logits[(int64_t)(t0 + t) * P.E + row] = s;
                } else {
                    P.shared_gate[t0 + t] = s;
                }
            }
        }
    }
    if (!waited) cluster_wait();
    cluster_arrive_release();
    cluster_wait();
    if (rank != 0 || warp >= nt) return;

    // ---- choice, one warp per token ----
    const int t = warp;
    const int E = P.E, K = P.top_k;
    float* lg = s_logit + (size_t)t * E;
    float* cs = s_c + (size_t)t * E;
    uint8_t* tk = s_taken + (size_t)t * E;
    for (int e = lane; e < E; e += 32) tk[e] = 0;
    int my_i = -1;
    float my_w = 0.0f;
    if (P.scoring == Q4K_ROUTE_SOFTMAX) {
        __syncwarp();
        choose(lg, tk, nullptr, E, E, K, lane, my_i);
        const float lmax = __shfl_sync(0xffffffffu, my_i >= 0 ? lg[my_i] : 0.0f, 0);
        const float p = (lane < K && my_i >= 0) ? expf(lg[my_i] - lmax) : 0.0f;
        float z = 0.0f;
        if (P.normalize) {  // over the chosen, in choice order
            for (int j = 0; j < K; ++j) z = __fadd_rn(z, __shfl_sync(0xffffffffu, p, j));
        } else {  // over all experts: each lane's in index order, then xor shuffles
            for (int e = lane; e < E; e += 32) z = __fadd_rn(z, expf(lg[e] - lmax));
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) z = __fadd_rn(z, __shfl_xor_sync(0xffffffffu, z, off));
        }
        my_w = p / z;
    } else {
        const int gsize = E / P.n_group;
        for (int e = lane; e < E; e += 32) {
            const float s = 1.0f / (1.0f + expf(-lg[e]));
            cs[e] = __fadd_rn(s, P.bias ? P.bias[e] : 0.0f);
        }
        __syncwarp();
        uint32_t allowed = 0xffffffffu;
        if (P.n_group > 1) {
            // lane g scores group g: the sum, largest first, of its `per` largest corrected scores
            float gs = -INFINITY;
            int gi = -1;
            if (lane < P.n_group) {
                float top[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) top[j] = -INFINITY;
                for (int e = lane * gsize; e < (lane + 1) * gsize; ++e) {
                    float v = rank_key(cs[e]);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {  // insertion into a descending list
                        if (j < P.per && v > top[j]) { const float o = top[j]; top[j] = v; v = o; }
                    }
                }
                gs = top[0];
#pragma unroll
                for (int j = 1; j < 16; ++j)
                    if (j < P.per) gs = __fadd_rn(gs, top[j]);
                gs = rank_key(gs);
                gi = lane;
            }
            allowed = 0u;
            for (int j = 0; j < P.topk_group; ++j) {
                float bv = gs;
                int bi = gi;
                warp_best(bv, bi);
                if (bi >= 0) allowed |= 1u << bi;
                if (lane == bi) gi = -1;
            }
        }
        __shared__ uint32_t s_allowed[kRWarps];
        if (lane == 0) s_allowed[warp] = allowed;
        __syncwarp();
        choose(cs, tk, P.n_group > 1 ? &s_allowed[warp] : nullptr, gsize, E, K, lane, my_i);
        const float s = (lane < K && my_i >= 0) ? 1.0f / (1.0f + expf(-lg[my_i])) : 0.0f;
        if (P.normalize) {
            float z = 0.0f;
            for (int j = 0; j < K; ++j) z = __fadd_rn(z, __shfl_sync(0xffffffffu, s, j));
            my_w = __fmul_rn(s / z, P.scale);
        } else {
            my_w = __fmul_rn(s, P.scale);
        }
    }
    if (lane < K) {
        P.ids[(int64_t)(t0 + t) * K + lane] = my_i;
        P.weights[(int64_t)(t0 + t) * K + lane] = my_w;
    }
}

template <int NCH, int TT>
cudaError_t launch_router_t(const RouterParams& P, int cs, size_t smem, cudaStream_t stream) {
    auto kern = router_kernel<NCH, TT>;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)cs, (unsigned)((P.m + P.tile - 1) / P.tile), 1);
    cfg.blockDim = dim3(kRThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

// Largest cluster (16, else 8) the device can schedule with the kernel's shared memory set to
// its largest plan; 0 if the attributes cannot be set. Worked out once per kernel.
template <int NCH, int TT>
int cluster_size_for() {
    static const int cs = [] {
        auto kern = router_kernel<NCH, TT>;
        const size_t smem = kRouterSmemMax;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) return 8;
        for (int c : {16, 8}) {
            cudaLaunchConfig_t cfg{};
            cfg.gridDim = dim3((unsigned)c, 1, 1);
            cfg.blockDim = dim3(kRThreads, 1, 1);
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = (unsigned)c;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) return c;
        }
        (void)cudaGetLastError();
        return 8;
    }();
    return cs;
}

template <int NCH, int TT>
cudaError_t dispatch_tt(RouterParams P, cudaStream_t stream) {
    const size_t per_token = (size_t)P.E * (2 * sizeof(float) + 1);
    P.tile = (int)std::min<size_t>((size_t)TT, std::max<size_t>(1, kRouterSmemBudget / per_token));
    P.tile = std::min(P.tile, std::max(P.m, 1));
    const size_t smem = (per_token * P.tile + 15) & ~(size_t)15;
    const int cs = cluster_size_for<NCH, TT>();
    if (cs == 0) return cudaErrorInvalidConfiguration;
    // at most 32768 token tiles per launch (the grid's y extent)
    const int per_launch = 32768 * P.tile;
    const int m = P.m;
    for (int t0 = 0; t0 < m; t0 += per_launch) {
        RouterParams Q = P;
        Q.m = std::min(per_launch, m - t0);
        Q.x = P.x + (int64_t)t0 * P.H;
        Q.ids = P.ids + (int64_t)t0 * P.top_k;
        Q.weights = P.weights + (int64_t)t0 * P.top_k;
        Q.logits = P.logits ? P.logits + (int64_t)t0 * P.E : nullptr;
        Q.shared_gate = P.shared_gate ? P.shared_gate + t0 : nullptr;
        const cudaError_t e = launch_router_t<NCH, TT>(Q, cs, smem, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int NCH>
cudaError_t dispatch_nch(const RouterParams& P, cudaStream_t stream) {
    if (P.m <= 1) return dispatch_tt<NCH, 1>(P, stream);
    return dispatch_tt<NCH, 8 / NCH>(P, stream);
}

}  // namespace

cudaError_t launch_router(const float* x, const uint16_t* w, const float* bias, const uint16_t* w_sg, int m, int E,
                          int H, int top_k, int scoring, int normalize, float scale, int n_group, int topk_group,
                          int32_t* ids, float* weights, float* logits, float* shared_gate, cudaStream_t stream) {
    if (m == 0) return cudaSuccess;
    RouterParams P{};
    P.x = x; P.w = w; P.bias = bias; P.w_sg = w_sg;
    P.ids = ids; P.weights = weights; P.logits = logits; P.shared_gate = shared_gate;
    P.m = m; P.E = E; P.H = H; P.top_k = top_k;
    P.scoring = scoring; P.normalize = normalize; P.scale = scale;
    P.n_group = scoring == Q4K_ROUTE_SOFTMAX ? 1 : n_group;
    P.topk_group = scoring == Q4K_ROUTE_SOFTMAX ? 1 : topk_group;
    P.per = std::max(1, top_k / std::max(1, P.topk_group));
    const int nch = (H / 8 + kRThreads - 1) / kRThreads;
    if (nch <= 1) return dispatch_nch<1>(P, stream);
    if (nch <= 2) return dispatch_nch<2>(P, stream);
    if (nch <= 4) return dispatch_nch<4>(P, stream);
    return dispatch_nch<8>(P, stream);
}

int router_max_hidden() { return 8 * 8 * kRThreads; }

}  // namespace q4k

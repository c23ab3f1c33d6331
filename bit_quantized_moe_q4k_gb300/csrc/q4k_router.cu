// q4k_router.cu -- the router of a MoE layer: gate logits, top-k choice and routing weights,
// producing the ids and weights the layer's bucketing and combine read.
//
// moeflux expert_forward.rs (MoeBuffers::gate_logits): the router's gate logits are one fp32
// per expert from a bf16 matvec of the layer input; its `noaux_tc` routing and the
// softmax + top-K + normalise routing (synth::expert_weights_seeded) turn them into the
// chosen experts and their weights.
//
// Two launches, the second a programmatic dependent of the first (its launch overlaps the
// first's run):
//  * router_logits_kernel: the gate matvec over every SM. A CTA takes up to 8 consecutive
//    expert rows (as few as keep about two CTAs per SM busy) of one token tile; each of its
//    threads holds 8-column chunks of the tile's activations in registers and issues the
//    loads of all its rows at once, so one HBM round trip serves the whole CTA.
//  * router_topk_kernel: one warp per token chooses from the logits (in shared memory) and
//    writes ids and weights.
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
#include "q4k_route.cuh"

namespace q4k {
namespace {

constexpr int kRThreads = 256;
constexpr int kRWarps = kRThreads / 32;
// the choice's per-token tables (logits, corrected scores)
constexpr size_t kTopkSmemBudget = 160 * 1024;

struct RouterParams {
    const float* x;         // [m, hidden]
    const uint16_t* w;      // [num_experts, hidden] bf16
    const float* bias;      // [num_experts] or null
    const uint16_t* w_sg;   // [hidden] bf16 shared-expert gate row, or null
    int32_t* ids;           // [m, top_k]
    float* weights;         // [m, top_k]
    float* logits;          // [m, num_experts]
    float* shared_gate;     // [m] (with w_sg)
    int m, E, H, top_k;
    int scoring, normalize;
    float scale;
    int n_group, topk_group, per;
    int rb;                 // rows per CTA of the logits kernel
    int tile;               // tokens per CTA (logits kernel: <= its TT; top-k kernel: warps)
};

__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prev() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Gate logits of rows [blockIdx.x*rb, +rb) of the (expert rows, then the shared-expert gate
// row) for the token tile blockIdx.y.
template <int NCH, int TT>
__global__ void __launch_bounds__(kRThreads, 1) router_logits_kernel(const RouterParams P) {
    constexpr int RB = 8 / NCH;  // a thread's weight registers: RB * NCH chunks of 16 bytes
    __shared__ float s_red[kRWarps][RB * TT];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.y * P.tile;
    const int nt = min(P.tile, P.m - t0);
    const int rows = P.E + (P.w_sg ? 1 : 0);
    const int r0 = blockIdx.x * P.rb;
    const int nchunk = P.H / 8;
    pdl_trigger();
    // the weights do not depend on the previous kernel: their loads go out before the wait
    uint4 wv[RB][NCH];
#pragma unroll
    for (int b = 0; b < RB; ++b) {
        const int row = r0 + b;
        const uint16_t* wr = row < P.E ? P.w + (int64_t)row * P.H : P.w_sg;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int q = tid + c * kRThreads;
            wv[b][c] = (b < P.rb && row < rows && q < nchunk) ? __ldg(reinterpret_cast<const uint4*>(wr) + q)
                                                              : make_uint4(0, 0, 0, 0);
        }
    }
    pdl_wait_prev();  // x may come from the previous kernel
    float xr[TT][NCH][8];
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int q = tid + c * kRThreads;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (t < nt && q < nchunk) {
                const float4* src = reinterpret_cast<const float4*>(P.x + (int64_t)(t0 + t) * P.H) + 2 * q;
                a = __ldcg(src);
                b = __ldcg(src + 1);
            }
            xr[t][c][0] = a.x; xr[t][c][1] = a.y; xr[t][c][2] = a.z; xr[t][c][3] = a.w;
            xr[t][c][4] = b.x; xr[t][c][5] = b.y; xr[t][c][6] = b.z; xr[t][c][7] = b.w;
        }
#pragma unroll
    for (int b = 0; b < RB; ++b) {
        if (b >= P.rb) break;
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            float s = 0.0f;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                const uint32_t u[4] = {wv[b][c].x, wv[b][c].y, wv[b][c].z, wv[b][c].w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    s = __fmaf_rn(route_bf16_lo(u[h]), xr[t][c][2 * h], s);
                    s = __fmaf_rn(route_bf16_hi(u[h]), xr[t][c][2 * h + 1], s);
                }
            }
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
            if (lane == 0) s_red[warp][b * TT + t] = s;
        }
    }
    __syncthreads();
    if (tid < P.rb * TT) {
        const int b = tid / TT, t = tid % TT;
        const int row = r0 + b;
        if (row < rows && t < nt) {
            float s = s_red[0][b * TT + t];
#pragma unroll
            for (int w = 1; w < kRWarps; ++w) s = __fadd_rn(s, s_red[w][b * TT + t]);
            if (row < P.E) P.logits[(int64_t)(t0 + t) * P.E + row] = s;
            else P.shared_gate[t0 + t] = s;
        }
    }
}

// The choice for the tile's tokens (token blockIdx.x * tile + warp) from their logits.
__global__ void __launch_bounds__(kRThreads) router_topk_kernel(const RouterParams P) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = P.E, K = P.top_k;
    // tables: logits [tile][E], corrected scores [tile][E], bias [E]
    float* s_lg = reinterpret_cast<float*>(smem);
    float* s_cs = s_lg + (size_t)P.tile * E;
    float* s_bias = s_cs + (size_t)P.tile * E;
    pdl_trigger();
    const int t_base = blockIdx.x * P.tile;
    const int nt = min(P.tile, P.m - t_base);
    const bool grouped = P.scoring != Q4K_ROUTE_SOFTMAX;
    if (grouped)  // a launch input: read before the wait
        for (int e = tid; e < E; e += kRThreads) s_bias[e] = P.bias ? __ldg(P.bias + e) : 0.0f;
    pdl_wait_prev();  // the logits kernel
    {   // the tile's logits: independent loads, four per thread in flight
        const float* src = P.logits + (int64_t)t_base * E;
        const int total = nt * E;
        for (int i0 = 0; i0 < total; i0 += 4 * kRThreads) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * kRThreads + tid;
                v[u] = i < total ? __ldcg(src + i) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * kRThreads + tid;
                if (i < total) s_lg[i] = v[u];
            }
        }
    }
    __syncthreads();
    if (warp >= nt) return;
    const int t = t_base + warp;
    float* lg = s_lg + (size_t)warp * E;
    float* cs = s_cs + (size_t)warp * E;
    RouteRule R{E, K, P.scoring, P.normalize, P.n_group, P.topk_group, P.per, P.scale};
    int my_i;
    float my_w;
    route_token(lg, cs, grouped ? s_bias : nullptr, R, lane, my_i, my_w);
    if (lane < K) {
        P.ids[(int64_t)t * K + lane] = my_i;
        P.weights[(int64_t)t * K + lane] = my_w;
    }
}

cudaError_t launch_pdl(const void* kern, dim3 grid, size_t smem, cudaStream_t stream, const RouterParams& P) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kRThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {const_cast<RouterParams*>(&P)};
    return cudaLaunchKernelExC(&cfg, kern, args);
}

template <int NCH, int TT>
cudaError_t launch_logits(RouterParams P, cudaStream_t stream) {
    constexpr int RB = 8 / NCH;
    P.tile = std::min(TT, P.m);
    const int tiles = (P.m + P.tile - 1) / P.tile;
    const int rows = P.E + (P.w_sg ? 1 : 0);
    // rows per CTA: as many as keep about two CTAs per SM (at most RB)
    const int64_t target = 2 * (int64_t)num_sms();
    const int64_t want = ((int64_t)rows * tiles + target - 1) / target;
    P.rb = (int)std::max<int64_t>(1, std::min<int64_t>(RB, want));
    const int blocks = (rows + P.rb - 1) / P.rb;
    for (int t0 = 0; t0 < tiles; t0 += 32768) {  // the grid's y extent
        RouterParams Q = P;
        const int nt = std::min(32768, tiles - t0);
        Q.m = std::min(P.m - t0 * P.tile, nt * P.tile);
        Q.x = P.x + (int64_t)t0 * P.tile * P.H;
        Q.logits = P.logits + (int64_t)t0 * P.tile * P.E;
        Q.shared_gate = P.shared_gate ? P.shared_gate + (int64_t)t0 * P.tile : nullptr;
        const cudaError_t e = launch_pdl(reinterpret_cast<const void*>(router_logits_kernel<NCH, TT>),
                                         dim3((unsigned)blocks, (unsigned)nt, 1), 0, stream, Q);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int NCH>
cudaError_t dispatch_nch(const RouterParams& P, cudaStream_t stream) {
    if (P.m <= 1) return launch_logits<NCH, 1>(P, stream);
    return launch_logits<NCH, 8 / NCH>(P, stream);
}

}  // namespace

int num_sms();

// The router's first launch alone: logits [m, E] (+ the shared gate logits with w_sg).
cudaError_t launch_router_logits(const float* x, const uint16_t* w, const uint16_t* w_sg, int m, int E, int H,
                                 float* logits, float* shared_gate, cudaStream_t stream) {
    if (m == 0) return cudaSuccess;
    RouterParams P{};
    P.x = x; P.w = w; P.w_sg = w_sg;
    P.logits = logits; P.shared_gate = shared_gate;
    P.m = m; P.E = E; P.H = H;
    const int nch = (H / 8 + kRThreads - 1) / kRThreads;
    return nch <= 1 ? dispatch_nch<1>(P, stream)
         : nch <= 2 ? dispatch_nch<2>(P, stream)
         : nch <= 4 ? dispatch_nch<4>(P, stream)
                    : dispatch_nch<8>(P, stream);
}

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
    cudaError_t e = launch_router_logits(x, w, w_sg, m, E, H, logits, shared_gate, stream);
    if (e != cudaSuccess) return e;
    // the choice: tokens per CTA (one warp each) as many as their tables fit
    RouterParams Q = P;
    Q.tile = (int)std::min<size_t>(kRWarps, std::max<size_t>(1, (kTopkSmemBudget - (size_t)E * 4) / ((size_t)E * 8)));
    const size_t smem = (size_t)Q.tile * E * 8 + (size_t)E * 4;
    static bool attr_set[64] = {};  // the largest plan, set once per device
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(router_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(kTopkSmemBudget + 16));
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    return launch_pdl(reinterpret_cast<const void*>(router_topk_kernel), dim3((unsigned)((m + Q.tile - 1) / Q.tile)),
                      (smem + 15) & ~(size_t)15, stream, Q);
}

int router_max_hidden() { return 8 * 8 * kRThreads; }

}  // namespace q4k

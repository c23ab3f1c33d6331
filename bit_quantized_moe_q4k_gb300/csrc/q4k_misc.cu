// q4k_misc.cu -- the layer's small kernels: pair bucketing, combine, the Q4_K quantizer
// (weight preparation) and the loads-only ceiling kernel used for measurement.
#include <cuda_fp16.h>

#include "q4k_bucket.cuh"
#include "q4k_internal.cuh"

namespace q4k {

// ------------------------------------------------------------------------------------------
// Pair bucketing: stable counting sort of the pairs by expert (one CTA).
// moeflux expert_forward.rs (`encode_moe_batched_permute_fuse`: bucket the (token, slot)
// tuples by expert id; `encode_moe_gather_id_fuse`: the map0 step builds per-expert pair
// lists on the GPU). Out-of-range ids form a trailing bucket after offsets[E].
constexpr int kBucketThreads = 1024;

__global__ void __launch_bounds__(kBucketThreads)
bucket_kernel(const int32_t* __restrict__ ids, int n_pairs, int num_experts, int32_t* __restrict__ counts,
              int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int* err_flag) {
    extern __shared__ int smem[];
    int* s_cnt = smem;                        // num_experts + 1 (last = invalid bucket)
    int* s_run = s_cnt + num_experts + 1;     // num_experts + 1 running cursors
    __shared__ int s_warp[33];
    __shared__ int s_bad;
    const int E = num_experts;
    block_histogram(ids, n_pairs, E, s_cnt, &s_bad);
    for (int e = threadIdx.x; e < E; e += blockDim.x) counts[e] = s_cnt[e];
    if (threadIdx.x == 0) {
        s_cnt[E] = s_bad;
        if (s_bad) raise_flag(err_flag, Q4K_ERR_EXPERT_ID);
    }
    __syncthreads();
    block_exclusive_scan(s_cnt, E + 1, s_warp);  // s_cnt[e] = offsets[e]
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        offsets[e] = e < E ? s_cnt[e] : s_cnt[E];
        s_run[e] = 0;
    }
    if (threadIdx.x == 0) offsets[E] = s_cnt[E];
    __syncthreads();
    // Stable scatter: chunks of blockDim pairs; within a chunk the warps take turns so that
    // lower pair indices always claim lower slots of their bucket.
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int base = 0; base < n_pairs; base += blockDim.x) {
        const int p = base + threadIdx.x;
        const bool live = p < n_pairs;
        int e = -1;
        if (live) { e = ids[p]; if (!id_valid(e, E)) e = E; }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        const int leader = __ffs(peers) - 1;
        const int active_warps = min((n_pairs - base + 31) >> 5, (int)(blockDim.x >> 5));
        for (int w = 0; w < active_warps; ++w) {
            if (warp == w) {
                int start = 0;
                if (live && lane == leader) {
                    start = s_run[e];
                    s_run[e] = start + __popc(peers);
                }
                start = __shfl_sync(peers, start, leader);
                if (live) perm[s_cnt[e] + start + rank] = p;
            }
            __syncthreads();
        }
    }
}

cudaError_t launch_bucket(const int32_t* ids, int n_pairs, int num_experts, int32_t* counts,
                          int32_t* offsets, int32_t* perm, int* err_flag, cudaStream_t stream) {
    size_t smem = sizeof(int) * 2 * (size_t)(num_experts + 1);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(bucket_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    bucket_kernel<<<1, kBucketThreads, smem, stream>>>(ids, n_pairs, num_experts, counts, offsets, perm, err_flag);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// Combine: hidden_out = h_mid + sum_k w_k * expert_out_k + g * shared_out
// (moeflux expert_forward.rs, `combine_kernel_name` and
// `encode_moe_combine_residual_n_tokens`). One thread per 4 consecutive hidden elements
// of one token. All of a thread's loads are issued before any sum (one round trip, not one per
// slot); the slot sum then runs in slot order. KS: slots the thread holds (8 for top_k <= 8,
// which keeps it at 64 registers, else 16). y may alias h_mid (each element is read before it
// is written by the same thread). ids != null (the layer's combine): a pair whose id is outside
// [0, num_experts) contributes nothing, as in the combine fused into the down launch, which gives
// the same sums bit for bit.
template <int KS>
__global__ void __launch_bounds__(256)
combine_kernel(const float* h_mid, const float* __restrict__ expert_out, const float* __restrict__ weights,
               const float* __restrict__ shared_out, const float* __restrict__ shared_gate, int shared_mode,
               int top_k, int hidden, float* y, const int32_t* __restrict__ ids, int num_experts) {
    const int t = blockIdx.y;
    const int h4 = blockIdx.x * blockDim.x + threadIdx.x;  // float4 index within the row
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (h4 * 4 >= hidden) return;
    const int64_t row = (int64_t)t * hidden + h4 * 4;
    // everything read here may come from earlier kernels (programmatic dependent launch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float4 e[KS];
    float w[KS];
    bool ok[KS];
#pragma unroll
    for (int s = 0; s < KS; ++s) {  // independent loads (the rows of bad ids exist, unused)
        const int64_t p = (int64_t)t * top_k + s;
        ok[s] = s < top_k && (!ids || id_valid(ids[p], num_experts));
        w[s] = s < top_k ? weights[p] : 0.0f;
        e[s] = s < top_k ? *reinterpret_cast<const float4*>(expert_out + p * hidden + h4 * 4)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const bool sh = shared_mode != Q4K_SHARED_NONE;
    const float4 so = sh ? *reinterpret_cast<const float4*>(shared_out + row) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float gl = sh && shared_mode == Q4K_SHARED_SIGMOID ? shared_gate[t] : 0.0f;
    float4 acc = *reinterpret_cast<const float4*>(h_mid + row);
#pragma unroll
    for (int s = 0; s < KS; ++s) {
        if (!ok[s]) continue;
        acc.x = fmaf(w[s], e[s].x, acc.x);
        acc.y = fmaf(w[s], e[s].y, acc.y);
        acc.z = fmaf(w[s], e[s].z, acc.z);
        acc.w = fmaf(w[s], e[s].w, acc.w);
    }
    if (sh) {
        const float g = shared_mode == Q4K_SHARED_SIGMOID ? 1.0f / (1.0f + expf(-gl)) : 1.0f;
        acc.x = fmaf(g, so.x, acc.x);
        acc.y = fmaf(g, so.y, acc.y);
        acc.z = fmaf(g, so.z, acc.z);
        acc.w = fmaf(g, so.w, acc.w);
    }
    *reinterpret_cast<float4*>(y + row) = acc;
}

cudaError_t launch_combine(const float* h_mid, const float* expert_out, const float* weights,
                           const float* shared_out, const float* shared_gate, int shared_mode, int m,
                           int top_k, int hidden, float* y, bool pdl, cudaStream_t stream, const int32_t* ids,
                           int num_experts) {
    const int threads = 256;
    dim3 grid((hidden / 4 + threads - 1) / threads, m);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, top_k <= 8 ? combine_kernel<8> : combine_kernel<Q4K_MAX_TOP_K>, h_mid, expert_out, weights, shared_out, shared_gate,
                              shared_mode, top_k, hidden, y, ids, num_experts);
}

// ------------------------------------------------------------------------------------------
// Q4_K quantizer (weight preparation). Eight threads per 256-weight block, one per
// 32-weight sub-block. Every arithmetic step is an explicit round-to-nearest binary32
// operation (no contraction), so the bytes are reproducible on any IEEE host.
__global__ void __launch_bounds__(256)
quantize_kernel(const float* __restrict__ x, int64_t n_blocks, uint8_t* __restrict__ out) {
    const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t blk = gt >> 3;
    const int j = (int)(gt & 7);
    const unsigned grp = 0xFFu << (threadIdx.x & 24);  // the 8 lanes of this block
    if (blk >= n_blocks) return;  // whole 8-lane groups leave together
    const float* xs = x + blk * kQK + 32 * j;
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float4 f = *reinterpret_cast<const float4*>(xs + 4 * i);
        v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    }
    float lo = 0.0f, hi = v[0];
#pragma unroll
    for (int i = 0; i < 32; ++i) { lo = fminf(lo, v[i]); hi = fmaxf(hi, v[i]); }
    const float scale = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
    // -lo, but +0 when lo is zero: the block's dmin = fp16(max mn / 63) must not become -0
    const float mn = __fsub_rn(0.0f, lo);
    float max_scale = scale, max_mn = mn;
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
        max_scale = fmaxf(max_scale, __shfl_xor_sync(grp, max_scale, off));
        max_mn = fmaxf(max_mn, __shfl_xor_sync(grp, max_mn, off));
    }
    const __half d16 = __float2half_rn(__fdiv_rn(max_scale, 63.0f));
    const __half dmin16 = __float2half_rn(__fdiv_rn(max_mn, 63.0f));
    const float d = __half2float(d16), dmin = __half2float(dmin16);
    int sc = d > 0.0f ? (int)rintf(__fdiv_rn(scale, d)) : 0;
    int mq = dmin > 0.0f ? (int)rintf(__fdiv_rn(mn, dmin)) : 0;
    sc = min(sc, 63);
    mq = min(mq, 63);
    const float ds = __fmul_rn(d, (float)sc);
    const float dm = __fmul_rn(dmin, (float)mq);
    // 32 codes of this sub-block, 4 bits each, packed low-to-high in 4 words of 8 codes
    uint32_t packed[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        int q = 0;
        if (ds > 0.0f) {
            q = (int)rintf(__fdiv_rn(__fadd_rn(v[i], dm), ds));
            q = max(0, min(15, q));
        }
        // code byte i of the 32-byte group holds this code in its low (j even) or high (j odd) nibble
        packed[i >> 3] |= (uint32_t)q << (4 * (i & 7));
    }
    // Spread 8 codes per word into bytes: byte b gets code b in its low nibble.
    uint32_t bytes[8];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t c = packed[w];
        bytes[2 * w] = (c & 0xFu) | ((c >> 4 & 0xFu) << 8) | ((c >> 8 & 0xFu) << 16) | ((c >> 12 & 0xFu) << 24);
        bytes[2 * w + 1] = (c >> 16 & 0xFu) | ((c >> 20 & 0xFu) << 8) | ((c >> 24 & 0xFu) << 16) | ((c >> 28 & 0xFu) << 24);
    }
    // Pair sub-blocks 2c (low nibbles) and 2c+1 (high nibbles) into the shared 32 code bytes.
    uint32_t mine[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        uint32_t other = __shfl_xor_sync(grp, bytes[w], 1);
        mine[w] = (j & 1) ? 0u : (bytes[w] | (other << 4));
    }
    uint8_t* ob = out + blk * kBlockBytes;
    if ((j & 1) == 0) {
        uint4* dst = reinterpret_cast<uint4*>(ob + 16 + 32 * (j >> 1));
        dst[0] = make_uint4(mine[0], mine[1], mine[2], mine[3]);
        dst[1] = make_uint4(mine[4], mine[5], mine[6], mine[7]);
    }
    // Header: d, dmin and the 12 scale bytes (GGML Q4_K placement).
    int scv[8], mnv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        scv[i] = __shfl_sync(grp, sc, (threadIdx.x & 24) + i);
        mnv[i] = __shfl_sync(grp, mq, (threadIdx.x & 24) + i);
    }
    if (j == 0) {
        uint8_t s[12];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s[i] = (uint8_t)(scv[i] | ((scv[i + 4] >> 4) << 6));
            s[i + 4] = (uint8_t)(mnv[i] | ((mnv[i + 4] >> 4) << 6));
            s[i + 8] = (uint8_t)((scv[i + 4] & 0xF) | ((mnv[i + 4] & 0xF) << 4));
        }
        const uint32_t h0 = (uint32_t)__half_as_ushort(d16) | ((uint32_t)__half_as_ushort(dmin16) << 16);
        uint32_t w1 = s[0] | (s[1] << 8) | (s[2] << 16) | ((uint32_t)s[3] << 24);
        uint32_t w2 = s[4] | (s[5] << 8) | (s[6] << 16) | ((uint32_t)s[7] << 24);
        uint32_t w3 = s[8] | (s[9] << 8) | (s[10] << 16) | ((uint32_t)s[11] << 24);
        *reinterpret_cast<uint4*>(ob) = make_uint4(h0, w1, w2, w3);
    }
}

cudaError_t launch_quantize(const float* x, int64_t rows, int k, uint8_t* out, cudaStream_t stream) {
    const int64_t n_blocks = rows * (k / kQK);
    const int64_t threads_total = n_blocks * 8;
    const int threads = 256;
    const int64_t grid = (threads_total + threads - 1) / threads;
    if (grid == 0) return cudaSuccess;
    quantize_kernel<<<(unsigned)grid, threads, 0, stream>>>(x, n_blocks, out);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// Loads-only ceiling: the weight stream's access pattern (coalesced 16-byte loads, several
// in flight per thread) with the arithmetic replaced by an XOR, after the `ld` kernel of
// cortiq-engine examples/mv_lab.rs ("ceiling of the access pattern").
constexpr int kCeilThreads = 512;

__global__ void __launch_bounds__(kCeilThreads)
stream_ceiling_kernel(const uint4* __restrict__ src, uint64_t n16, uint32_t* __restrict__ sink) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t acc = 0;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride);
        uint4 c = __ldcs(src + i + 2 * stride), d = __ldcs(src + i + 3 * stride);
        acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
    }
    for (; i < n16; i += stride) {
        uint4 a = __ldcs(src + i);
        acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, off);
    __shared__ uint32_t s[kCeilThreads / 32];
    if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t r = 0;
        for (int w = 0; w < kCeilThreads / 32; ++w) r ^= s[w];
        sink[blockIdx.x] = r;
    }
}

int stream_ceiling_grid() { return num_sms() * 4; }

cudaError_t launch_stream_ceiling(const void* src, uint64_t bytes, uint32_t* sink, cudaStream_t stream) {
    stream_ceiling_kernel<<<stream_ceiling_grid(), kCeilThreads, 0, stream>>>(
        reinterpret_cast<const uint4*>(src), bytes / 16, sink);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// Gather of a few small buffers into device memory in one launch (the host-buffer layer call
// uses it to read its page-locked inputs straight from host memory: one launch instead of one
// copy-engine transfer per buffer). Sizes are multiples of 4 bytes; 4-byte words.
// A thread loads its word of every buffer before storing any, so the reads of host memory
// cost one round trip. The next kernel (the layer, launched as a programmatic dependent, which
// waits for this kernel before reading its results) may start its prologue right away; this
// launch itself is ordinary, since it overwrites buffers the previous kernel reads.
__global__ void __launch_bounds__(256) gather_kernel(const GatherSpec G) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t w = blockIdx.x * blockDim.x + threadIdx.x;; w += stride) {
        uint32_t v[5];
        bool any = false;
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            if (i < G.n && w < G.bytes[i] / 4) {
                v[i] = static_cast<const uint32_t*>(G.src[i])[w];
                any = true;
            }
        }
#pragma unroll
        for (int i = 0; i < 5; ++i)
            if (i < G.n && w < G.bytes[i] / 4) static_cast<uint32_t*>(G.dst[i])[w] = v[i];
        if (!any) break;
    }
}

cudaError_t launch_gather(const GatherSpec& g, cudaStream_t stream) {
    uint32_t words = 0;
    for (int i = 0; i < g.n; ++i) words = g.bytes[i] / 4 > words ? g.bytes[i] / 4 : words;
    if (words == 0) return cudaSuccess;
    const uint32_t grid = (words + 255) / 256 < 64 ? (words + 255) / 256 : 64;
    gather_kernel<<<grid, 256, 0, stream>>>(g);
    return cudaGetLastError();
}

}  // namespace q4k

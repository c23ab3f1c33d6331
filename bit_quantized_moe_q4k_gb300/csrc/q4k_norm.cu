// q4k_norm.cu -- RMSNorm chained after a MoE layer's combine: the next layer's input norm.
//
// moeflux expert_forward.rs (ChainToNormed, the chain appendix of the K-expert encoder):
// after the combine, rms_norm_sum_sq then rms_norm_apply_bf16 with the next layer's
// input-norm weight (bf16) and eps turn the combine's output into the next layer's normed
// input. Here both steps are one kernel, one CTA per token:
//   out[t, h] = x[t, h] * r_t * bf16(w[h]),  r_t = 1 / sqrt(sum_h x[t, h]^2 / hidden + eps)
// in fp32: each thread squares and adds its float4 columns (h = 4*(tid + 256 i)) left to
// right, the 32 lanes of a warp are added by xor shuffles (1 .. 16), the 8 warps in warp
// order; sqrt and the division are IEEE (correctly rounded). Launched as a programmatic
// dependent of the layer: the launch overlaps the layer's tail and waits for it before
// reading x.
#include <cuda_runtime.h>
#include <stdint.h>

#include "q4k_internal.cuh"

namespace q4k {
namespace {

constexpr int kNThreads = 256;

__global__ void __launch_bounds__(kNThreads) rms_norm_kernel(const float* x, const uint16_t* __restrict__ w,
                                                             int hidden, float eps, float* out) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ float s_part[kNThreads / 32];
    __shared__ float s_r;
    const int t = blockIdx.x, tid = threadIdx.x;
    const float4* xr = reinterpret_cast<const float4*>(x + (int64_t)t * hidden);
    const int nq = hidden / 4;
    float ss = 0.0f;
    for (int q = tid; q < nq; q += kNThreads) {
        const float4 v = __ldcg(xr + q);  // written by the previous kernel: read from L2
        ss = __fmaf_rn(v.x, v.x, ss);
        ss = __fmaf_rn(v.y, v.y, ss);
        ss = __fmaf_rn(v.z, v.z, ss);
        ss = __fmaf_rn(v.w, v.w, ss);
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
    if ((tid & 31) == 0) s_part[tid >> 5] = ss;
    __syncthreads();
    if (tid == 0) {
        float s = s_part[0];
#pragma unroll
        for (int i = 1; i < kNThreads / 32; ++i) s = __fadd_rn(s, s_part[i]);
        s_r = 1.0f / sqrtf(__fadd_rn(__fdiv_rn(s, (float)hidden), eps));
    }
    __syncthreads();
    const float r = s_r;
    float4* o = reinterpret_cast<float4*>(out + (int64_t)t * hidden);
    const uint2* wq = reinterpret_cast<const uint2*>(w);
    for (int q = tid; q < nq; q += kNThreads) {
        const float4 v = __ldcg(xr + q);
        const uint2 b = __ldg(wq + q);
        float4 y;
        y.x = __fmul_rn(__fmul_rn(v.x, r), __uint_as_float(b.x << 16));
        y.y = __fmul_rn(__fmul_rn(v.y, r), __uint_as_float(b.x & 0xFFFF0000u));
        y.z = __fmul_rn(__fmul_rn(v.z, r), __uint_as_float(b.y << 16));
        y.w = __fmul_rn(__fmul_rn(v.w, r), __uint_as_float(b.y & 0xFFFF0000u));
        o[q] = y;
    }
}

}  // namespace

cudaError_t launch_rms_norm(const float* x, const uint16_t* w, int m, int hidden, float eps, float* out,
                            cudaStream_t stream) {
    if (m == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)m);
    cfg.blockDim = dim3(kNThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rms_norm_kernel, x, w, hidden, eps, out);
}

}  // namespace q4k

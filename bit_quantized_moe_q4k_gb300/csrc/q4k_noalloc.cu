// q4k_noalloc.cu -- q4k_expert_ffn_forward_noalloc: the routed expert FFN with its scratch in
// a fixed, library-owned device array instead of a caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory when they run the layer. A plugin
// hosted by an application that owns every device allocation cannot call cudaMalloc itself;
// a latency-critical loop cannot afford the implicit synchronisation cudaMalloc/cudaFree may
// cause; a process whose device memory is fully reserved up front has nothing left to
// allocate from. Such callers still pass their own inputs and outputs, but the intermediate
// gate|up activations (m*top_k*inter floats) go to the array below.
//
// The array is 4 MiB (kNoAllocScratchBytes) of global memory that every GPU which loads
// this library keeps until the process exits. It is shared by every call on a device and
// keeps the last call's contents; the FFN overwrites every row it reads, so nothing in it
// needs clearing between calls. Calls that overlap on the GPU (concurrent streams, or
// several host threads) race on it: serialise them.
#include <cstdint>
#include <mutex>

#include "q4k_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevicesNoAlloc = 64;
void* g_scratch_addr[kMaxDevicesNoAlloc] = {};
std::mutex g_scratch_mutex;

// Device address of g_noalloc_scratch for the current device. The host-side name of a
// __device__ variable is only a stand-in, so the address is looked up once per device (with
// that device current) and reused.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevicesNoAlloc) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

bool aligned16_na(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int shape_ok(int num_experts, int m, int top_k, int n, int k) {
    if (m < 0 || num_experts < 1) return Q4K_ERR_SHAPE;
    if (num_experts > q4k::kMaxExperts) return Q4K_ERR_LIMIT;
    if (top_k < 1 || top_k > Q4K_MAX_TOP_K) return Q4K_ERR_TOPK;
    if (n < 1 || n % 4 != 0 || k < 1 || k % q4k::kQK != 0) return Q4K_ERR_SHAPE;
    if (k > q4k::kMaxK) return Q4K_ERR_LIMIT;
    return Q4K_OK;
}

}  // namespace

extern "C" size_t q4k_expert_ffn_noalloc_max_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int q4k_expert_ffn_forward_noalloc(const void* d_w_gate, const void* d_w_up, const void* d_w_down,
                                              int num_experts, const float* d_h_post, const int32_t* d_ids, int m,
                                              int top_k, int hidden, int inter, float* d_expert_out, int* d_err_flag,
                                              cudaStream_t stream) {
    int st = shape_ok(num_experts, m, top_k, inter, hidden);
    if (!st) st = shape_ok(num_experts, m, top_k, hidden, inter);
    if (st) {
        q4k::set_last_error(st, "q4k_expert_ffn_forward_noalloc: invalid shape or top_k");
        return st;
    }
    if (!d_w_gate || !d_w_up || !d_w_down || !d_h_post || !d_ids || !d_expert_out) {
        q4k::set_last_error(Q4K_ERR_NULL, "q4k_expert_ffn_forward_noalloc: NULL pointer argument");
        return Q4K_ERR_NULL;
    }
    if (!aligned16_na(d_w_gate) || !aligned16_na(d_w_up) || !aligned16_na(d_w_down) || !aligned16_na(d_h_post)) {
        q4k::set_last_error(Q4K_ERR_ALIGN, "q4k_expert_ffn_forward_noalloc: slabs and h_post must be 16-byte aligned");
        return Q4K_ERR_ALIGN;
    }
    const size_t need = (size_t)m * top_k * inter * sizeof(float);
    if (need > kNoAllocScratchBytes) {
        q4k::set_last_error(Q4K_ERR_LIMIT,
                            "q4k_expert_ffn_forward_noalloc: m*top_k*inter*4 bytes exceed the 4 MiB static scratch");
        return Q4K_ERR_LIMIT;
    }
    if (m == 0) return Q4K_OK;
    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        q4k::set_last_error(Q4K_ERR_CUDA, cudaGetErrorString(e));
        return Q4K_ERR_CUDA;
    }
    float* act = static_cast<float*>(scratch);
    q4k::GemvGroup g{static_cast<const uint8_t*>(d_w_gate), static_cast<const uint8_t*>(d_w_up), d_ids, d_h_post,
                     hidden, 0, act, num_experts, m, top_k, inter, hidden};
    e = q4k::launch_idgemv(&g, 1, true, false, d_err_flag, stream);
    if (e == cudaSuccess) {
        q4k::GemvGroup d{static_cast<const uint8_t*>(d_w_down), nullptr, d_ids, act, (int64_t)top_k * inter, inter,
                         d_expert_out, num_experts, m, top_k, hidden, inter};
        e = q4k::launch_idgemv(&d, 1, false, true, d_err_flag, stream);
    }
    if (e != cudaSuccess) {
        q4k::set_last_error(Q4K_ERR_CUDA, cudaGetErrorString(e));
        return Q4K_ERR_CUDA;
    }
    return Q4K_OK;
}

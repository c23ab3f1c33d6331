// q4k_internal.cuh -- declarations shared by the CUDA translation units of libq4kmoe.
// Nothing here is part of the C ABI (that is include/q4kmoe.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "q4kmoe.h"

namespace q4k {

constexpr int kQK = 256;          // weights per Q4_K super-block
constexpr int kBlockBytes = 144;  // bytes per super-block
constexpr int kMaxExperts = 4096; // bucketing bound (shared-memory tables)
constexpr int kMaxK = 65536;

// Device error flag helper: records the first error code, never traps.
__device__ __forceinline__ void raise_flag(int* flag, int code) {
    if (flag) atomicCAS(flag, 0, code);
}

// -------------------------------------------------------------------------------------------
// Per-CTA pair bucketing (the map0 step of the layer: bucket (token, slot) pairs by expert).
// Computed redundantly by every CTA of a GEMV launch from the ids in L2, so no separate
// launch and no global synchronisation is needed before the weight stream starts.
struct BucketView {
    int n_experts_used;  // U: experts with at least one valid pair
};

// Launchers (defined in q4k_misc.cu / q4k_gemv.cu). All return cudaError_t of the launch.
cudaError_t launch_bucket(const int32_t* ids, int n_pairs, int num_experts, int32_t* counts,
                          int32_t* offsets, int32_t* perm, int* err_flag, cudaStream_t stream);
// True (once) when the calling thread's last id-GEMV launch joined a side stream back into its
// stream: the next launch should then not be a programmatic dependent.
bool take_after_join();
cudaError_t launch_combine(const float* h_mid, const float* expert_out, const float* weights,
                           const float* shared_out, const float* shared_gate, int shared_mode, int m,
                           int top_k, int hidden, float* y, bool pdl, cudaStream_t stream,
                           const int32_t* ids = nullptr, int num_experts = 0);
cudaError_t launch_fmt4(int fmt, const uint8_t* w, const uint8_t* w2, uint64_t expert_stride, uint64_t s_off,
                        uint64_t b_off, int gs, int num_experts, const float* a, int64_t outer, int64_t inner,
                        const int32_t* ids, int m, int top_k, int n, int k, float* out, int* err_flag,
                        cudaStream_t stream);
cudaError_t launch_router(const float* x, const uint16_t* w, const float* bias, const uint16_t* w_sg, int m, int E,
                          int H, int top_k, int scoring, int normalize, float scale, int n_group, int topk_group,
                          int32_t* ids, float* weights, float* logits, float* shared_gate, cudaStream_t stream);
int router_max_hidden();
cudaError_t launch_rms_norm(const float* x, const uint16_t* w, int m, int hidden, float eps, float* out,
                            cudaStream_t stream);
cudaError_t launch_quantize(const float* x, int64_t rows, int k, uint8_t* out, cudaStream_t stream);
cudaError_t launch_stream_ceiling(const void* src, uint64_t bytes, uint32_t* sink, cudaStream_t stream);
// Up to 5 small copies (sizes multiples of 4 bytes) in one launch; sources may be host memory
// the device can address (page-locked, its device view).
struct GatherSpec {
    const void* src[5];
    void* dst[5];
    uint32_t bytes[5];
    int n;
};
cudaError_t launch_gather(const GatherSpec& g, cudaStream_t stream);
int stream_ceiling_grid();

// One projection group of an id-GEMV launch: a stacked slab and how its pairs read rows.
struct GemvGroup {
    const uint8_t* w;        // slab base (16-byte aligned), expert e at w + e * n * row_bytes
    const uint8_t* w2;       // second slab read with the same rows (up, for the fused gate|up), or null
    const int32_t* ids;      // [m * top_k] expert ids, or null = every pair uses expert 0
    const float* a;          // activations
    int64_t outer, inner;    // src1 walk in floats
    float* out;              // [m * top_k, n] output rows
    int num_experts, m, top_k, n, k;
};

// Launch the bucketed Q4_K id-GEMV over up to two groups in one grid (the routed experts
// and the shared expert of a layer). fused_swiglu: out = silu(w . x) * (w2 . x).
// pdl: the launch may start while the previous kernel of the stream drains (programmatic
// dependent launch); the kernel waits for it before reading activations, or, with
// pdl_wait_first, before reading anything (for the first launch of a layer, whose ids and
// activations the previous kernel may have written).
// The combine fused into a down launch (group 0 = routed experts, group 1 = shared expert):
// the last CTA to finish a row tile forms, for those rows of every token,
//   y = h_mid + sum_s weights[t*top_k+s] * out0[t*top_k+s] + g_t * out1[t]
// in slot order (deterministic). counters: one per row tile (n_counters words; the launch
// fails with cudaErrorInvalidValue if its tiling needs more), zero on entry, left zero.
struct CombineSpec {
    float* y;
    const float* h_mid;
    const float* weights;
    const float* shared_gate;
    int shared_mode;
    unsigned* counters;
    int n_counters;
};

// tc_min > 0: experts with at least tc_min pairs run on the tensor-core grouped GEMM
// (q4k_tc.cu) first, using tc_img[g] (tc_image_bytes of the group) as scratch; the rest run on
// the id-GEMV kernel. combine: fuse the combine into this (down) launch. zero / n_zero: CTA 0
// zeroes these words before anything else (the gate|up launch prepares the counters the
// following down launch uses).
// Rows of a one-slab launch quantized once by launch_prestage (per group, or null): pair p's
// staged planes at planes[g] + p * (k/64) * 144 bytes, its (delta, sum X) at meta[g] + p * (k/32).
struct PreStaged {
    const uint8_t* planes[2];
    const float2* meta[2];
};
// Bytes of `rows` staged rows of length k (planes and (delta, sum X) pairs).
int64_t prestage_bytes(int rows, int k);
// Quantize the activation rows of the groups with planes into PreStaged (a programmatic
// dependent launch that waits for the previous kernel before reading).
cudaError_t launch_prestage(const GemvGroup* groups, int n_groups, const PreStaged& pre, cudaStream_t stream);

cudaError_t launch_idgemv(const GemvGroup* groups, int n_groups, bool fused_swiglu, bool pdl, int* err_flag,
                          cudaStream_t stream, int tc_min = 0, uint8_t* const* tc_img = nullptr,
                          const CombineSpec* combine = nullptr, unsigned* zero = nullptr, int n_zero = 0,
                          bool pdl_wait_first = false, const PreStaged* pre = nullptr);
// rows per id-GEMV work item for a given k (bucketed kernel)
int idgemv_tile_rows(int k);
cudaError_t launch_tc(const GemvGroup* groups, int n_groups, bool fused, int tc_min, uint8_t* const* img,
                      int* err_flag, cudaStream_t stream, bool pdl = true);
size_t tc_image_bytes(int n_pairs, int k, int tc_min);
bool tc_fits(const GemvGroup* groups, int n_groups);  // the tensor-core kernel's shared memory plan fits

// The small-batch layer in one persistent launch (q4k_layer.cu): gu / dn the groups of the
// gate|up and down halves (routed, then shared; their float outputs unused: the results go to
// tagged words in the sync area), cb the combine (counters unused). sync: sync_words words of
// the layer workspace (layer_sync_words), any contents. Returns
// cudaErrorNotSupported, before launching anything, where it does not apply (more than 32
// pairs in a group, a sync area too small, rows too long for its shared memory).
size_t layer_sync_words(int m, int top_k, int hidden, int inter, int shared_inter);
// Both halves' work items fit one round of the CTAs the device's SMs hold at once.
bool layer_one_round(int m, int top_k, int hidden, int inter, int shared_inter);
// Which kernel a single-launch layer of these sizes takes on the current device: 2 the wide
// kernel, 1 the four-warp kernel (or no device to ask), 0 none (the layer takes two launches).
int layer_kernel_kind(int m, int top_k, int num_experts, int hidden, int inter, int shared_inter);

cudaError_t launch_layer_persistent(const GemvGroup* gu, const GemvGroup* dn, int n_groups, const CombineSpec& cb,
                                    uint64_t* sync, size_t sync_words, int* err_flag, cudaStream_t stream);

int num_sms();

// Limit of every bounded wait inside the single-launch layer kernels, in nanoseconds: the
// environment variable Q4K_WAIT_NS when set to a positive number (read at every launch), else
// 2 s. A wait that runs out raises Q4K_ERR_TIMEOUT in the device error flag.
uint64_t wait_limit_ns();

// Record the calling thread's last error text (read back by q4k_last_error_string).
void set_last_error(int status, const char* message);

}  // namespace q4k

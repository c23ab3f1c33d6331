/*
 * q4kmoe.h -- C ABI of the GB300 (sm_103a) Q4_K mixture-of-experts layer library.
 *
 * The operations follow the studied pages' statement of the problem:
 *   [P1] ferrum-kernels 0.7.7, src/backend/metal/q4_k_moe_id_gemv_batched.rs
 *        (`dispatch_gemv_q4k_moe_id_batched_on_encoder`: argument list, the
 *        preconditions k % 256 == 0, n % 4 == 0, the row and expert strides
 *        nb01 = (k/256)*144 and nb02 = n*nb01, the src1 outer/inner walk);
 *   [P2] moeflux 0.1.0-pre.3, src/riir/moe/expert_forward.rs (the expert FFN
 *        gate -> up -> SwiGLU -> down, `ExpertPayload`, the `MAX_K` = 16 slot
 *        bound and `BadK`, the sigmoid-gated / unscaled shared expert in
 *        `combine_kernel_name`, the batched combine
 *        `encode_moe_combine_residual_n_tokens`, and the expert bucketing of
 *        `encode_moe_batched_permute_fuse` / `encode_moe_gather_id_fuse`);
 *   [P3] cortiq-engine 0.7.7, examples/mv_lab.rs (4-bit matvec kernel variants and
 *        the loads-only `ld` kernel that gives the access pattern's ceiling).
 *
 * Data formats
 *   Q4_K block: 256 weights in 144 bytes: fp16 d, fp16 dmin, 12 bytes of
 *   packed 6-bit scales and mins (GGML Q4_K placement), 128 bytes of 4-bit
 *   codes; w = d*sc*q - dmin*m. A projection with n outputs and k inputs is
 *   n rows of k/256 blocks; a stacked slab is num_experts such matrices back
 *   to back (expert e starts at byte e*n*(k/256)*144).
 *   Activations, outputs and routing weights are fp32, ids are int32.
 *   A (token, slot) pair has index p = token*top_k + slot.
 *
 * Conventions of every call
 *   - Pointers named d_* or documented as device memory are device pointers
 *     owned by the caller; the library allocates no device memory and keeps no
 *     pointer past the call. The one global device state is the static scratch
 *     array of q4k_expert_ffn_forward_noalloc (4 MiB per device, part of the
 *     library image); after a cudaDeviceReset the process must not call that
 *     entry point again (the address it keeps belongs to the old context). A call
 *     whose experts take the tensor-core path also keeps, per device and host
 *     thread, one CUDA stream and two events (created on first use, made anew if
 *     they stop working): its tensor-core kernels run on that stream beside its
 *     id-GEMV kernel, joined back into `stream` before anything reads their rows.
 *   - Waits inside a kernel for work of other CTAs of the same launch are bounded
 *     in time: the environment variable Q4K_WAIT_NS (nanoseconds, read at every
 *     call; default 2 s) sets the limit, after which the kernel stops waiting, sets
 *     *err_flag to Q4K_ERR_TIMEOUT and returns.
 *   - Calls are asynchronous on `stream` (the last argument) and return a
 *     q4k_status. Host-side validation happens before anything is enqueued;
 *     on an error status nothing was enqueued.
 *   - Expert ids are range-checked on the device: a pair whose id is outside
 *     [0, num_experts) gets an all-zero output row and, when `err_flag` is
 *     not NULL, the device int *err_flag is set to Q4K_ERR_EXPERT_ID. No trap,
 *     no host synchronisation. The caller zeroes *err_flag before the call.
 *   - Scratch memory comes from a caller-provided device `workspace` of at
 *     least the size the matching *_workspace_size() returns (256-byte aligned).
 *   - q4k_last_error_string() describes the last non-OK status of the calling
 *     thread.
 *   - m == 0 is an empty batch: the call validates, enqueues nothing and
 *     returns Q4K_OK.
 */
#ifndef Q4KMOE_H
#define Q4KMOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    Q4K_OK = 0,
    Q4K_ERR_NULL = 1,      /* a required pointer is NULL                                    */
    Q4K_ERR_SHAPE = 2,     /* k % 256 != 0, n % 4 != 0, m < 0, num_experts < 1, n or k < 1   */
    Q4K_ERR_TOPK = 3,      /* top_k outside [1, 16]                                          */
    Q4K_ERR_WORKSPACE = 4, /* workspace NULL, misaligned or smaller than required            */
    Q4K_ERR_CUDA = 5,      /* a CUDA runtime call or launch failed                           */
    Q4K_ERR_EXPERT_ID = 6, /* device flag value: some id was outside [0, num_experts)        */
    Q4K_ERR_ALIGN = 7,     /* slab not 16-byte aligned, or activation rows not 16-byte aligned */
    Q4K_ERR_MODE = 8,      /* shared_mode not in {0, 1, 2}                                   */
    Q4K_ERR_LIMIT = 9,     /* a size beyond an implementation limit (see each call)          */
    Q4K_ERR_TIMEOUT = 10   /* device flag value: a pipeline wait in a kernel gave up (bounded) */
} q4k_status;

#define Q4K_MAX_TOP_K 16
#define Q4K_SHARED_NONE 0
#define Q4K_SHARED_SIGMOID 1  /* g_t = 1 / (1 + exp(-shared_gate[t])) */
#define Q4K_SHARED_UNSCALED 2 /* g_t = 1                               */

/* Text of the calling thread's last non-OK status (never NULL). */
const char* q4k_last_error_string(void);

/* Library version string. */
const char* q4k_version(void);

/* ---------------------------------------------------------------------------------
 * Workspace sizing. Returns the bytes of device scratch the calls below need for
 * these sizes (0 on invalid sizes). q4k_moe_workspace_size covers q4k_moe_id_gemv
 * with n <= n_max, k <= k_max and q4k_expert_ffn_forward with hidden, inter <=
 * max(n_max, k_max); q4k_moe_layer_workspace_size covers q4k_moe_layer_forward.
 */
size_t q4k_moe_workspace_size(int m, int top_k, int num_experts, int n_max, int k_max);
size_t q4k_moe_layer_workspace_size(int m, int top_k, int num_experts, int hidden, int inter,
                                    int shared_inter);

/* ---------------------------------------------------------------------------------
 * q4k_moe_bucket -- pair bucketing [P2: bucket (token, slot) tuples by expert id].
 * Stable counting sort of the n_pairs pairs by expert id:
 *   d_counts[e]  = number of pairs with id e                       (num_experts ints)
 *   d_offsets[e] = exclusive prefix sum of d_counts, d_offsets[E] = valid pairs (E+1 ints)
 *   d_perm[d_offsets[e] .. d_offsets[e+1]) = the pairs with id e, increasing
 *   d_perm[d_offsets[E] .. n_pairs) = pairs with an out-of-range id, increasing.
 * The result is unique, so it is bit-exact with any correct implementation.
 * Limit: num_experts <= 4096 (Q4K_ERR_LIMIT otherwise).
 */
int q4k_moe_bucket(const int32_t* d_ids, int n_pairs, int num_experts, int32_t* d_counts,
                   int32_t* d_offsets, int32_t* d_perm, int* d_err_flag, cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * q4k_moe_id_gemv -- batched MoE indirect-dispatch GEMV [P1].
 * For every pair p < m*top_k, with t = p / top_k and s = p % top_k:
 *   out[p, r] = sum_c W_{ids[p]}[r, c] * a[t*src1_outer_stride + s*src1_inner_stride + c]
 * for r < n, c < k. W_e is the Q4_K [n, k] matrix of expert e in the slab at
 * d_w_stacked + w_byte_offset. Strides are in floats: gate/up use (k, 0) (the
 * token's row is broadcast to its slots), down uses (top_k*k, k) (one row per
 * pair). Pairs are bucketed by expert on the device so each touched slab row
 * is streamed once per call, whatever the number of pairs sharing it.
 *   d_w_stacked + w_byte_offset: 16-byte aligned, num_experts*n*(k/256)*144 bytes
 *   d_a: 16-byte aligned; strides multiples of 4 floats
 *   d_out: [m*top_k, n] fp32
 * d_workspace is optional here: when it holds at least q4k_moe_workspace_size(m, top_k,
 * num_experts, n, k) bytes (256-byte aligned), experts whose bucket holds at least t pairs
 * run on the tcgen05 tensor-core grouped GEMM; all others on the id-GEMV kernel. t is the
 * environment variable Q4K_TC_MIN when set (0 disables the path), else 2 when
 * m*top_k >= 2*num_experts or num_experts >= 64, else 4.
 * Limits: num_experts <= 4096, k <= 65536.
 */
int q4k_moe_id_gemv(const void* d_w_stacked, uint64_t w_byte_offset, int num_experts,
                    const float* d_a, int64_t src1_outer_stride, int64_t src1_inner_stride,
                    const int32_t* d_ids, int m, int top_k, int n, int k, float* d_out,
                    void* d_workspace, size_t ws_bytes, int* d_err_flag, cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * q4k_expert_ffn_forward -- routed expert FFN [P2: gate, up, SwiGLU, down].
 *   g[p, i] = gemv(W_gate, h_post; strides (hidden, 0))
 *   u[p, i] = gemv(W_up,   h_post; strides (hidden, 0))
 *   act[p, i] = silu(g) * u,  silu(x) = x / (1 + exp(-x))   (fused into the gate|up pass)
 *   expert_out[p, h] = gemv(W_down, act; strides (top_k*inter, inter))
 * d_w_gate / d_w_up: slabs of [num_experts][inter, hidden]; d_w_down: [num_experts][hidden, inter].
 * d_h_post: [m, hidden]; d_expert_out: [m*top_k, hidden]. The shared expert is this call
 * with num_experts = 1, top_k = 1 and all ids 0.
 */
int q4k_expert_ffn_forward(const void* d_w_gate, const void* d_w_up, const void* d_w_down,
                           int num_experts, const float* d_h_post, const int32_t* d_ids, int m,
                           int top_k, int hidden, int inter, float* d_expert_out,
                           void* d_workspace, size_t ws_bytes, int* d_err_flag, cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * q4k_expert_ffn_forward_noalloc -- q4k_expert_ffn_forward for callers that cannot allocate
 * device memory (no counterpart in the studied pages; an addition of this library).
 * Same computation, arguments and errors as q4k_expert_ffn_forward without the workspace:
 * the gate|up activations live in a 4 MiB array that the library keeps in every device's
 * global memory for the life of the process. The call allocates nothing. It serves code
 * that runs where it may not call cudaMalloc: a plugin inside an application that owns all
 * device allocations, a latency-critical loop that must not take the synchronisation an
 * allocation can cause, or a process whose device memory is fully reserved in advance.
 *   - Limit: m*top_k*inter*4 bytes <= q4k_expert_ffn_noalloc_max_scratch_bytes() (4 MiB);
 *     larger sizes return Q4K_ERR_LIMIT.
 *   - The first call on a device looks up the array's device address (with that device
 *     current) and keeps it; make that first call before any stream capture. A device
 *     reset (cudaDeviceReset) after that first call is not supported: the kept address
 *     belongs to the context the reset destroyed.
 *   - Every call on a device shares the array and leaves its contents behind; the call
 *     overwrites all it reads, so nothing needs clearing. Calls that overlap on the GPU
 *     (other streams, other host threads) race on it and must be serialised by the caller.
 *   - Large buckets do not take the tensor-core path here (it needs workspace images).
 */
size_t q4k_expert_ffn_noalloc_max_scratch_bytes(void);
int q4k_expert_ffn_forward_noalloc(const void* d_w_gate, const void* d_w_up, const void* d_w_down,
                                   int num_experts, const float* d_h_post, const int32_t* d_ids, int m,
                                   int top_k, int hidden, int inter, float* d_expert_out, int* d_err_flag,
                                   cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * moe_combine_residual -- combine [P2: hidden_out = h_mid + sum_k w_k * expert_out_k
 * + shared term].
 *   hidden_out[t, h] = h_mid[t, h] + sum_{s<top_k} weights[t*top_k+s] * expert_out[t*top_k+s, h]
 *                      + g_t * shared_out[t, h]
 * with g_t per shared_mode (NONE: no term, shared_out / shared_gate may be NULL;
 * SIGMOID: g_t = 1/(1+exp(-shared_gate[t])); UNSCALED: g_t = 1, shared_gate may be NULL).
 * The slot sum runs in slot order (deterministic, no atomics). hidden_out may alias
 * h_mid. Requires hidden % 4 == 0 and 16-byte aligned rows.
 */
int moe_combine_residual(const float* d_h_mid, const float* d_expert_out, const float* d_weights,
                         const float* d_shared_out, const float* d_shared_gate, int shared_mode,
                         int m, int top_k, int hidden, float* d_hidden_out, cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * q4k_moe_layer_forward -- one MoE layer: routed FFN, shared-expert FFN and combine.
 *   y = moe_combine_residual(h_mid, q4k_expert_ffn_forward(routed),
 *                            weights, q4k_expert_ffn_forward(shared), shared_gate)
 * Shared slabs (one expert, intermediate shared_inter) are NULL and shared_inter 0
 * when shared_mode is NONE. All device pointers; d_y [m, hidden] may alias d_h_mid.
 * Contains no host synchronisation, so it can be captured in a CUDA graph.
 * Launches: a layer with at most 32 routed pairs (m*top_k <= 32), no bucket large
 * enough for the tensor-core path, and halves whose work items each fit one round of the
 * CTAs the device holds at once (a decode layer) is ONE persistent launch whose CTAs
 * hand results to each other as launch-tagged words (and tagged flags) at the start of the
 * workspace; any other layer is a gate|up launch and a down launch with the combine fused
 * into it (+ the tensor-core kernels of a half that uses them); beyond 4 tokens the combine
 * is a launch of its own, over all outputs, after the down launch. All give the same
 * results bit for bit. The environment variable Q4K_SINGLE_LAUNCH=1 takes every layer the
 * single launch can run (the first condition alone) that way, =0 none. The workspace
 * needs no initialisation: the flag words of a launch carry a tag derived from a
 * generation word that the launch advances, so leftovers of earlier calls (or of
 * anything else) never match; its counters are used only when the previous call on the
 * workspace zeroed them and stamped them with this call's tag (else the call polls flags).
 * Concurrent calls on one workspace race, as with any scratch. The single launch is a
 * cooperative launch, so the driver starts it only with every CTA resident; when the
 * driver refuses that grid (fewer CTAs fit than the occupancy query said, e.g. SMs held by
 * another client) the call runs the two launches instead. After a device error flag
 * Q4K_ERR_TIMEOUT (a bounded wait gave up) zero the workspace before its next use.
 */
int q4k_moe_layer_forward(const void* d_w_gate, const void* d_w_up, const void* d_w_down,
                          int num_experts, const void* d_ws_gate, const void* d_ws_up,
                          const void* d_ws_down, int shared_inter, int shared_mode,
                          const float* d_h_post, const float* d_h_mid, const int32_t* d_ids,
                          const float* d_weights, const float* d_shared_gate, int m, int top_k,
                          int hidden, int inter, float* d_y, void* d_workspace, size_t ws_bytes,
                          int* d_err_flag, cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * The two halves of q4k_moe_layer_forward, for callers that schedule the layer
 * themselves (the fused gate + up + SiLU batched id-GEMV of ferrum-kernels'
 * q4_k_moe_id_gate_up_silu_batched, then the down projection), each running the
 * routed experts and the shared expert in one launch:
 *   q4k_moe_layer_gate_up: d_act[p, :] = silu(W_gate . x) * (W_up . x) for the routed pairs
 *     (x = h_post row of the pair's token) and d_act_shared[t, :] likewise for the shared
 *     expert (d_act [m*top_k, inter], d_act_shared [m, shared_inter]).
 *   q4k_moe_layer_down: d_expert_out[p, :] = W_down . d_act[p, :] and
 *     d_shared_out[t, :] = W_sdown . d_act_shared[t, :].
 * shared_inter == 0 (and NULL shared pointers) means no shared expert.
 */
int q4k_moe_layer_gate_up(const void* d_w_gate, const void* d_w_up, int num_experts, const void* d_ws_gate,
                          const void* d_ws_up, int shared_inter, const float* d_h_post, const int32_t* d_ids,
                          int m, int top_k, int hidden, int inter, float* d_act, float* d_act_shared,
                          void* d_workspace, size_t ws_bytes, int* d_err_flag, cudaStream_t stream);
int q4k_moe_layer_down(const void* d_w_down, int num_experts, const void* d_ws_down, int shared_inter,
                       const float* d_act, const float* d_act_shared, const int32_t* d_ids, int m, int top_k,
                       int hidden, int inter, float* d_expert_out, float* d_shared_out, void* d_workspace,
                       size_t ws_bytes, int* d_err_flag, cudaStream_t stream);
/* Optional workspace of one half (k_routed = hidden for gate|up, inter for down; k_shared =
 * hidden / shared_inter): with at least this many bytes (256-byte aligned), experts whose
 * bucket holds many tokens run on the tensor-core grouped GEMM. 0 when that path is off. */
size_t q4k_moe_layer_half_workspace_size(int m, int top_k, int k_routed, int shared_inter, int k_shared);

/* Number of kernels one q4k_moe_layer_forward call with its full workspace launches for these
 * sizes on the current device (1 for the single-launch layer; else 2, plus 2 per half that
 * takes the tensor-core path, plus 1 for the pre-staging of down rows of 4096 or more
 * elements, plus 1 for the combine beyond 4 tokens). 0 on invalid sizes. */
int q4k_moe_layer_launch_count(int m, int top_k, int num_experts, int hidden, int inter, int shared_inter);

/* Which kernels one q4k_moe_layer_forward call runs for these sizes on the current device
 * (the environment switches included):
 *   Q4K_PATH_PERSISTENT one persistent launch for the whole layer (a decode layer);
 *   Q4K_PATH_PERSISTENT_WIDE the same with 256-thread CTAs, each taking at most one work item of
 *                       each half from tiles in shared memory (decode layers that allow it;
 *                       Q4K_LAYER_WIDE=0 switches it off);
 *   Q4K_PATH_TWO_LAUNCH a gate|up launch and a down launch with the combine fused, or after
 *                       it beyond 4 tokens (plus the tensor-core kernels of a half that uses
 *                       them).
 * Both give the same results bit for bit. -1 on invalid sizes. */
#define Q4K_PATH_TWO_LAUNCH 0
#define Q4K_PATH_PERSISTENT 1
#define Q4K_PATH_PERSISTENT_WIDE 2
int q4k_moe_layer_path(int m, int top_k, int num_experts, int hidden, int inter, int shared_inter);

/* ---------------------------------------------------------------------------------
 * q4k_moe_layer_forward_host -- the same layer with the per-step inputs and the
 * output in HOST memory. Weights and the workspace stay in device memory. The inputs
 * h_post, h_mid, ids, weights and shared_gate land in the staging area behind the
 * layer's workspace, the layer runs, y lands in host memory, all on `stream`; the
 * call returns once this is enqueued, so the caller synchronises `stream` before
 * reading y. Page-locked host buffers (cudaHostAlloc / cudaHostRegister, as
 * reported by cudaPointerGetAttributes) are read and written by the kernels
 * through their device view: one gather launch for all inputs, and the fused
 * combine stores y into host memory. Other host memory goes through
 * cudaMemcpyAsync, one transfer per buffer.
 * Workspace: q4k_moe_layer_workspace_size(...) + q4k_moe_layer_host_staging_size(...).
 */
size_t q4k_moe_layer_host_staging_size(int m, int top_k, int hidden);
int q4k_moe_layer_forward_host(const void* d_w_gate, const void* d_w_up, const void* d_w_down,
                               int num_experts, const void* d_ws_gate, const void* d_ws_up,
                               const void* d_ws_down, int shared_inter, int shared_mode,
                               const float* h_post, const float* h_mid, const int32_t* ids,
                               const float* weights, const float* shared_gate, int m, int top_k,
                               int hidden, int inter, float* y, void* d_workspace,
                               size_t ws_bytes, int* d_err_flag, cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * q4k_moe_id_gemv_fmt -- the batched id-GEMV of q4k_moe_id_gemv over two other 4-bit
 * weight formats (same pair walk, bucketing, outputs and id checks; d_w2 != NULL gives the
 * fused gate|up form out = silu(W . a) * (W2 . a), W2 read with the same offsets):
 *   Q4K_FMT_AFFINE4 [P2: the MLX-style affine expert blob, weights | scales | biases bound
 *     at three offsets, GROUP_SIZE]: expert e's [n, k] matrix starts at
 *     M = d_w + w_byte_offset + e*expert_stride: codes at M (row r: k/2 bytes from r*k/2;
 *     weight c of the row in nibble c%2 of byte c/2, low nibble first), bf16 scales
 *     [n, k/group_size] at M + scales_offset, bf16 biases [n, k/group_size] at
 *     M + biases_offset; w = scale * q + bias. group_size 32, 64 or 128.
 *   Q4K_FMT_Q4TP [P3: the q4tp matrix of mv_lab.rs' production kernel]: M as above holds
 *     the codes (row r group g's 32 weights in the 16 bytes at (r*k/32 + g)*16, weight order
 *     as above), then binary16 (base, step) per row at M + n*k/2 + 4r, then 5-bit group codes
 *     at M + n*k/2 + 4n with k/32*5/8 bytes per row (group g in bits 5g..5g+4, LSB first);
 *     w = (q - 8) * 2^(base + code*step). scales_offset, biases_offset, group_size unused.
 * Alignment: d_w (+ offset) and expert_stride multiples of 16; affine offsets multiples of 4.
 * Limits and the rest as q4k_moe_id_gemv (k % 256 == 0, n % 4 == 0, num_experts <= 4096).
 */
#define Q4K_FMT_AFFINE4 1
#define Q4K_FMT_Q4TP 2
int q4k_moe_id_gemv_fmt(int fmt, const void* d_w, const void* d_w2, uint64_t w_byte_offset,
                        uint64_t expert_stride, uint64_t scales_offset, uint64_t biases_offset,
                        int group_size, int num_experts, const float* d_a, int64_t src1_outer_stride,
                        int64_t src1_inner_stride, const int32_t* d_ids, int m, int top_k, int n, int k,
                        float* d_out, int* d_err_flag, cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * q4k_moe_router -- the layer's router [P2: MoeBuffers::gate_logits, the `noaux_tc`
 * routing, synth::expert_weights_seeded]: gate logits, top-k choice and routing weights,
 * written where q4k_moe_layer_forward reads ids, weights and shared_gate.
 *   logits[t, e] = sum_h bf16(w_router[e, h]) * x[t, h]   (fp32)
 *   scoring Q4K_ROUTE_SOFTMAX: the top_k largest logits, weight = softmax over all experts
 *     (normalize: divided by the chosen experts' sum).
 *   scoring Q4K_ROUTE_SIGMOID_GROUPED (noaux_tc): s = sigmoid(logit), the choice on
 *     s + bias (bias NULL: 0) among the experts of the topk_group best of n_group groups of
 *     consecutive ids, a group scored by the sum of its max(1, top_k/topk_group) best
 *     s + bias; weight = s (normalize: divided by the chosen s' sum) * scale.
 *   Choice order: larger score first, equal scores by the lower id; ids [m, top_k] int32 in
 *   that order, weights [m, top_k] fp32. d_logits [m, num_experts] fp32 (required) receives
 *   the logits, which the choice then reads. d_w_shared_gate (optional, bf16 [hidden]) adds
 *   the shared expert's gate logit d_shared_gate[t] = sum_h bf16(w_shared_gate[h]) * x[t, h].
 * Layouts: d_x [m, hidden] fp32; d_w_router [num_experts, hidden] bf16 bits (uint16),
 * both 16-byte aligned. Limits: hidden % 8 == 0, hidden <= 16384; num_experts <= 4096;
 * top_k <= min(16, num_experts); grouped: n_group <= 32 divides num_experts,
 * 1 <= topk_group <= n_group, max(1, top_k/topk_group) <= min(16, num_experts/n_group),
 * top_k <= topk_group * num_experts/n_group. Two launches: the gate matvec over all SMs,
 * then the choice (one warp per token), each a programmatic dependent of the kernel before
 * it in the stream; the result is the same bits at every call and for any m.
 */
#define Q4K_ROUTE_SOFTMAX 0
#define Q4K_ROUTE_SIGMOID_GROUPED 1
int q4k_moe_router(const float* d_x, const uint16_t* d_w_router, const float* d_bias,
                   const uint16_t* d_w_shared_gate, int m, int num_experts, int hidden, int top_k,
                   int scoring, int normalize, float scale, int n_group, int topk_group,
                   int32_t* d_ids, float* d_weights, float* d_logits, float* d_shared_gate,
                   cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * q4k_moe_layer_forward_routed -- the decode MoE block from the layer input: the router
 * (q4k_moe_router's logits, choice and weights, with d_w_shared_gate giving the shared
 * expert's gate logit), the layer (q4k_moe_layer_forward) and, when d_w_norm is given, the
 * next layer's input norm (q4k_rms_norm's formula) into d_normed.
 *   Arguments: those of q4k_moe_layer_forward without ids, weights and shared_gate, those of
 *   q4k_moe_router (w_router bf16 [num_experts, hidden], bias, scoring rule); d_w_norm bf16
 *   [hidden] (8-byte aligned) and eps, or NULL for no norm; d_normed [m, hidden] (may alias
 *   d_y); d_ids_out / d_weights_out [m, top_k] (both or neither) receive the choice.
 *   A sigmoid-gated shared expert needs d_w_shared_gate.
 * Launches: q4k_moe_router's two, q4k_moe_layer_forward's, then q4k_rms_norm's, each a
 * programmatic dependent of the kernel before it where that is safe (the persistent layer is a
 * cooperative launch); the ids, weights, y and normed are those of the three calls made one after
 * the other, bit for bit.
 * Workspace: q4k_moe_layer_routed_workspace_size(...) bytes, any contents (as the layer's).
 */
size_t q4k_moe_layer_routed_workspace_size(int m, int top_k, int num_experts, int hidden, int inter,
                                           int shared_inter);
int q4k_moe_layer_forward_routed(const void* d_w_gate, const void* d_w_up, const void* d_w_down,
                                 int num_experts, const void* d_ws_gate, const void* d_ws_up,
                                 const void* d_ws_down, int shared_inter, int shared_mode,
                                 const float* d_h_post, const float* d_h_mid,
                                 const uint16_t* d_w_router, const float* d_bias,
                                 const uint16_t* d_w_shared_gate, int scoring, int normalize,
                                 float scale, int n_group, int topk_group, int m, int top_k,
                                 int hidden, int inter, float* d_y, const uint16_t* d_w_norm,
                                 float eps, float* d_normed, int32_t* d_ids_out,
                                 float* d_weights_out, void* d_workspace, size_t ws_bytes,
                                 int* d_err_flag, cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * q4k_rms_norm -- RMSNorm chained after the combine [P2: ChainToNormed, rms_norm_sum_sq +
 * rms_norm_apply_bf16]: the next layer's normed input from this layer's output.
 *   out[t, h] = x[t, h] / sqrt(sum_h x[t, h]^2 / hidden + eps) * bf16(w[h])   (fp32)
 * d_x, d_out [m, hidden] fp32 (d_out may alias d_x), d_w bf16 [hidden]; 16-byte aligned
 * rows (hidden % 4 == 0), d_w 8-byte aligned. One launch, a programmatic dependent of the
 * previous kernel (its launch overlaps that kernel's tail).
 */
int q4k_rms_norm(const float* d_x, const uint16_t* d_w, int m, int hidden, float eps, float* d_out,
                 cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * q4k_quantize_rows -- fp32 [rows, k] -> Q4_K bytes [rows, k/256*144] on the device
 * (weight preparation; not part of the layer: the [P1] tests make their slabs by
 * quantizing fp32 weights with candle's Q4K, whose steps the page does not show, so
 * this is a min/max quantizer of the Q4_K format). Per 32-weight sub-block:
 * lo = min(0, min x), hi = max x, scale = (hi-lo)/15, mn = -lo; d = fp16(max scale/63),
 * dmin = fp16(max mn/63); sc = min(63, rint(scale/d)), m = min(63, rint(mn/dmin));
 * q = clamp(rint((x + dmin*m)/(d*sc)), 0, 15); every step one IEEE binary32
 * operation rounded to nearest even, so the bytes are reproducible bit for bit.
 * d_x 16-byte aligned; k % 256 == 0.
 */
int q4k_quantize_rows(const float* d_x, int64_t rows, int k, void* d_out, cudaStream_t stream);

/* ---------------------------------------------------------------------------------
 * q4k_stream_ceiling -- loads-only kernel [P3 `ld`] over `bytes` of device memory (16-byte
 * aligned, bytes % 16 == 0): the same coalesced 16-byte loads as the GEMV's weight
 * stream, reduced to one XOR word per CTA in d_sink (grid-sized, caller-provided,
 * at least q4k_stream_ceiling_sink_words() ints). A measurement tool: its
 * bandwidth is the ceiling the weight stream can reach.
 */
int q4k_stream_ceiling_sink_words(void);
int q4k_stream_ceiling(const void* d_src, uint64_t bytes, uint32_t* d_sink, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif

// q4k_api.cu -- the C ABI of libq4kmoe (declared in include/q4kmoe.h): host-side
// validation, workspace layout and kernel sequencing. No compute happens here.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <string>

#include "q4k_internal.cuh"

using namespace q4k;

namespace {

thread_local std::string g_last_error;

int fail(int status, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

int cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return Q4K_OK;
    return fail(Q4K_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by the GEMV-style calls (ferrum-kernels batched GEMV preconditions:
// k % 256 == 0, n % 4 == 0, top_k > 0, m > 0; top_k bounded by the slot limit of 16 of
// moeflux's MAX_K / BadK).
int check_gemv_shape(int num_experts, int m, int top_k, int n, int k) {
    if (m < 0) return fail(Q4K_ERR_SHAPE, "m must be >= 0 (got %d)", m);
    if (num_experts < 1) return fail(Q4K_ERR_SHAPE, "num_experts must be >= 1 (got %d)", num_experts);
    if (num_experts > kMaxExperts) return fail(Q4K_ERR_LIMIT, "num_experts must be <= %d (got %d)", kMaxExperts, num_experts);
    if (top_k < 1 || top_k > Q4K_MAX_TOP_K) return fail(Q4K_ERR_TOPK, "top_k must be in [1, %d] (got %d)", Q4K_MAX_TOP_K, top_k);
    if (n < 1 || n % 4 != 0) return fail(Q4K_ERR_SHAPE, "n must be a positive multiple of 4 (got %d)", n);
    if (k < 1 || k % kQK != 0) return fail(Q4K_ERR_SHAPE, "k must be a positive multiple of 256 (got %d)", k);
    if (k > kMaxK) return fail(Q4K_ERR_LIMIT, "k must be <= %d (got %d)", kMaxK, k);
    if ((int64_t)m * top_k > (int64_t)1 << 24) return fail(Q4K_ERR_LIMIT, "m*top_k too large (%lld)", (long long)m * top_k);
    return Q4K_OK;
}

// Tensor-core path policy: experts whose bucket holds at least t pairs run on the tcgen05
// grouped GEMM (q4k_tc.cu), the others on the id-GEMV kernel, the tensor-core launch first.
// t is the environment variable Q4K_TC_MIN when set (0 disables the path); otherwise 2 when
// the batch averages at least two pairs per expert; else, with at least 64 experts (about one
// pair each on average, but routed ids crowd some experts), 3 for gate|up and 2 for down (the
// down rows are short, and its buckets of two pairs run better on the tensor cores): on the
// Zipf-distributed Qwen3-like m = 16 layer 90.6 us against 92.9 us with 3 for both halves and
// 97.4 us with 2 for both (one GB300); else 8 (few experts with about one pair each: the
// path's two launches find hardly a bucket to take; Mixtral-like m = 4 200 us against
// 220-265 us with 2-4). A launch uses the path only when some bucket can reach t and the
// caller's workspace holds the activation images.
int tc_min_env() {
    static int v = [] {
        const char* s = getenv("Q4K_TC_MIN");
        return s ? atoi(s) : -1;
    }();
    return v;
}

int tc_min_for(int routed_pairs, int num_experts, bool down) {
    if (tc_min_env() >= 0) return tc_min_env();
    if ((int64_t)routed_pairs >= 2 * (int64_t)num_experts) return 2;
    if (num_experts >= 64) return down ? 2 : 3;
    return 8;
}

// Switch (environment, read at every call): Q4K_SINGLE_LAUNCH=1 runs every layer the single
// launch can take that way, 0 none; unset (-1): the layers each of whose halves fits one round
// of resident CTAs (there the saved launch is worth most; larger layers stream better as two).
int single_launch_setting() {
    const char* s = getenv("Q4K_SINGLE_LAUNCH");
    return s ? (atoi(s) != 0 ? 1 : 0) : -1;
}

// Workspace sizes do not depend on the expert count: size for the smallest threshold.
int tc_min_sizing() { return tc_min_env() >= 0 ? tc_min_env() : 2; }

// Worth it only with enough work to spread over the SMs: at least ~64 items of 128 weight
// rows x a chunk of <= 32 tokens (a single shared expert with a few row tiles stays on the
// id-GEMV kernel). Chunks: at least ceil(pairs / 32), and up to one per expert that can
// reach t pairs when the buckets are spread (min(experts, pairs / t)).
bool tc_wanted(int n_pairs, int num_experts, int n_rows, int t) {
    if (t <= 0 || n_pairs < t || (int64_t)n_pairs * 4 < (int64_t)t * num_experts) return false;
    const int64_t chunks = std::max<int64_t>((n_pairs + 31) / 32, std::min<int64_t>(num_experts, n_pairs / t));
    const int64_t items = chunks * ((n_rows + 127) / 128);
    return items >= 64;
}

// Would the two-launch layer send some bucket of either half to the tensor-core path?
bool layer_wants_tc(int m, int top_k, int num_experts, int hidden, int inter, int shared_inter) {
    const int tg = tc_min_for(m * top_k, num_experts, false), td = tc_min_for(m * top_k, num_experts, true);
    const bool sh = shared_inter > 0;
    return tc_wanted(m * top_k, num_experts, inter, tg) || (sh && tc_wanted(m, 1, shared_inter, tg)) ||
           tc_wanted(m * top_k, num_experts, hidden, td) || (sh && tc_wanted(m, 1, hidden, td));
}

// The two-launch layer fuses the combine into the down launch (the last item of a row tile
// combines it) up to this many tokens. Beyond, that one CTA's share (tokens x tile rows) grows
// long and holds the launch up, so the combine runs as a launch of its own over all outputs.
constexpr int kFusedCombineMaxM = 4;

// The layer runs as one persistent launch (q4k_layer.cu): a few pairs, no tensor-core bucket.
bool layer_single_launch(int m, int top_k, int num_experts, int hidden, int inter, int shared_inter) {
    const int setting = single_launch_setting();
    if (setting == 0 || layer_sync_words(m, top_k, hidden, inter, shared_inter) == 0 ||
        layer_wants_tc(m, top_k, num_experts, hidden, inter, shared_inter))
        return false;
    return setting == 1 || layer_one_round(m, top_k, hidden, inter, shared_inter);
}

size_t tc_scratch(int n_pairs, int k) {
    const int t = tc_min_sizing();
    return t > 0 ? align_up(tc_image_bytes(n_pairs, k, t)) : 0;
}

// FFN scratch: act [m*top_k, inter], then tensor-core images of gate|up (k = hidden) and down (k = inter)
size_t ffn_scratch(int m, int top_k, int hidden, int inter) {
    return align_up((size_t)m * top_k * inter * sizeof(float)) + tc_scratch(m * top_k, hidden) +
           tc_scratch(m * top_k, inter);
}

// Down rows at least this long are quantized once before the down launch (launch_prestage)
// rather than in every CTA that takes one of their items.
constexpr int kPrestageMinK = 4096;

// Shapes and rule of a router call (q4k_moe_router, q4k_moe_layer_forward_routed).
int check_router_args(int m, int num_experts, int hidden, int top_k, int scoring, int n_group, int topk_group) {
    if (m < 0) return fail(Q4K_ERR_SHAPE, "m must be >= 0 (got %d)", m);
    if (num_experts < 1) return fail(Q4K_ERR_SHAPE, "num_experts must be >= 1 (got %d)", num_experts);
    if (num_experts > kMaxExperts) return fail(Q4K_ERR_LIMIT, "num_experts must be <= %d (got %d)", kMaxExperts, num_experts);
    if (top_k < 1 || top_k > Q4K_MAX_TOP_K || top_k > num_experts)
        return fail(Q4K_ERR_TOPK, "top_k must be in [1, min(16, num_experts)] (got %d)", top_k);
    if (hidden < 8 || hidden % 8 != 0) return fail(Q4K_ERR_SHAPE, "hidden must be a positive multiple of 8 (got %d)", hidden);
    if (hidden > router_max_hidden()) return fail(Q4K_ERR_LIMIT, "hidden must be <= %d (got %d)", router_max_hidden(), hidden);
    if (scoring != Q4K_ROUTE_SOFTMAX && scoring != Q4K_ROUTE_SIGMOID_GROUPED)
        return fail(Q4K_ERR_MODE, "scoring must be Q4K_ROUTE_SOFTMAX or Q4K_ROUTE_SIGMOID_GROUPED (got %d)", scoring);
    if (scoring == Q4K_ROUTE_SIGMOID_GROUPED) {
        if (n_group < 1 || n_group > 32 || num_experts % n_group != 0)
            return fail(Q4K_ERR_SHAPE, "n_group must be in [1, 32] and divide num_experts (got %d)", n_group);
        if (topk_group < 1 || topk_group > n_group)
            return fail(Q4K_ERR_SHAPE, "topk_group must be in [1, n_group] (got %d)", topk_group);
        const int gsize = num_experts / n_group, per = std::max(1, top_k / topk_group);
        if (per > std::min(16, gsize) || top_k > topk_group * gsize)
            return fail(Q4K_ERR_SHAPE, "top_k %d cannot be chosen from %d groups of %d", top_k, topk_group, gsize);
    }
    return Q4K_OK;
}

// Scratch of the routed layer behind the layer's own workspace: the router's logits, the
// shared gate logits, ids and weights.
struct RouteScratch {
    size_t logits, sg, ids, weights, total;
};

RouteScratch route_scratch(size_t base, int m, int top_k, int num_experts, int hidden) {
    RouteScratch r{};
    size_t off = base;
    r.logits = off;  off += align_up((size_t)m * num_experts * sizeof(float));
    r.sg = off;      off += align_up((size_t)m * sizeof(float));
    r.ids = off;     off += align_up((size_t)m * top_k * sizeof(int32_t));
    r.weights = off; off += align_up((size_t)m * top_k * sizeof(float));
    r.total = off;
    return r;
}

struct LayerScratch {
    size_t sync, act, act_shared, eout, shared_out, tc_gu, tc_dn, counters, pre, pre_shared, total;
    size_t n_sync_words;  // 0: these shapes always take the two-launch layer
    int n_counters;
};

LayerScratch layer_scratch(int m, int top_k, int hidden, int inter, int shared_inter) {
    LayerScratch s{};
    size_t off = 0;
    // the single-launch layer's generation word, start tags and item flags come first, so the
    // generation word stays at offset 0 whatever the shapes of later calls
    s.n_sync_words = layer_sync_words(m, top_k, hidden, inter, shared_inter);
    s.sync = off;       off += align_up(s.n_sync_words * sizeof(uint64_t));
    s.act = off;        off += align_up((size_t)m * top_k * inter * sizeof(float));
    s.act_shared = off; off += align_up((size_t)m * shared_inter * sizeof(float));
    s.eout = off;       off += align_up((size_t)m * top_k * hidden * sizeof(float));
    s.shared_out = off; off += align_up((size_t)m * hidden * sizeof(float));
    s.tc_gu = off;      off += tc_scratch(m * top_k, hidden) + (shared_inter > 0 ? tc_scratch(m, hidden) : 0);
    s.tc_dn = off;      off += tc_scratch(m * top_k, inter) + (shared_inter > 0 ? tc_scratch(m, shared_inter) : 0);
    // combine counters of the down launch: one per row tile of hidden, for any tiling
    s.n_counters = hidden;
    s.counters = off;   off += align_up((size_t)s.n_counters * sizeof(unsigned));
    // staged down rows (routed pairs, then the shared expert's tokens) where they are long
    s.pre = off;        off += inter >= kPrestageMinK ? align_up((size_t)prestage_bytes(m * top_k, inter)) : 0;
    s.pre_shared = off; off += shared_inter >= kPrestageMinK ? align_up((size_t)prestage_bytes(m, shared_inter)) : 0;
    s.total = off;
    return s;
}

// The device's address of page-locked host memory (cudaHostAlloc / cudaHostRegister), usable by
// kernels on the current device; false for any other host memory (pageable, unknown).
bool host_device_view(const void* p, const void** out) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error of the query
        return false;
    }
    if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return false;
    *out = a.devicePointer;
    return true;
}

int check_workspace(void* ws, size_t ws_bytes, size_t need) {
    if (need == 0) return Q4K_OK;
    if (!ws) return fail(Q4K_ERR_WORKSPACE, "workspace is NULL but %zu bytes are needed", need);
    if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return fail(Q4K_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (ws_bytes < need) return fail(Q4K_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, need);
    return Q4K_OK;
}

// The groups of the two halves of a layer: routed experts, then (shared_inter > 0) the
// shared expert. Returns the group count.
int gate_up_groups(const void* w_gate, const void* w_up, int num_experts, const float* h_post, const int32_t* ids,
                   int m, int top_k, int hidden, int inter, float* act, const void* ws_gate, const void* ws_up,
                   int shared_inter, float* act_shared, GemvGroup* g) {
    g[0] = GemvGroup{static_cast<const uint8_t*>(w_gate), static_cast<const uint8_t*>(w_up), ids, h_post,
                     hidden, 0, act, num_experts, m, top_k, inter, hidden};
    if (shared_inter <= 0) return 1;
    g[1] = GemvGroup{static_cast<const uint8_t*>(ws_gate), static_cast<const uint8_t*>(ws_up), nullptr, h_post,
                     hidden, 0, act_shared, 1, m, 1, shared_inter, hidden};
    return 2;
}

int down_groups(const void* w_down, int num_experts, const float* act, const int32_t* ids, int m, int top_k,
                int hidden, int inter, float* expert_out, const void* ws_down, int shared_inter,
                const float* act_shared, float* shared_out, GemvGroup* g) {
    g[0] = GemvGroup{static_cast<const uint8_t*>(w_down), nullptr, ids, act, (int64_t)top_k * inter, inter,
                     expert_out, num_experts, m, top_k, hidden, inter};
    if (shared_inter <= 0) return 1;
    g[1] = GemvGroup{static_cast<const uint8_t*>(ws_down), nullptr, nullptr, act_shared, shared_inter, 0,
                     shared_out, 1, m, 1, hidden, shared_inter};
    return 2;
}

// Gate|up + SwiGLU of the routed experts and (when shared_inter > 0) the shared expert, in
// one launch; then the down projections of both, in one launch.
int run_gate_up(const void* w_gate, const void* w_up, int num_experts, const float* h_post, const int32_t* ids,
                int m, int top_k, int hidden, int inter, float* act, const void* ws_gate, const void* ws_up,
                int shared_inter, float* act_shared, int* err_flag, cudaStream_t stream, uint8_t* tc_ws = nullptr,
                unsigned* zero = nullptr, int n_zero = 0) {
    GemvGroup g[2] = {};
    const int ng = gate_up_groups(w_gate, w_up, num_experts, h_post, ids, m, top_k, hidden, inter, act, ws_gate,
                                  ws_up, shared_inter, act_shared, g);
    int tc = 0;
    uint8_t* img[2] = {nullptr, nullptr};
    const int t = tc_min_for(m * top_k, num_experts, false);
    if (tc_ws && (tc_wanted(m * top_k, num_experts, inter, t) || (shared_inter > 0 && tc_wanted(m, 1, shared_inter, t)))) {
        tc = t;
        img[0] = tc_ws;
        img[1] = tc_ws + tc_scratch(m * top_k, hidden);
    }
    // a programmatic dependent launch that waits before reading anything: only the launch of its
    // CTAs overlaps the previous kernel's tail
    return cuda_status(launch_idgemv(g, ng, true, true, err_flag, stream, tc, img, nullptr, zero, n_zero, true),
                       "gate|up launch");
}

int run_down(const void* w_down, int num_experts, const float* act, const int32_t* ids, int m, int top_k,
             int hidden, int inter, float* expert_out, const void* ws_down, int shared_inter, const float* act_shared,
             float* shared_out, int* err_flag, cudaStream_t stream, uint8_t* tc_ws = nullptr,
             const CombineSpec* combine = nullptr, uint8_t* pre_ws = nullptr, uint8_t* pre_shared_ws = nullptr) {
    GemvGroup g[2] = {};
    const int ng = down_groups(w_down, num_experts, act, ids, m, top_k, hidden, inter, expert_out, ws_down,
                               shared_inter, act_shared, shared_out, g);
    // long rows: quantize each once (a launch between gate|up and down) for the down items to copy
    PreStaged pre{};
    uint8_t* pre_ws_g[2] = {inter >= kPrestageMinK ? pre_ws : nullptr,
                            shared_inter >= kPrestageMinK ? pre_shared_ws : nullptr};
    bool any_pre = false;
    for (int gi = 0; gi < ng; ++gi) {
        if (!pre_ws_g[gi]) continue;
        const int rows = g[gi].m * g[gi].top_k;
        pre.planes[gi] = pre_ws_g[gi];
        pre.meta[gi] = reinterpret_cast<const float2*>(pre_ws_g[gi] + (int64_t)rows * (g[gi].k / 64) * 144);
        any_pre = true;
    }
    if (any_pre) {
        const int st = cuda_status(launch_prestage(g, ng, pre, stream), "prestage launch");
        if (st) return st;
    }
    int tc = 0;
    uint8_t* img[2] = {nullptr, nullptr};
    const int t = tc_min_for(m * top_k, num_experts, true);
    if (tc_ws && (tc_wanted(m * top_k, num_experts, hidden, t) || (shared_inter > 0 && tc_wanted(m, 1, hidden, t)))) {
        tc = t;
        img[0] = tc_ws;
        img[1] = tc_ws + tc_scratch(m * top_k, inter);
    }
    return cuda_status(launch_idgemv(g, ng, false, true, err_flag, stream, tc, img, combine, nullptr, 0, false,
                                     any_pre ? &pre : nullptr),
                       "down launch");
}

int run_ffn(const void* w_gate, const void* w_up, const void* w_down, int num_experts, const float* h_post,
            const int32_t* ids, int m, int top_k, int hidden, int inter, float* act, float* expert_out,
            const void* ws_gate, const void* ws_up, const void* ws_down, int shared_inter, float* act_shared,
            float* shared_out, int* err_flag, cudaStream_t stream, uint8_t* tc_gu = nullptr,
            uint8_t* tc_dn = nullptr) {
    int st = run_gate_up(w_gate, w_up, num_experts, h_post, ids, m, top_k, hidden, inter, act, ws_gate, ws_up,
                         shared_inter, act_shared, err_flag, stream, tc_gu);
    if (st) return st;
    return run_down(w_down, num_experts, act, ids, m, top_k, hidden, inter, expert_out, ws_down, shared_inter,
                    act_shared, shared_out, err_flag, stream, tc_dn);
}

// Tensor-core image scratch of one half of the layer: routed group then shared group.
size_t tc_half_scratch(int m, int top_k, int k_routed, int shared_inter, int k_shared) {
    return tc_scratch(m * top_k, k_routed) + (shared_inter > 0 ? tc_scratch(m, k_shared) : 0);
}

// Validation shared by the layer entry points (shapes of both projections, shared expert).
int check_layer(const void* w_a, const void* w_b, int num_experts, int shared_inter, const void* s_a,
                const void* s_b, int m, int top_k, int hidden, int inter) {
    int st = check_gemv_shape(num_experts, m, top_k, inter, hidden);
    if (!st) st = check_gemv_shape(num_experts, m, top_k, hidden, inter);
    if (st) return st;
    if (shared_inter < 0) return fail(Q4K_ERR_SHAPE, "shared_inter must be >= 0");
    if (shared_inter > 0) {
        st = check_gemv_shape(1, m, 1, shared_inter, hidden);
        if (!st) st = check_gemv_shape(1, m, 1, hidden, shared_inter);
        if (st) return st;
        if (!s_a || (s_b == nullptr && w_b != nullptr)) return fail(Q4K_ERR_NULL, "shared expert slab is NULL");
        if (!aligned16(s_a) || (s_b && !aligned16(s_b))) return fail(Q4K_ERR_ALIGN, "shared slabs must be 16-byte aligned");
    }
    if (!w_a) return fail(Q4K_ERR_NULL, "NULL slab");
    if (!aligned16(w_a) || (w_b && !aligned16(w_b))) return fail(Q4K_ERR_ALIGN, "slabs must be 16-byte aligned");
    return Q4K_OK;
}

}  // namespace

void q4k::set_last_error(int status, const char* message) { fail(status, "%s", message); }

extern "C" {

const char* q4k_last_error_string(void) { return g_last_error.c_str(); }

const char* q4k_version(void) { return "libq4kmoe 0.1 (sm_103a)"; }

size_t q4k_moe_workspace_size(int m, int top_k, int num_experts, int n_max, int k_max) {
    if (m < 0 || top_k < 1 || top_k > Q4K_MAX_TOP_K || num_experts < 1 || n_max < 1 || k_max < 1) return 0;
    const int mx = n_max > k_max ? n_max : k_max;
    return ffn_scratch(m, top_k, mx, mx);
}

size_t q4k_moe_layer_workspace_size(int m, int top_k, int num_experts, int hidden, int inter, int shared_inter) {
    if (m < 0 || top_k < 1 || top_k > Q4K_MAX_TOP_K || num_experts < 1 || hidden < 1 || inter < 1 || shared_inter < 0)
        return 0;
    return layer_scratch(m, top_k, hidden, inter, shared_inter).total;
}

int q4k_moe_layer_launch_count(int m, int top_k, int num_experts, int hidden, int inter, int shared_inter) {
    if (m <= 0 || top_k < 1 || num_experts < 1) return 0;
    if (layer_single_launch(m, top_k, num_experts, hidden, inter, shared_inter)) return 1;
    const int tg = tc_min_for(m * top_k, num_experts, false), td = tc_min_for(m * top_k, num_experts, true);
    const bool tc_gu = tc_wanted(m * top_k, num_experts, inter, tg) || (shared_inter > 0 && tc_wanted(m, 1, shared_inter, tg));
    const bool tc_dn = tc_wanted(m * top_k, num_experts, hidden, td) || (shared_inter > 0 && tc_wanted(m, 1, hidden, td));
    // the down rows' pre-staging (a launch between the halves) for rows of kPrestageMinK or more
    const bool pre = inter >= kPrestageMinK || (shared_inter > 0 && shared_inter >= kPrestageMinK);
    return 2 + (tc_gu ? 2 : 0) + (tc_dn ? 2 : 0) + (pre ? 1 : 0) + (m > kFusedCombineMaxM ? 1 : 0);
}

int q4k_moe_layer_path(int m, int top_k, int num_experts, int hidden, int inter, int shared_inter) {
    if (m <= 0 || top_k < 1 || top_k > Q4K_MAX_TOP_K || num_experts < 1 || hidden < 1 || inter < 1 ||
        shared_inter < 0)
        return -1;
    if (layer_single_launch(m, top_k, num_experts, hidden, inter, shared_inter))
        return layer_kernel_kind(m, top_k, num_experts, hidden, inter, shared_inter) == 2 ? Q4K_PATH_PERSISTENT_WIDE
                                                                              : Q4K_PATH_PERSISTENT;
    return Q4K_PATH_TWO_LAUNCH;
}

size_t q4k_moe_layer_half_workspace_size(int m, int top_k, int k_routed, int shared_inter, int k_shared) {
    if (m < 0 || top_k < 1 || top_k > Q4K_MAX_TOP_K || k_routed < 1 || shared_inter < 0) return 0;
    return tc_half_scratch(m, top_k, k_routed, shared_inter, k_shared);
}

size_t q4k_moe_layer_host_staging_size(int m, int top_k, int hidden) {
    if (m < 0 || top_k < 1 || hidden < 1) return 0;
    return align_up((size_t)m * hidden * 4) * 3 + align_up((size_t)m * top_k * 4) * 2 + align_up((size_t)m * 4);
}

int q4k_moe_bucket(const int32_t* d_ids, int n_pairs, int num_experts, int32_t* d_counts, int32_t* d_offsets,
                   int32_t* d_perm, int* d_err_flag, cudaStream_t stream) {
    if (n_pairs < 0) return fail(Q4K_ERR_SHAPE, "n_pairs must be >= 0 (got %d)", n_pairs);
    if (num_experts < 1) return fail(Q4K_ERR_SHAPE, "num_experts must be >= 1 (got %d)", num_experts);
    if (num_experts > kMaxExperts) return fail(Q4K_ERR_LIMIT, "num_experts must be <= %d", kMaxExperts);
    if (!d_counts || !d_offsets || (n_pairs > 0 && (!d_ids || !d_perm))) return fail(Q4K_ERR_NULL, "NULL pointer argument");
    return cuda_status(launch_bucket(d_ids, n_pairs, num_experts, d_counts, d_offsets, d_perm, d_err_flag, stream),
                       "bucket launch");
}

int q4k_moe_id_gemv(const void* d_w_stacked, uint64_t w_byte_offset, int num_experts, const float* d_a,
                    int64_t src1_outer_stride, int64_t src1_inner_stride, const int32_t* d_ids, int m, int top_k,
                    int n, int k, float* d_out, void* d_workspace, size_t ws_bytes, int* d_err_flag,
                    cudaStream_t stream) {
    int st = check_gemv_shape(num_experts, m, top_k, n, k);
    if (st) return st;
    if (!d_w_stacked || !d_a || !d_ids || !d_out) return fail(Q4K_ERR_NULL, "NULL pointer argument");
    const uint8_t* w = static_cast<const uint8_t*>(d_w_stacked) + w_byte_offset;
    if (!aligned16(w)) return fail(Q4K_ERR_ALIGN, "weights (base + byte offset) must be 16-byte aligned");
    if (!aligned16(d_a) || src1_outer_stride % 4 || src1_inner_stride % 4 || src1_outer_stride < 0 ||
        src1_inner_stride < 0)
        return fail(Q4K_ERR_ALIGN, "activations must be 16-byte aligned with non-negative strides that are multiples of 4 floats");
    if (m == 0) return Q4K_OK;
    GemvGroup g{w, nullptr, d_ids, d_a, src1_outer_stride, src1_inner_stride, d_out, num_experts, m, top_k, n, k};
    // the workspace is optional: with room for the activation images, large buckets take
    // the tensor-core path
    int tc = 0;
    uint8_t* img[1] = {static_cast<uint8_t*>(d_workspace)};
    const size_t need = tc_scratch(m * top_k, k);
    if (d_workspace && need > 0 && ws_bytes >= need && (reinterpret_cast<uintptr_t>(d_workspace) & 255) == 0 &&
        tc_wanted(m * top_k, num_experts, n, tc_min_for(m * top_k, num_experts, false)))
        tc = tc_min_for(m * top_k, num_experts, false);
    return cuda_status(launch_idgemv(&g, 1, false, false, d_err_flag, stream, tc, img), "id-gemv launch");
}

int q4k_expert_ffn_forward(const void* d_w_gate, const void* d_w_up, const void* d_w_down, int num_experts,
                           const float* d_h_post, const int32_t* d_ids, int m, int top_k, int hidden, int inter,
                           float* d_expert_out, void* d_workspace, size_t ws_bytes, int* d_err_flag,
                           cudaStream_t stream) {
    int st = check_gemv_shape(num_experts, m, top_k, inter, hidden);
    if (!st) st = check_gemv_shape(num_experts, m, top_k, hidden, inter);
    if (st) return st;
    if (!d_w_gate || !d_w_up || !d_w_down || !d_h_post || !d_ids || !d_expert_out)
        return fail(Q4K_ERR_NULL, "NULL pointer argument");
    if (!aligned16(d_w_gate) || !aligned16(d_w_up) || !aligned16(d_w_down) || !aligned16(d_h_post))
        return fail(Q4K_ERR_ALIGN, "slabs and h_post must be 16-byte aligned");
    st = check_workspace(d_workspace, ws_bytes, ffn_scratch(m, top_k, hidden, inter));
    if (st) return st;
    if (m == 0) return Q4K_OK;
    float* act = static_cast<float*>(d_workspace);
    uint8_t* tc_gu = static_cast<uint8_t*>(d_workspace) + align_up((size_t)m * top_k * inter * sizeof(float));
    uint8_t* tc_dn = tc_gu + tc_scratch(m * top_k, hidden);
    return run_ffn(d_w_gate, d_w_up, d_w_down, num_experts, d_h_post, d_ids, m, top_k, hidden, inter, act,
                   d_expert_out, nullptr, nullptr, nullptr, 0, nullptr, nullptr, d_err_flag, stream, tc_gu, tc_dn);
}

int moe_combine_residual(const float* d_h_mid, const float* d_expert_out, const float* d_weights,
                         const float* d_shared_out, const float* d_shared_gate, int shared_mode, int m, int top_k,
                         int hidden, float* d_hidden_out, cudaStream_t stream) {
    if (m < 0) return fail(Q4K_ERR_SHAPE, "m must be >= 0 (got %d)", m);
    if (top_k < 1 || top_k > Q4K_MAX_TOP_K) return fail(Q4K_ERR_TOPK, "top_k must be in [1, %d] (got %d)", Q4K_MAX_TOP_K, top_k);
    if (hidden < 4 || hidden % 4 != 0) return fail(Q4K_ERR_SHAPE, "hidden must be a positive multiple of 4 (got %d)", hidden);
    if (shared_mode < 0 || shared_mode > 2) return fail(Q4K_ERR_MODE, "shared_mode must be 0, 1 or 2 (got %d)", shared_mode);
    if (!d_h_mid || !d_expert_out || !d_weights || !d_hidden_out) return fail(Q4K_ERR_NULL, "NULL pointer argument");
    if (shared_mode != Q4K_SHARED_NONE && !d_shared_out) return fail(Q4K_ERR_NULL, "shared_out is NULL");
    if (shared_mode == Q4K_SHARED_SIGMOID && !d_shared_gate) return fail(Q4K_ERR_NULL, "shared_gate is NULL");
    if (!aligned16(d_h_mid) || !aligned16(d_expert_out) || !aligned16(d_hidden_out) ||
        (d_shared_out && !aligned16(d_shared_out)))
        return fail(Q4K_ERR_ALIGN, "rows must be 16-byte aligned");
    if (m == 0) return Q4K_OK;
    return cuda_status(launch_combine(d_h_mid, d_expert_out, d_weights, d_shared_out, d_shared_gate, shared_mode, m,
                                      top_k, hidden, d_hidden_out, false, stream),
                       "combine launch");
}

int q4k_moe_layer_forward(const void* d_w_gate, const void* d_w_up, const void* d_w_down, int num_experts,
                          const void* d_ws_gate, const void* d_ws_up, const void* d_ws_down, int shared_inter,
                          int shared_mode, const float* d_h_post, const float* d_h_mid, const int32_t* d_ids,
                          const float* d_weights, const float* d_shared_gate, int m, int top_k, int hidden,
                          int inter, float* d_y, void* d_workspace, size_t ws_bytes, int* d_err_flag,
                          cudaStream_t stream) {
    int st = check_gemv_shape(num_experts, m, top_k, inter, hidden);
    if (!st) st = check_gemv_shape(num_experts, m, top_k, hidden, inter);
    if (st) return st;
    if (shared_mode < 0 || shared_mode > 2) return fail(Q4K_ERR_MODE, "shared_mode must be 0, 1 or 2 (got %d)", shared_mode);
    if (shared_mode == Q4K_SHARED_NONE) {
        shared_inter = 0;
    } else {
        if (shared_inter < 1) return fail(Q4K_ERR_SHAPE, "shared_inter must be >= 1 with a shared expert");
        st = check_gemv_shape(1, m, 1, shared_inter, hidden);
        if (!st) st = check_gemv_shape(1, m, 1, hidden, shared_inter);
        if (st) return st;
        if (!d_ws_gate || !d_ws_up || !d_ws_down) return fail(Q4K_ERR_NULL, "shared expert slabs are NULL");
        if (!aligned16(d_ws_gate) || !aligned16(d_ws_up) || !aligned16(d_ws_down))
            return fail(Q4K_ERR_ALIGN, "shared slabs must be 16-byte aligned");
        if (shared_mode == Q4K_SHARED_SIGMOID && !d_shared_gate) return fail(Q4K_ERR_NULL, "shared_gate is NULL");
    }
    if (!d_w_gate || !d_w_up || !d_w_down || !d_h_post || !d_h_mid || !d_ids || !d_weights || !d_y)
        return fail(Q4K_ERR_NULL, "NULL pointer argument");
    if (!aligned16(d_w_gate) || !aligned16(d_w_up) || !aligned16(d_w_down) || !aligned16(d_h_post) ||
        !aligned16(d_h_mid) || !aligned16(d_y))
        return fail(Q4K_ERR_ALIGN, "slabs and activation rows must be 16-byte aligned");
    const LayerScratch ls = layer_scratch(m, top_k, hidden, inter, shared_inter);
    st = check_workspace(d_workspace, ws_bytes, ls.total);
    if (st) return st;
    if (m == 0) return Q4K_OK;
    uint8_t* ws = static_cast<uint8_t*>(d_workspace);
    float* act = reinterpret_cast<float*>(ws + ls.act);
    float* act_shared = reinterpret_cast<float*>(ws + ls.act_shared);
    float* eout = reinterpret_cast<float*>(ws + ls.eout);
    float* sout = reinterpret_cast<float*>(ws + ls.shared_out);
    // a few pairs and no tensor-core bucket: the whole layer in one persistent launch
    if (layer_single_launch(m, top_k, num_experts, hidden, inter, shared_inter)) {
        GemvGroup gu[2] = {}, dn[2] = {};
        const int ng = gate_up_groups(d_w_gate, d_w_up, num_experts, d_h_post, d_ids, m, top_k, hidden, inter, act,
                                      d_ws_gate, d_ws_up, shared_inter, act_shared, gu);
        down_groups(d_w_down, num_experts, act, d_ids, m, top_k, hidden, inter, eout, d_ws_down, shared_inter,
                    act_shared, sout, dn);
        const CombineSpec cb1{d_y, d_h_mid, d_weights, d_shared_gate, shared_mode, nullptr, 0};
        const cudaError_t e = launch_layer_persistent(gu, dn, ng, cb1, reinterpret_cast<uint64_t*>(ws + ls.sync),
                                                      ls.n_sync_words, d_err_flag, stream);
        if (e != cudaErrorNotSupported) return cuda_status(e, "layer launch");
    }
    // two launches: gate|up + SwiGLU (routed and shared; it also zeroes the combine counters),
    // then down (routed and shared) with the combine fused into its last CTA per row tile; for
    // more than kFusedCombineMaxM tokens the combine is a third launch
    const bool fuse = m <= kFusedCombineMaxM;
    unsigned* counters = reinterpret_cast<unsigned*>(ws + ls.counters);
    st = run_gate_up(d_w_gate, d_w_up, num_experts, d_h_post, d_ids, m, top_k, hidden, inter, act, d_ws_gate, d_ws_up,
                     shared_inter, act_shared, d_err_flag, stream, ws + ls.tc_gu, fuse ? counters : nullptr,
                     fuse ? ls.n_counters : 0);
    if (st) return st;
    CombineSpec cb{d_y, d_h_mid, d_weights, d_shared_gate, shared_mode, counters, ls.n_counters};
    st = run_down(d_w_down, num_experts, act, d_ids, m, top_k, hidden, inter, eout, d_ws_down, shared_inter,
                  act_shared, sout, d_err_flag, stream, ws + ls.tc_dn, fuse ? &cb : nullptr, ws + ls.pre,
                  ws + ls.pre_shared);
    if (st || fuse) return st;
    return cuda_status(launch_combine(d_h_mid, eout, d_weights, shared_mode != Q4K_SHARED_NONE ? sout : nullptr,
                                      d_shared_gate, shared_mode, m, top_k, hidden, d_y, !take_after_join(), stream,
                                      d_ids, num_experts),
                       "combine launch");
}

size_t q4k_moe_layer_routed_workspace_size(int m, int top_k, int num_experts, int hidden, int inter,
                                           int shared_inter) {
    const size_t base = q4k_moe_layer_workspace_size(m, top_k, num_experts, hidden, inter, shared_inter);
    if (base == 0 || num_experts < 1 || num_experts > kMaxExperts || hidden < 1) return 0;
    return route_scratch(align_up(base), m, top_k, num_experts, hidden).total;
}

int q4k_moe_layer_forward_routed(const void* d_w_gate, const void* d_w_up, const void* d_w_down, int num_experts,
                                 const void* d_ws_gate, const void* d_ws_up, const void* d_ws_down, int shared_inter,
                                 int shared_mode, const float* d_h_post, const float* d_h_mid,
                                 const uint16_t* d_w_router, const float* d_bias, const uint16_t* d_w_shared_gate,
                                 int scoring, int normalize, float scale, int n_group, int topk_group, int m,
                                 int top_k, int hidden, int inter, float* d_y, const uint16_t* d_w_norm, float eps,
                                 float* d_normed, int32_t* d_ids_out, float* d_weights_out, void* d_workspace,
                                 size_t ws_bytes, int* d_err_flag, cudaStream_t stream) {
    int st = check_router_args(m, num_experts, hidden, top_k, scoring, n_group, topk_group);
    if (st) return st;
    st = check_gemv_shape(num_experts, m, top_k, inter, hidden);
    if (!st) st = check_gemv_shape(num_experts, m, top_k, hidden, inter);
    if (st) return st;
    if (shared_mode < 0 || shared_mode > 2) return fail(Q4K_ERR_MODE, "shared_mode must be 0, 1 or 2 (got %d)", shared_mode);
    if (shared_mode == Q4K_SHARED_NONE) shared_inter = 0;
    else if (shared_inter < 1) return fail(Q4K_ERR_SHAPE, "shared_inter must be >= 1 with a shared expert");
    if (!d_w_router) return fail(Q4K_ERR_NULL, "w_router is NULL");
    if (shared_mode == Q4K_SHARED_SIGMOID && !d_w_shared_gate)
        return fail(Q4K_ERR_NULL, "a sigmoid-gated shared expert needs w_shared_gate");
    if (d_w_norm && !d_normed) return fail(Q4K_ERR_NULL, "w_norm given without normed");
    if ((d_ids_out == nullptr) != (d_weights_out == nullptr))
        return fail(Q4K_ERR_NULL, "ids_out and weights_out are given together or not at all");
    if (!aligned16(d_w_router) || (d_w_shared_gate && !aligned16(d_w_shared_gate)) ||
        (d_normed && !aligned16(d_normed)) || (d_w_norm && (reinterpret_cast<uintptr_t>(d_w_norm) & 7u)))
        return fail(Q4K_ERR_ALIGN, "w_router, w_shared_gate and normed must be 16-byte aligned, w_norm 8-byte");
    const size_t base = align_up(q4k_moe_layer_workspace_size(m, top_k, num_experts, hidden, inter, shared_inter));
    const RouteScratch rs = route_scratch(base, m, top_k, num_experts, hidden);
    st = check_workspace(d_workspace, ws_bytes, rs.total);
    if (st) return st;
    if (m == 0) return Q4K_OK;
    uint8_t* ws = static_cast<uint8_t*>(d_workspace);
    int32_t* ids = d_ids_out ? d_ids_out : reinterpret_cast<int32_t*>(ws + rs.ids);
    float* wts = d_weights_out ? d_weights_out : reinterpret_cast<float*>(ws + rs.weights);
    float* logits = reinterpret_cast<float*>(ws + rs.logits);
    float* sg = reinterpret_cast<float*>(ws + rs.sg);
    const uint16_t* wsg = shared_mode == Q4K_SHARED_NONE ? nullptr : d_w_shared_gate;
    // the router's two launches, the layer, the norm: each a programmatic dependent of the one
    // before where that is safe (measured faster than choosing in every CTA of the layer)
    st = q4k_moe_router(d_h_post, d_w_router, d_bias, wsg, m, num_experts, hidden, top_k, scoring, normalize, scale,
                        n_group, topk_group, ids, wts, logits, wsg ? sg : nullptr, stream);
    if (st) return st;
    st = q4k_moe_layer_forward(d_w_gate, d_w_up, d_w_down, num_experts, d_ws_gate, d_ws_up, d_ws_down, shared_inter,
                               shared_mode, d_h_post, d_h_mid, ids, wts, wsg ? sg : nullptr, m, top_k, hidden, inter,
                               d_y, d_workspace, base, d_err_flag, stream);
    if (st || !d_w_norm) return st;
    return q4k_rms_norm(d_y, d_w_norm, m, hidden, eps, d_normed, stream);
}

int q4k_moe_layer_gate_up(const void* d_w_gate, const void* d_w_up, int num_experts, const void* d_ws_gate,
                          const void* d_ws_up, int shared_inter, const float* d_h_post, const int32_t* d_ids, int m,
                          int top_k, int hidden, int inter, float* d_act, float* d_act_shared, void* d_workspace,
                          size_t ws_bytes, int* d_err_flag, cudaStream_t stream) {
    if (!d_w_up) return fail(Q4K_ERR_NULL, "NULL up slab");
    if (shared_inter > 0 && !d_ws_up) return fail(Q4K_ERR_NULL, "NULL shared up slab");
    int st = check_layer(d_w_gate, d_w_up, num_experts, shared_inter, d_ws_gate, d_ws_up, m, top_k, hidden, inter);
    if (st) return st;
    if (!d_h_post || !d_ids || !d_act || (shared_inter > 0 && !d_act_shared)) return fail(Q4K_ERR_NULL, "NULL pointer argument");
    if (!aligned16(d_h_post)) return fail(Q4K_ERR_ALIGN, "h_post must be 16-byte aligned");
    if (m == 0) return Q4K_OK;
    const size_t need = tc_half_scratch(m, top_k, hidden, shared_inter, hidden);
    uint8_t* tc_ws = (d_workspace && ws_bytes >= need && (reinterpret_cast<uintptr_t>(d_workspace) & 255) == 0)
                         ? static_cast<uint8_t*>(d_workspace) : nullptr;
    return run_gate_up(d_w_gate, d_w_up, num_experts, d_h_post, d_ids, m, top_k, hidden, inter, d_act, d_ws_gate,
                       d_ws_up, shared_inter, d_act_shared, d_err_flag, stream, tc_ws);
}

int q4k_moe_layer_down(const void* d_w_down, int num_experts, const void* d_ws_down, int shared_inter,
                       const float* d_act, const float* d_act_shared, const int32_t* d_ids, int m, int top_k,
                       int hidden, int inter, float* d_expert_out, float* d_shared_out, void* d_workspace,
                       size_t ws_bytes, int* d_err_flag, cudaStream_t stream) {
    int st = check_layer(d_w_down, nullptr, num_experts, shared_inter, d_ws_down, nullptr, m, top_k, hidden, inter);
    if (st) return st;
    if (!d_act || !d_ids || !d_expert_out || (shared_inter > 0 && (!d_act_shared || !d_shared_out)))
        return fail(Q4K_ERR_NULL, "NULL pointer argument");
    if (!aligned16(d_act) || (d_act_shared && !aligned16(d_act_shared)))
        return fail(Q4K_ERR_ALIGN, "act rows must be 16-byte aligned");
    if (m == 0) return Q4K_OK;
    const size_t need = tc_half_scratch(m, top_k, inter, shared_inter, shared_inter);
    uint8_t* tc_ws = (d_workspace && ws_bytes >= need && (reinterpret_cast<uintptr_t>(d_workspace) & 255) == 0)
                         ? static_cast<uint8_t*>(d_workspace) : nullptr;
    return run_down(d_w_down, num_experts, d_act, d_ids, m, top_k, hidden, inter, d_expert_out, d_ws_down,
                    shared_inter, d_act_shared, d_shared_out, d_err_flag, stream, tc_ws);
}

int q4k_moe_layer_forward_host(const void* d_w_gate, const void* d_w_up, const void* d_w_down, int num_experts,
                               const void* d_ws_gate, const void* d_ws_up, const void* d_ws_down, int shared_inter,
                               int shared_mode, const float* h_post, const float* h_mid, const int32_t* ids,
                               const float* weights, const float* shared_gate, int m, int top_k, int hidden,
                               int inter, float* y, void* d_workspace, size_t ws_bytes, int* d_err_flag,
                               cudaStream_t stream) {
    int st = check_gemv_shape(num_experts, m, top_k, inter, hidden);
    if (st) return st;
    if (!h_post || !h_mid || !ids || !weights || !y) return fail(Q4K_ERR_NULL, "NULL host pointer argument");
    if (shared_mode == Q4K_SHARED_SIGMOID && !shared_gate) return fail(Q4K_ERR_NULL, "shared_gate is NULL");
    const int sh = shared_mode == Q4K_SHARED_NONE ? 0 : shared_inter;
    const size_t layer_bytes = layer_scratch(m, top_k, hidden, inter, sh).total;
    const size_t stage_bytes = q4k_moe_layer_host_staging_size(m, top_k, hidden);
    st = check_workspace(d_workspace, ws_bytes, layer_bytes + stage_bytes);
    if (st) return st;
    if (m == 0) return Q4K_OK;
    uint8_t* ws = static_cast<uint8_t*>(d_workspace);
    uint8_t* stage = ws + layer_bytes;
    const size_t mh = (size_t)m * hidden * 4, mt = (size_t)m * top_k * 4;
    float* dh_post = reinterpret_cast<float*>(stage);
    float* dh_mid = reinterpret_cast<float*>(stage + align_up(mh));
    float* dy = reinterpret_cast<float*>(stage + 2 * align_up(mh));
    int32_t* dids = reinterpret_cast<int32_t*>(stage + 3 * align_up(mh));
    float* dw = reinterpret_cast<float*>(stage + 3 * align_up(mh) + align_up(mt));
    float* dgate = reinterpret_cast<float*>(stage + 3 * align_up(mh) + 2 * align_up(mt));
    // Page-locked host buffers have a device view: the inputs are then gathered by one kernel
    // reading host memory, and the combine writes y into host memory. Any other host memory
    // goes through the copy engine (one transfer per buffer).
    const void* src[5] = {h_post, h_mid, ids, weights, shared_gate};
    void* dst[5] = {dh_post, dh_mid, dids, dw, dgate};
    const size_t bytes[5] = {mh, mh, mt, mt, shared_gate ? (size_t)m * 4 : 0};
    const void* view[5] = {};
    bool mapped = true;
    for (int i = 0; i < 5 && mapped; ++i) mapped = bytes[i] == 0 || host_device_view(src[i], &view[i]);
    cudaError_t e = cudaSuccess;
    if (mapped && mh <= 0xFFFFFFFFu) {
        GatherSpec g{};
        for (int i = 0; i < 5; ++i)
            if (bytes[i]) {
                g.src[g.n] = view[i];
                g.dst[g.n] = dst[i];
                g.bytes[g.n] = (uint32_t)bytes[i];
                ++g.n;
            }
        e = launch_gather(g, stream);
    } else {
        for (int i = 0; i < 5 && e == cudaSuccess; ++i)
            if (bytes[i]) e = cudaMemcpyAsync(dst[i], src[i], bytes[i], cudaMemcpyHostToDevice, stream);
    }
    if (e != cudaSuccess) return cuda_status(e, "host-to-device copy");
    const void* y_view = nullptr;
    const bool y_mapped = host_device_view(y, &y_view);
    float* y_dev = y_mapped ? static_cast<float*>(const_cast<void*>(y_view)) : dy;
    st = q4k_moe_layer_forward(d_w_gate, d_w_up, d_w_down, num_experts, d_ws_gate, d_ws_up, d_ws_down, sh,
                               shared_mode, dh_post, dh_mid, dids, dw, shared_gate ? dgate : nullptr, m, top_k,
                               hidden, inter, y_dev, d_workspace, layer_bytes, d_err_flag, stream);
    if (st || y_mapped) return st;
    return cuda_status(cudaMemcpyAsync(y, dy, mh, cudaMemcpyDeviceToHost, stream), "device-to-host copy");
}

int q4k_moe_id_gemv_fmt(int fmt, const void* d_w, const void* d_w2, uint64_t w_byte_offset, uint64_t expert_stride,
                        uint64_t scales_offset, uint64_t biases_offset, int group_size, int num_experts,
                        const float* d_a, int64_t src1_outer_stride, int64_t src1_inner_stride, const int32_t* d_ids,
                        int m, int top_k, int n, int k, float* d_out, int* d_err_flag, cudaStream_t stream) {
    if (fmt != Q4K_FMT_AFFINE4 && fmt != Q4K_FMT_Q4TP)
        return fail(Q4K_ERR_MODE, "fmt must be Q4K_FMT_AFFINE4 or Q4K_FMT_Q4TP (got %d)", fmt);
    int st = check_gemv_shape(num_experts, m, top_k, n, k);
    if (st != Q4K_OK) return st;
    if (fmt == Q4K_FMT_AFFINE4) {
        if (group_size != 32 && group_size != 64 && group_size != 128)
            return fail(Q4K_ERR_SHAPE, "group_size must be 32, 64 or 128 (got %d)", group_size);
        if (scales_offset % 4 != 0 || biases_offset % 4 != 0)
            return fail(Q4K_ERR_ALIGN, "scales and biases offsets must be multiples of 4");
    }
    const uint64_t mat = fmt == Q4K_FMT_AFFINE4
                             ? (uint64_t)n * (k / 2)
                             : (uint64_t)n * (k / 2) + 4ull * n + (uint64_t)n * ((k / 32) * 5 / 8);
    if (expert_stride % 16 != 0 || (num_experts > 1 && expert_stride < mat))
        return fail(Q4K_ERR_SHAPE, "expert_stride must be a multiple of 16 holding the codes (%llu bytes)",
                    (unsigned long long)mat);
    if (m == 0) return Q4K_OK;
    if (!d_w || !d_a || !d_ids || !d_out) return fail(Q4K_ERR_NULL, "w, a, ids and out are required");
    const uint8_t* w = static_cast<const uint8_t*>(d_w) + w_byte_offset;
    const uint8_t* w2 = d_w2 ? static_cast<const uint8_t*>(d_w2) + w_byte_offset : nullptr;
    if (!aligned16(w) || (w2 && !aligned16(w2))) return fail(Q4K_ERR_ALIGN, "slabs (+ offset) must be 16-byte aligned");
    if (!aligned16(d_a) || src1_outer_stride % 4 != 0 || src1_inner_stride % 4 != 0)
        return fail(Q4K_ERR_ALIGN, "activation rows must be 16-byte aligned");
    return cuda_status(launch_fmt4(fmt, w, w2, expert_stride, scales_offset, biases_offset, group_size, num_experts,
                                   d_a, src1_outer_stride, src1_inner_stride, d_ids, m, top_k, n, k, d_out,
                                   d_err_flag, stream),
                       "fmt4 id-GEMV launch");
}

int q4k_moe_router(const float* d_x, const uint16_t* d_w_router, const float* d_bias, const uint16_t* d_w_shared_gate,
                   int m, int num_experts, int hidden, int top_k, int scoring, int normalize, float scale, int n_group,
                   int topk_group, int32_t* d_ids, float* d_weights, float* d_logits, float* d_shared_gate,
                   cudaStream_t stream) {
    const int rst = check_router_args(m, num_experts, hidden, top_k, scoring, n_group, topk_group);
    if (rst != Q4K_OK) return rst;
    if (m == 0) return Q4K_OK;
    if (!d_x || !d_w_router || !d_ids || !d_weights || !d_logits)
        return fail(Q4K_ERR_NULL, "x, w_router, ids, weights and logits are required");
    if (d_w_shared_gate && !d_shared_gate) return fail(Q4K_ERR_NULL, "w_shared_gate given without shared_gate");
    if (!aligned16(d_x) || !aligned16(d_w_router) || (d_w_shared_gate && !aligned16(d_w_shared_gate)))
        return fail(Q4K_ERR_ALIGN, "x, w_router and w_shared_gate must be 16-byte aligned");
    return cuda_status(launch_router(d_x, d_w_router, d_bias, d_w_shared_gate, m, num_experts, hidden, top_k, scoring,
                                     normalize ? 1 : 0, scale, n_group, topk_group, d_ids, d_weights, d_logits,
                                     d_shared_gate, stream),
                       "router launch");
}

int q4k_rms_norm(const float* d_x, const uint16_t* d_w, int m, int hidden, float eps, float* d_out, cudaStream_t stream) {
    if (m < 0) return fail(Q4K_ERR_SHAPE, "m must be >= 0 (got %d)", m);
    if (hidden < 4 || hidden % 4 != 0) return fail(Q4K_ERR_SHAPE, "hidden must be a positive multiple of 4 (got %d)", hidden);
    if (m == 0) return Q4K_OK;
    if (!d_x || !d_w || !d_out) return fail(Q4K_ERR_NULL, "x, w and out are required");
    if (!aligned16(d_x) || !aligned16(d_out) || (reinterpret_cast<uintptr_t>(d_w) & 7u))
        return fail(Q4K_ERR_ALIGN, "x and out must be 16-byte aligned, w 8-byte aligned");
    return cuda_status(launch_rms_norm(d_x, d_w, m, hidden, eps, d_out, stream), "rms_norm launch");
}

int q4k_quantize_rows(const float* d_x, int64_t rows, int k, void* d_out, cudaStream_t stream) {
    if (rows < 0) return fail(Q4K_ERR_SHAPE, "rows must be >= 0");
    if (k < 1 || k % kQK != 0) return fail(Q4K_ERR_SHAPE, "k must be a positive multiple of 256 (got %d)", k);
    if (rows > 0 && (!d_x || !d_out)) return fail(Q4K_ERR_NULL, "NULL pointer argument");
    if (!aligned16(d_x) || !aligned16(d_out)) return fail(Q4K_ERR_ALIGN, "x and out must be 16-byte aligned");
    if (rows == 0) return Q4K_OK;
    return cuda_status(launch_quantize(d_x, rows, k, static_cast<uint8_t*>(d_out), stream), "quantize launch");
}

int q4k_stream_ceiling_sink_words(void) { return stream_ceiling_grid(); }

int q4k_stream_ceiling(const void* d_src, uint64_t bytes, uint32_t* d_sink, cudaStream_t stream) {
    if (!d_src || !d_sink) return fail(Q4K_ERR_NULL, "NULL pointer argument");
    if (!aligned16(d_src) || bytes % 16) return fail(Q4K_ERR_ALIGN, "source must be 16-byte aligned, bytes % 16 == 0");
    return cuda_status(launch_stream_ceiling(d_src, bytes, d_sink, stream), "ceiling launch");
}

}  // extern "C"

// q4k_gemv.cu -- the bucketed Q4_K MoE id-GEMV (and its fused gate|up + SwiGLU form).
//
// What it computes (ferrum-kernels q4_k_moe_id_gemv_batched.rs,
// `dispatch_gemv_q4k_moe_id_batched_on_encoder`): for every (token, slot) pair p,
//   out[p, r] = sum_c W_{ids[p]}[r, c] * a[t*outer + s*inner + c],  t = p / top_k, s = p % top_k.
// With a second slab (moeflux expert_forward.rs: gate, up, SwiGLU) the launch computes
//   out[p, r] = silu(Wg . x) * (Wu . x).
//
// How (GB300 design):
//  * Pairs are bucketed by expert inside every CTA (histogram + scan of the ids in shared
//    memory), so each touched slab row tile is streamed from HBM once per launch no matter
//    how many pairs of the batch picked that expert. Work item = (group, expert, row tile,
//    chunk of <= kTB tokens of that expert's bucket), row tiles of one chunk consecutive;
//    each CTA takes a contiguous range of items, so its staged rows carry over, and CTAs on
//    other chunks of the same expert read the same tiles at about the same time (L2 hits).
//  * The item's activation rows are staged in shared memory as 16-bit fixed point per
//    32-element sub-block: X = rint(x / delta), delta = max|x| / 32767, split into a low
//    byte plane (unsigned) and a high byte plane (signed), with sum(X) per sub-block.
//  * Weights are read with coalesced 16-byte loads; a lane owns one 64-weight group (32
//    code bytes = sub-blocks 2c and 2c+1) of one block of one row. The codes are used as
//    bytes directly (w & 0x0F0F0F0F, (w >> 4) & 0x0F0F0F0F) by dp4a against the two
//    activation planes, so the integer sum S_j = sum_i q_i X_i of a sub-block is exact.
//  * Per sub-block the Q4_K algebra folds the minimum into the activation sum:
//      sum_i w_i x_i = delta_j * (d*sc_j * S_j - dmin*m_j * sum_i X_i).
//  * Lanes sharing a row reduce with warp shuffles; the epilogue writes the pair's row
//    (optionally silu(g) * u).
#include <algorithm>
#include <cstdlib>

#include "q4k_gemv_common.cuh"

namespace q4k {

struct GemvParams {
    GroupDev g[kMaxGroups];
    int n_groups;
    int tb;                 // tokens per work item (<= kTB)
    int hist_off[kMaxGroups];  // int offsets of each group's tables in shared memory
    int x_off;              // byte offset of the staged activations
    int meta_off;           // byte offset of the per-sub-block (delta, sumX) pairs
    int kmax;               // largest k of the groups (sizes the staging area)
    int tc_min;             // > 0: experts with at least this many pairs are left to the tensor-core path
    int* err_flag;
    int has_combine;        // fuse the combine (group 0 routed, group 1 shared) into this launch
    CombineSpec cb;
    unsigned* zero;         // CTA 0 zeroes zero[0..n_zero) first
    int n_zero;
    int fast;               // every group has at most 32 pairs: bucket with one warp per group
    int wait_first;         // wait for the previous kernel before reading anything (first launch of a layer)
    const uint8_t* pre_planes[kMaxGroups];  // group's rows already staged by prestage_kernel (or null)
    const float2* pre_meta[kMaxGroups];
};

// Copy `bytes` (a multiple of 16, both ends 16-byte aligned) from global into shared memory
// with the block's threads by asynchronous copies: no registers held while the item's weight
// ring is live. The caller waits (cp.async.wait_group) and synchronises the block.
__device__ __forceinline__ void copy_block16(const uint8_t* src, uint8_t* dst, int64_t bytes) {
    const int64_t n = bytes / 16;
    for (int64_t i = threadIdx.x; i < n; i += kThreads)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst + 16 * i)), "l"(src + 16 * i)
                     : "memory");
}

// The item's rows as prestage_kernel left them (pair p's planes at planes + p * (k/64) * 144,
// its (delta, sum X) pairs at meta + p * (k/32)): copied, not quantized again.
__device__ __forceinline__ void copy_staged(const uint8_t* planes, const float2* metas, int k, const int* pairs,
                                            int nt, uint8_t* xs, float2* meta) {
    const int64_t pb = (int64_t)(k / 64) * kPairBytes;
    const int nsb = k / 32;
    for (int t = 0; t < nt; ++t) {
        const int p = pairs[t];
        copy_block16(planes + (int64_t)p * pb, xs + t * pb, pb);
        copy_block16(reinterpret_cast<const uint8_t*>(metas + (int64_t)p * nsb),
                     reinterpret_cast<uint8_t*>(meta + (int64_t)t * nsb), (int64_t)nsb * 8);
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Combine of rows [r0, r1) of every token, run by the last CTA of a row tile.
__device__ void combine_rows(const GemvParams& P, int r0, int r1) {
    const GroupDev& R = P.g[0];
    const bool shared = P.cb.shared_mode != Q4K_SHARED_NONE && P.n_groups > 1;
    combine_span(P.cb, R.out, R.ids, R.num_experts, R.n_pairs, R.top_k, R.n, shared ? P.g[1].out : nullptr, r0, r1,
                 threadIdx.x, blockDim.x);
}

template <bool FUSED, int TB>
__global__ void __launch_bounds__(kThreads, FUSED ? 3 : 4)
idgemv_kernel(const __grid_constant__ GemvParams P) {
    extern __shared__ __align__(16) uint8_t smem[];
    int* s_int = reinterpret_cast<int*>(smem);
    __shared__ int s_warp[33];
    __shared__ int s_bad[kMaxGroups];
    __shared__ int s_items[kMaxGroups + 1];
    __shared__ int s_pairs[kTB];
    __shared__ int s_item_info[5];  // group, expert, tile, tokens, chunk
    __shared__ int64_t s_rows[kTB];  // activation row offsets currently staged
    __shared__ int s_staged_group, s_staged_nt, s_restage;
    __shared__ int s_pairs_key[3];  // (group, expert, chunk) whose pairs are in s_pairs

    // the next launch (down, which reads the ids before its own wait) may start only once the
    // ids are complete: with wait_first, trigger it after the wait
    if (P.wait_first) pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0) { s_staged_group = -1; s_staged_nt = 0; }
    if (P.zero && blockIdx.x == 0)
        for (int i = threadIdx.x; i < P.n_zero; i += kThreads) P.zero[i] = 0u;
    __shared__ int s_last;

    __shared__ FastGroup s_fast[kMaxGroups];
    // ---- bucketing prologue (ids are inputs of the layer, not results of the previous kernel)
    if (threadIdx.x == 0) s_items[0] = 0;
    if (P.fast) {
        if (warp_id_of_thread() < P.n_groups) {
            const int gi = warp_id_of_thread();
            const GroupDev& G = P.g[gi];
            fast_bucket(G.ids, G.n_pairs, G.num_experts, G.tiles, TB, P.tc_min, s_fast[gi], &s_bad[gi]);
        }
        __syncthreads();
        if (threadIdx.x == 0)
            for (int gi = 0; gi < P.n_groups; ++gi) s_items[gi + 1] = s_items[gi] + s_fast[gi].start[s_fast[gi].U];
        __syncthreads();
    }
    for (int gi = 0; gi < P.n_groups && !P.fast; ++gi) {
        const GroupDev& G = P.g[gi];
        int* cnt = s_int + P.hist_off[gi];
        int* start = cnt + G.num_experts;
        if (G.ids) {
            block_histogram(G.ids, G.n_pairs, G.num_experts, cnt, &s_bad[gi]);
        } else {
            if (threadIdx.x == 0) { cnt[0] = G.n_pairs; s_bad[gi] = 0; }
            __syncthreads();
        }
        for (int e = threadIdx.x; e < G.num_experts; e += kThreads)
            start[e] = (P.tc_min > 0 && cnt[e] >= P.tc_min) ? 0 : ((cnt[e] + TB - 1) / TB) * G.tiles;
        __syncthreads();
        const int total = block_exclusive_scan(start, G.num_experts, s_warp);
        if (threadIdx.x == 0) s_items[gi + 1] = s_items[gi] + total;
        __syncthreads();
    }
    const int total_items = s_items[P.n_groups];
    uint8_t* xs = smem + P.x_off;
    float2* meta = reinterpret_cast<float2*>(smem + P.meta_off);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // each CTA takes a contiguous range of items: consecutive row tiles of one expert and
    // chunk, so the staged activation rows and the bucket's pair list carry over
    const int per_cta = (total_items + gridDim.x - 1) / gridDim.x;
    const int item_begin = blockIdx.x * per_cta;
    const int item_end = min(total_items, item_begin + per_cta);
    if (threadIdx.x == 0) { s_pairs_key[0] = -1; }
    for (int item = item_begin; item < item_end; ++item) {
        // ---- locate the item: group, expert (search over the item offsets), tile, chunk
        if (P.fast) {
            if (warp == 0) {
                const FastLoc L = fast_locate(s_fast, s_items, P.g, P.n_groups, TB, item, s_pairs);
                const int gi = L.gi, nt = L.nt;
                if (lane == 0) {
                    s_item_info[0] = gi;
                    s_item_info[1] = L.e;
                    s_item_info[2] = L.tile;
                    s_item_info[3] = nt;
                    s_item_info[4] = L.chunk;
                    s_pairs_key[0] = gi; s_pairs_key[1] = L.e; s_pairs_key[2] = L.chunk;
                }
                __syncwarp();
                // the same activation rows as the staged ones need no restaging
                const GroupDev& G = P.g[gi];
                bool same = s_staged_group == gi && s_staged_nt == nt;
                if (lane < nt) {
                    const int p = s_pairs[lane];
                    const int64_t arow = (int64_t)(p / G.top_k) * G.outer + (int64_t)(p % G.top_k) * G.inner;
                    same = same && s_rows[lane] == arow;
                }
                same = __all_sync(0xffffffffu, same);
                if (lane == 0) s_restage = same ? 0 : 1;
            }
        } else if (threadIdx.x == 0) {
            int gi = 0;
            while (gi + 1 < P.n_groups && item >= s_items[gi + 1]) ++gi;
            const GroupDev& G = P.g[gi];
            const int* cnt = s_int + P.hist_off[gi];
            const int* start = cnt + G.num_experts;
            const int local = item - s_items[gi];
            int lo = 0, hi = G.num_experts - 1;  // last e with start[e] <= local (it has items)
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (start[mid] <= local) lo = mid; else hi = mid - 1;
            }
            const int in_e = local - start[lo];
            const int chunk = in_e / G.tiles;  // tiles of one chunk run together (no restaging)
            s_item_info[0] = gi;
            s_item_info[1] = lo;
            s_item_info[2] = in_e % G.tiles;
            s_item_info[3] = min(TB, cnt[lo] - chunk * TB);
            s_item_info[4] = chunk;
        }
        __syncthreads();
        const int gi = s_item_info[0], e = s_item_info[1], tile = s_item_info[2], nt = s_item_info[3];
        const int chunk = s_item_info[4];
        const GroupDev& G = P.g[gi];

        // ---- start the weight stream before staging (independent of the activations)
        ItemLane<FUSED ? kFused : kOne> L;
        item_issue<FUSED ? kFused : kOne>(G, e, tile, lane, warp, L);
        // the next item of this CTA is usually the next row tile of the same slab: start its
        // rows into L2 (copy engine, no registers), so its loads need not wait for HBM
        if (threadIdx.x == 0 && item + 1 < item_end && tile + 1 < G.tiles) {
            const int tr = item_tile_rows(G.lg_split, FUSED ? kFused : kOne);
            const int r1 = (tile + 1) * tr, rows = min(tr, G.n - r1);
            const int64_t off = (int64_t)e * G.nb02 + (int64_t)r1 * G.nb01;
            bulk_prefetch_l2(G.w + off, (uint32_t)(rows * G.nb01));
            if (FUSED) bulk_prefetch_l2(G.w2 + off, (uint32_t)(rows * G.nb01));
        }

        if (!P.fast && warp == 0) {
            const bool have = s_pairs_key[0] == gi && s_pairs_key[1] == e && s_pairs_key[2] == chunk;
            if (!have) {
                if (G.ids) {
                    warp_gather_bucket(G.ids, G.n_pairs, e, chunk * TB, nt, s_pairs);
                } else if (lane < nt) {
                    s_pairs[lane] = chunk * TB + lane;
                }
                __syncwarp();
                if (lane == 0) { s_pairs_key[0] = gi; s_pairs_key[1] = e; s_pairs_key[2] = chunk; }
            }
            __syncwarp();
            // the same activation rows as the staged ones (e.g. every item of a broadcast
            // gate/up walk at m = 1) need no restaging
            bool same = s_staged_group == gi && s_staged_nt == nt;
            if (lane < nt) {
                const int p = s_pairs[lane];
                const int64_t arow = (int64_t)(p / G.top_k) * G.outer + (int64_t)(p % G.top_k) * G.inner;
                same = same && s_rows[lane] == arow;
            }
            same = __all_sync(0xffffffffu, same);
            if (lane == 0) s_restage = same ? 0 : 1;
        }
        if (!P.fast) __syncthreads();
        const bool restage = s_restage != 0;
        if (item == item_begin) pdl_wait();  // the activations may come from the previous kernel
        if (restage) {
            if (warp == 0 && lane < nt) {
                const int p = s_pairs[lane];
                s_rows[lane] = (int64_t)(p / G.top_k) * G.outer + (int64_t)(p % G.top_k) * G.inner;
            }
            if (threadIdx.x == 0) { s_staged_group = gi; s_staged_nt = nt; }
            bool copied = false;
            if constexpr (!FUSED) {  // (down launches only)
                if (P.pre_planes[gi]) {
                    copy_staged(P.pre_planes[gi], P.pre_meta[gi], G.k, s_pairs, nt, xs, meta);
                    copied = true;
                }
            }
            if (!copied) stage_rows(G, s_pairs, nt, xs, meta);
        }
        __syncthreads();

        // ---- main loop over this lane's blocks, kDepth of them in flight; reduce; write
        item_compute<FUSED ? kFused : kOne, TB>(G, L, s_pairs, nt, xs, meta, lane);
        __syncthreads();  // s_pairs / staged rows are rewritten by the next item
        if (P.has_combine) {
            // every item of this row tile, from either group, counts once; the last one combines
            if (threadIdx.x == 0) {
                __threadfence();
                const unsigned expected = (unsigned)(total_items / G.tiles);
                const unsigned prev = atomicAdd(&P.cb.counters[tile], 1u);
                s_last = prev + 1u == expected;
            }
            __syncthreads();
            if (s_last) {
                __threadfence();
                const int tr = G.n > 0 ? kWarps * (8 >> G.lg_split) : 0;
                combine_rows(P, tile * tr, min(G.n, (tile + 1) * tr));
                if (threadIdx.x == 0) P.cb.counters[tile] = 0u;
            }
            __syncthreads();
        }
    }
    // every expert went to the tensor-core path: no item here counts, so combine every tile
    if (P.has_combine && total_items == 0) {
        pdl_wait();
        const GroupDev& G = P.g[0];
        const int tr = kWarps * (8 >> G.lg_split);
        for (int tile = blockIdx.x; tile < G.tiles; tile += gridDim.x) combine_rows(P, tile * tr, min(G.n, (tile + 1) * tr));
    }
    // out-of-range ids: flag and zero their rows (CTA 0, after the previous kernel is done)
    if (blockIdx.x == 0) {
        pdl_wait();
        for (int gi = 0; gi < P.n_groups; ++gi) {
            const GroupDev& G = P.g[gi];
            if (!G.ids || s_bad[gi] == 0) continue;
            if (threadIdx.x == 0) raise_flag(P.err_flag, Q4K_ERR_EXPERT_ID);
            for (int p = 0; p < G.n_pairs; ++p) {
                if (id_valid(G.ids[p], G.num_experts)) continue;
                for (int r = threadIdx.x; r < G.n; r += kThreads) G.out[(int64_t)p * G.n + r] = 0.0f;
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
static int g_num_sms = 0;
constexpr int kMaxDevices = 64;
constexpr size_t kSmemLimit = 200 * 1024;
static bool g_smem_attr_set[4][kMaxDevices] = {};

int num_sms() {
    if (g_num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 1;
    }
    return g_num_sms;
}

int idgemv_tile_rows(int k) { return kWarps * (8 >> lg_split_for(k)); }

cudaError_t launch_idgemv_kernel(const GemvGroup* groups, int n_groups, bool fused_swiglu, bool pdl, int* err_flag,
                                 cudaStream_t stream, int tc_min, const CombineSpec* combine, unsigned* zero,
                                 int n_zero, bool pdl_wait_first, const PreStaged* pre);

// A second stream and two events per device for the calling host thread: the tensor-core
// kernels of a launch run on it beside the id-GEMV kernel (they take disjoint experts and write
// disjoint rows). Created on first use; null when creation failed (the launch then stays on
// one stream).
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    bool tried = false;
};

// Set when a launch has joined its side stream back into the caller's stream: the next launch
// of this host thread is then an ordinary one, so no programmatic overlap has to be trusted to
// respect the join (a launch right after a join may read rows the side stream wrote).
thread_local bool t_after_join = false;

bool take_after_join() {
    const bool v = t_after_join;
    t_after_join = false;
    return v;
}

static SideStream* side_stream(int dev) {
    thread_local SideStream t_side[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    SideStream& s = t_side[dev];
    if (!s.tried) {
        s.tried = true;
        if (cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            s.stream = nullptr;
        }
    }
    return s.stream ? &s : nullptr;
}

cudaError_t launch_idgemv(const GemvGroup* groups, int n_groups, bool fused_swiglu, bool pdl, int* err_flag,
                          cudaStream_t stream, int tc_min, uint8_t* const* tc_img, const CombineSpec* combine,
                          unsigned* zero, int n_zero, bool pdl_wait_first, const PreStaged* pre) {
    if (tc_min > 0 && !tc_fits(groups, n_groups)) tc_min = 0;  // too many experts for its tables
    const bool after_join = take_after_join();
    if (after_join) pdl = false;
    // With the tensor-core path the launch forks: its kernels go to the side stream after an
    // event on `stream` (so they see everything issued before), the id-GEMV kernel stays on
    // `stream`, and `stream` waits for the side stream's event after it. Not with a fused
    // combine, which reads the tensor-core rows: then the tensor-core kernels come first.
    SideStream* side = nullptr;
    if (tc_min > 0 && !combine) {
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) side = side_stream(dev);
    }
    if (tc_min > 0 && side) {
        cudaError_t e = cudaEventRecord(side->fork, stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
        if (e != cudaSuccess) {
            // the side stream or its events are gone (e.g. after a device reset): make new ones
            // next time, and run this launch on one stream
            cudaGetLastError();
            side->tried = false;
            side->stream = nullptr;
            side = nullptr;
        }
    }
    if (tc_min > 0 && side) {
        cudaError_t e = launch_tc(groups, n_groups, fused_swiglu, tc_min, tc_img, err_flag, side->stream);
        if (e == cudaSuccess) e = cudaEventRecord(side->join, side->stream);
        if (e != cudaSuccess) return e;
    } else if (tc_min > 0) {
        cudaError_t e = launch_tc(groups, n_groups, fused_swiglu, tc_min, tc_img, err_flag, stream, !after_join);
        if (e != cudaSuccess) return e;
        pdl = false;  // the tensor-core kernels precede this launch in the stream
    }
    // (the join: the rest of the launch runs through launch_idgemv_kernel, then `stream` waits)
    const cudaError_t ke = launch_idgemv_kernel(groups, n_groups, fused_swiglu, pdl, err_flag, stream, tc_min, combine,
                                                zero, n_zero, pdl_wait_first, pre);
    if (tc_min > 0 && side) {
        const cudaError_t je = cudaStreamWaitEvent(stream, side->join, 0);
        t_after_join = true;
        if (ke == cudaSuccess) return je;
    }
    return ke;
}

// The id-GEMV kernel's launch (after any tensor-core launches of the same call).
cudaError_t launch_idgemv_kernel(const GemvGroup* groups, int n_groups, bool fused_swiglu, bool pdl, int* err_flag,
                                 cudaStream_t stream, int tc_min, const CombineSpec* combine, unsigned* zero,
                                 int n_zero, bool pdl_wait_first, const PreStaged* pre) {
    GemvParams P{};
    P.n_groups = n_groups;
    P.err_flag = err_flag;
    P.tc_min = tc_min;
    P.zero = zero;
    P.n_zero = zero ? n_zero : 0;
    P.wait_first = (pdl && pdl_wait_first) ? 1 : 0;
    for (int gi = 0; pre && gi < n_groups; ++gi) {
        P.pre_planes[gi] = pre->planes[gi];
        P.pre_meta[gi] = pre->meta[gi];
    }
    if (combine) {
        P.has_combine = 1;
        P.cb = *combine;
    }
    // Tokens per work item: 1 when every bucket this kernel handles holds about one pair
    // (decode with distinct experts), which keeps the inner loop small; else up to 4.
    int tb = 1;
    for (int gi = 0; gi < n_groups; ++gi) {
        const int64_t pairs = (int64_t)groups[gi].m * groups[gi].top_k;
        const bool to_tc = tc_min > 0 && pairs >= (int64_t)tc_min * groups[gi].num_experts;
        if (!to_tc && pairs > groups[gi].num_experts) tb = kTB;
    }
    // buckets of tc_min or more pairs went to the tensor-core path: with tc_min = 2 every
    // bucket left here holds one pair
    if (tc_min > 0 && tc_min <= 2) tb = 1;
    int ints = 0, kmax = 0;
    int64_t max_items = 0;
    for (int gi = 0; gi < n_groups; ++gi) {
        const GemvGroup& S = groups[gi];
        // with the combine fused, every group uses group 0's row tiles (one counter per tile)
        P.g[gi] = group_dev(S, (combine && gi > 0) ? P.g[0].lg_split : lg_split_for(S.k));
        const GroupDev& G = P.g[gi];
        P.hist_off[gi] = ints;
        ints += 2 * S.num_experts;
        kmax = S.k > kmax ? S.k : kmax;
        max_items += (int64_t)G.n_pairs * G.tiles;
    }
    if (combine && P.g[0].tiles > combine->n_counters) return cudaErrorInvalidValue;
    if (max_items == 0 && !combine) return cudaSuccess;
    if (max_items == 0) max_items = 1;
    P.kmax = kmax;
    // at most 32 pairs per group: one warp per group buckets them in registers, and the
    // histogram tables are not needed
    P.fast = n_groups <= kWarps ? 1 : 0;
    for (int gi = 0; gi < n_groups; ++gi) P.fast &= P.g[gi].n_pairs <= 32 ? 1 : 0;
    if (P.fast) ints = 0;
    // tokens per item also bounded so the staged rows fit in ~150 KB of shared memory
    const int64_t per_tok = (int64_t)(kmax / 64) * kPairBytes + (int64_t)(kmax / 32) * 8;
    while (tb > 1 && per_tok * tb > 150 * 1024) tb >>= 1;
    if (tb != 1 && tb != kTB) tb = 1;
    P.tb = tb;
    int off = ((ints * 4) + 15) & ~15;
    P.x_off = off;
    off += (int)(per_tok * tb - (int64_t)(kmax / 32) * 8 * tb);
    off = (off + 15) & ~15;
    P.meta_off = off;
    off += (kmax / 32) * 8 * tb;
    const size_t smem = (size_t)off;
    if (smem > kSmemLimit) return cudaErrorInvalidValue;
    const int kind = (fused_swiglu ? 2 : 0) + (tb == 1 ? 0 : 1);
    void (*kern)(GemvParams) = nullptr;
    switch (kind) {
        case 0: kern = idgemv_kernel<false, 1>; break;
        case 1: kern = idgemv_kernel<false, kTB>; break;
        case 2: kern = idgemv_kernel<true, 1>; break;
        default: kern = idgemv_kernel<true, kTB>; break;
    }
    // The dynamic shared memory limit is raised once per device and kernel (outside any
    // stream capture the caller may start later); launches only query occupancy.
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!g_smem_attr_set[kind][dev]) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
        if (err != cudaSuccess) return err;
        g_smem_attr_set[kind][dev] = true;
    }
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)num_sms() * per_sm;
    if (grid > max_items) grid = max_items;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

// ------------------------------------------------------------------------------------------
// Activation rows of a down launch quantized once into the staged format, for the down
// items to copy instead of quantizing them again in every CTA that takes an item of the row
// (long rows: ~600 CTAs share the 2 rows of a Mixtral-like m = 1 down launch). The same
// arithmetic as the in-kernel staging (stage_row), sub-block by sub-block, so the planes are
// identical. Grid (rows, slices of kPreSlice elements, groups); a programmatic dependent of
// the gate|up launch that waits for it before reading.
constexpr int kPreSlice = 2048;

struct PreStageParams {
    const float* a[kMaxGroups];
    int64_t outer[kMaxGroups], inner[kMaxGroups];
    int top_k[kMaxGroups], rows[kMaxGroups], k[kMaxGroups];
    uint8_t* planes[kMaxGroups];
    float2* meta[kMaxGroups];
    int n_groups;
};

__global__ void __launch_bounds__(kThreads) prestage_kernel(const __grid_constant__ PreStageParams P) {
    pdl_wait();
    pdl_launch_dependents();
    const int g = blockIdx.z, r = blockIdx.x, s0 = blockIdx.y * kPreSlice;
    if (g >= P.n_groups || P.planes[g] == nullptr || r >= P.rows[g] || s0 >= P.k[g]) return;
    const int k = P.k[g], len = min(kPreSlice, k - s0);
    const float* row = P.a[g] + (int64_t)(r / P.top_k[g]) * P.outer[g] + (int64_t)(r % P.top_k[g]) * P.inner[g];
    const int64_t pb = (int64_t)(k / 64) * kPairBytes;
    stage_row<0>(row + s0, len, P.planes[g] + (int64_t)r * pb + (s0 / 64) * kPairBytes,
                 P.meta[g] + (int64_t)r * (k / 32) + s0 / 32);
}

int64_t prestage_bytes(int rows, int k) {
    return (int64_t)rows * ((int64_t)(k / 64) * kPairBytes + (int64_t)(k / 32) * 8);
}

cudaError_t launch_prestage(const GemvGroup* groups, int n_groups, const PreStaged& pre, cudaStream_t stream) {
    PreStageParams P{};
    P.n_groups = n_groups;
    int rows = 0, slices = 0;
    for (int gi = 0; gi < n_groups; ++gi) {
        const GemvGroup& S = groups[gi];
        P.a[gi] = S.a; P.outer[gi] = S.outer; P.inner[gi] = S.inner; P.top_k[gi] = S.top_k;
        P.rows[gi] = S.m * S.top_k; P.k[gi] = S.k;
        P.planes[gi] = const_cast<uint8_t*>(pre.planes[gi]);
        P.meta[gi] = const_cast<float2*>(pre.meta[gi]);
        if (!P.planes[gi]) continue;
        rows = std::max(rows, P.rows[gi]);
        slices = std::max(slices, (S.k + kPreSlice - 1) / kPreSlice);
    }
    if (rows == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows, (unsigned)slices, (unsigned)n_groups);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = take_after_join() ? 0 : 1;  // an ordinary launch right after a join
    return cudaLaunchKernelEx(&cfg, prestage_kernel, P);
}

}  // namespace q4k

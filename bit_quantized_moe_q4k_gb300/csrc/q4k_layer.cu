// q4k_layer.cu -- a small-batch MoE layer in ONE persistent launch: gate|up + SwiGLU of the
// routed experts and the shared expert, their down projections, and the combine.
//
// What it computes (moeflux expert_forward.rs: gate, up, SwiGLU, down, then the batched
// combine y = h_mid + sum_s w_s * expert_out_s + g * shared_out; ferrum-kernels
// q4_k_moe_id_gemv_batched.rs for each projection): exactly what the two-launch layer of
// q4k_gemv.cu computes, bit for bit -- the same work items, activation staging, integer dot
// products, lane reductions and combine order.
//
// Why one launch: with a few tokens the layer moves ~24 MB of weights in ~3.5 us of HBM time
// but takes several times that in latency. A second launch re-reads and re-buckets the ids,
// and can only start once the first launch's CTAs leave the SMs. Here every CTA buckets the
// pairs of both halves once; moves its gate|up item's activation row and weight tiles, and
// then its down tile, into shared memory with bulk copies (outside the SM's load queue);
// starts its down item as soon as the activations of that bucket chunk are written; and the
// CTA of each row tile's last down item combines that tile.
//
// Hand-off between CTAs without zero-initialised state. A launch's tag is next_tag(generation
// word); the generation word is advanced to the tag at the end of the launch (by CTA 0, once
// every CTA has recorded that it read the old value), and a launch count with it. Every result
// a CTA hands to another -- an activation of a gate|up row, a row of an expert's down output --
// is stored as one 64-bit word holding the float under a 32-bit tag made of the launch count
// (bit 31 set, so never zero; no two of the last 2^31 launches share it). CTA 0
// also leaves a stamp for the next launch: its tag bound to this launch's shapes. A launch that
// finds the stamp meant for it (the previous launch on this memory had the same shapes, so it
// wrote every word this one reads, under another tag) takes a word whose tag matches as
// written: readers poll the words themselves, one round trip after the last write. Otherwise
// (the first call on this memory, a call of another shape or after a call with ids out of
// range, a cleared workspace) the words
// could hold anything, and every item also publishes a 64-bit tagged flag (a release store)
// that its readers wait for (acquire) before they read its words. Every wait is bounded in
// time; one that gives up raises Q4K_ERR_TIMEOUT. The waits need every CTA of the grid
// resident at once: the grid is capped at what the SMs hold, it is a cooperative launch (the
// driver starts it only with every CTA resident), and CTAs never wait on a CTA that is itself
// waiting (gate|up items never wait; down items wait only on gate|up items; a combine waits
// only on down items).
#include <algorithm>
#include <cstdlib>
#include <type_traits>

#include "q4k_gemv_common.cuh"
#include "q4k_sm100.cuh"
#include "q4k_sync.cuh"

namespace q4k {

constexpr int kLayerMaxCtas = 1024;   // start-tag words in the sync area
constexpr int kLayerMaxPairs = 32;    // per group: one warp buckets a group
constexpr uint32_t kLayerMaxPolls = 1u << 26;
constexpr int kCbRows = 256;          // h_mid elements of a combine tile kept in shared memory
constexpr int kSyncHead = 4;          // generation word, stamp for the next launch, launch count, pad

// A 4-byte asynchronous copy global -> shared (completes at cp_async_wait_all).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void ld_relaxed_v2(const uint64_t* p, uint64_t& a, uint64_t& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

// The 32-bit tag of every result word of a launch: its launch count, bit 31 set (never zero);
// the words of the last 2^31 launches never carry the tag of this one.
__device__ __forceinline__ uint32_t word_tag(uint64_t count) { return (uint32_t)count | 0x80000000u; }
__device__ __forceinline__ bool word_ready(uint64_t w, uint32_t tag32) { return (uint32_t)(w >> 32) == tag32; }
__device__ __forceinline__ float word_value(uint64_t w) { return __uint_as_float((uint32_t)w); }

struct LayerParams {
    GroupDev a[kMaxGroups];  // gate|up + SwiGLU: routed experts, shared expert
    GroupDev b[kMaxGroups];  // down, same groups (the shared one on the routed row tiles)
    int n_groups;
    int x_off, meta_off;      // dynamic shared memory: staged rows of the larger k
    int slot_off;             // ... and the copy of the CTA's first down tile (use_slot)
    int use_slot;
    int raw_off;              // ... and the gate|up items' raw activation rows (use_xcopy; when
    int use_xcopy;            //     use_slot too they share the slot's space: slot_shares_raw)
    int slot_shares_raw;
    int atile_off, atile_bytes;  // ... and a gate|up item's weight tiles, gate then up (use_atile)
    int use_atile;
    CombineSpec cb;           // y, h_mid, weights, shared_gate, shared_mode (no counters)
    uint64_t* gen;            // [kSyncHead]: generation word, the stamp the previous launch left
                              // for this one, the launch count
    uint64_t shape;           // this launch's shapes, hashed
    uint64_t* cta_tag;        // [kLayerMaxCtas] tag each CTA read
    uint64_t* flag_a;         // [cap_a] one per gate|up item (flag mode)
    uint64_t* flag_b;         // [cap_b] one per down item (flag mode)
    int cap_a, cap_b;
    uint64_t* act64[kMaxGroups];  // gate|up outputs (the down inputs) as tagged words, [pairs, n]
    uint64_t* out64[kMaxGroups];  // down outputs as tagged words, [pairs, hidden]
    int* err_flag;
    uint64_t wait_ns;         // limit of every wait
};

// The stamp for the launch with the given tag and shapes.
__device__ __forceinline__ uint64_t launch_stamp(uint64_t tag, uint64_t shape) { return mix64(tag ^ shape); }

// Block-wide: wait until flags[index(j)] == tag for all j < n. Each thread owns j = tid,
// tid + kThreads, ...; it re-reads only those it has not yet seen set (up to 8 loads per
// round). The reads are acquire loads, so every flag was acquired before the barrier that
// ends the wait, and what any thread of the block does after it is ordered after the
// flags' releases. True when all are set; false once the wait has run for limit_ns or
// kLayerMaxPolls rounds. Uniform over the block.
template <int NTHR = kThreads, class Index>
__device__ __forceinline__ bool wait_tags(const uint64_t* flags, int n, uint64_t tag, uint64_t limit_ns, Index index) {
    int j = threadIdx.x;
    const uint64_t t0 = sm100::global_timer_ns();
    for (uint32_t round = 0;; ++round) {
        uint64_t v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int jj = j + u * NTHR;
            v[u] = jj < n ? ld_acquire_u64(flags + index(jj)) : tag;
        }
        int seen = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (v[u] != tag) break;
            ++seen;
        }
        j += seen * NTHR;
        if (__syncthreads_and(j >= n)) return true;
        const bool late = round >= kLayerMaxPolls || sm100::global_timer_ns() - t0 > limit_ns;
        if (__syncthreads_or(late)) return false;
        __nanosleep(32);
    }
}

// Publish an item in flag mode: its words were stored by this block's threads (the caller
// synchronised the block); one thread stores the tag with release order at GPU scope, which
// makes those words visible first. It is a thread of the last warp: warp 0 locates the next item.
template <int NTHR = kThreads>
__device__ __forceinline__ void publish(uint64_t* flag, uint64_t tag) {
    if (threadIdx.x == NTHR - 32) asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(flag), "l"(tag) : "memory");
}

// Stage the activation rows of an item's nt pairs (k values each) from tagged words: a64 holds
// pair p's row at (p / top_k) * outer + (p % top_k) * inner words. A thread reads four words per
// float4 of the row and re-reads those not yet written by this launch until all are, then they
// are quantized as stage_row does. False when a word was still missing after limit_ns (the
// rows are staged all the same, from what was read). All threads of the block take part.
template <int NTHR = kThreads>
__device__ __forceinline__ bool stage_rows_tagged(const uint64_t* a64, int64_t outer, int64_t inner, int top_k,
                                                  const int* s_pairs, int nt, int k, uint32_t tag32,
                                                  uint64_t limit_ns, uint8_t* xs, float2* meta) {
    constexpr int U = 2;  // float4s per thread and pass
    const int64_t tok_bytes = (int64_t)(k / 64) * kPairBytes;
    const int nf = k / 4;
    bool ok = true;
    const uint64_t t0 = sm100::global_timer_ns();
    for (int t = 0; t < nt; ++t) {
        const int p = s_pairs[t];
        const uint64_t* row = a64 + (int64_t)(p / top_k) * outer + (int64_t)(p % top_k) * inner;
        for (int f0 = 0; f0 < nf; f0 += NTHR * U) {
            uint64_t w[U][4];
            unsigned pending = 0;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int f = f0 + u * NTHR + threadIdx.x;
                if (f < nf) {
                    ld_relaxed_v2(row + 4 * f, w[u][0], w[u][1]);
                    ld_relaxed_v2(row + 4 * f + 2, w[u][2], w[u][3]);
                    pending |= 1u << u;
                } else {
                    w[u][0] = w[u][1] = w[u][2] = w[u][3] = 0;
                }
            }
            for (uint32_t round = 0; pending; ++round) {
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (((pending >> u) & 1u) && word_ready(w[u][0], tag32) && word_ready(w[u][1], tag32) &&
                        word_ready(w[u][2], tag32) && word_ready(w[u][3], tag32))
                        pending &= ~(1u << u);
                if (!pending) break;
                if (round >= kLayerMaxPolls || sm100::global_timer_ns() - t0 > limit_ns) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if ((pending >> u) & 1u) {
                        const int f = f0 + u * NTHR + threadIdx.x;
                        ld_relaxed_v2(row + 4 * f, w[u][0], w[u][1]);
                        ld_relaxed_v2(row + 4 * f + 2, w[u][2], w[u][3]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int f = f0 + u * NTHR + threadIdx.x;  // groups of 8 threads are all in or all out
                if (f0 + u * NTHR >= nf) break;
                const float4 v = make_float4(word_value(w[u][0]), word_value(w[u][1]), word_value(w[u][2]),
                                             word_value(w[u][3]));
                stage_quad(v, f, f < nf, xs + t * tok_bytes, meta + t * (k / 32));
            }
        }
    }
    return __syncthreads_and(ok);
}

// The inputs of a row tile's combine that do not come from this launch (h_mid of the tile's
// rows for every token, routing weights, ids, shared-expert gate logits), copied into shared
// memory while the tile's last down item runs, so the combine's only global loads are the
// expert rows.
struct CombineStage {
    float h[kCbRows];       // h_mid[t][r0 + i] at t*span + i, when m*span <= kCbRows
    float w[kLayerMaxPairs];
    int id[kLayerMaxPairs];
    float g[kLayerMaxPairs];  // shared_gate[t]
};

// Issue the copies of tile [r0, r0 + span) (all threads). The caller waits with
// cp_async_wait_all and a block barrier before reading.
template <int NTHR = kThreads>
__device__ __forceinline__ void combine_stage_issue(const CombineSpec& cb, const int32_t* ids, int n_pairs, int T,
                                                    int H, bool shared, int r0, int span, CombineStage& S) {
    const int m = n_pairs / T;
    if (m * span <= kCbRows)
        for (int idx = threadIdx.x; idx < m * span; idx += NTHR)
            cp_async4(&S.h[idx], cb.h_mid + (int64_t)(idx / span) * H + r0 + idx % span);
    for (int p = threadIdx.x; p < n_pairs; p += NTHR) {
        cp_async4(&S.w[p], cb.weights + p);
        if (ids) cp_async4(&S.id[p], ids + p);
        else S.id[p] = 0;
    }
    if (shared)
        for (int t = threadIdx.x; t < m; t += NTHR) cp_async4(&S.g[t], cb.shared_gate + t);
}

// The combine of rows [r0, r1) of every token from the tagged expert rows (out0: the routed
// pairs' rows, out1: the shared expert's, or null) and the staged inputs:
//   y = h_mid + sum_s w[t*T+s] * out0[t*T+s] + g_t * out1[t]   (slots in order; pairs whose id
// is out of range contribute nothing and their rows are not read) -- the same sums in the same
// order as combine_span. A thread re-reads the words not yet written by this launch until all
// are. False when one was still missing after limit_ns (y is written all the same).
template <int NTHR = kThreads>
__device__ __forceinline__ bool combine_tagged(const CombineSpec& cb, const uint64_t* out0, const uint64_t* out1,
                                               int num_experts, int n_pairs, int T, int H, int r0, int r1,
                                               const CombineStage& S, uint32_t tag32, uint64_t limit_ns) {
    const int m = n_pairs / T;
    const int span = r1 - r0;
    const bool staged_h = m * span <= kCbRows;
    bool ok = true;
    const uint64_t t0 = sm100::global_timer_ns();
    for (int idx = threadIdx.x; idx < m * span; idx += NTHR) {
        const int t = idx / span, r = r0 + idx % span;
        const int64_t o = (int64_t)t * H + r;
        uint64_t v[Q4K_MAX_TOP_K];
        uint64_t sh = 0;
        unsigned need = 0;
#pragma unroll
        for (int s = 0; s < Q4K_MAX_TOP_K; ++s) {
            v[s] = 0;
            if (s < T && id_valid(S.id[t * T + s], num_experts)) need |= 1u << s;
        }
        if (out1) need |= 1u << Q4K_MAX_TOP_K;
        for (uint32_t round = 0;; ++round) {
#pragma unroll
            for (int s = 0; s < Q4K_MAX_TOP_K; ++s)
                if ((need >> s) & 1u) v[s] = ld_relaxed_u64(out0 + (int64_t)(t * T + s) * H + r);
            if ((need >> Q4K_MAX_TOP_K) & 1u) sh = ld_relaxed_u64(out1 + o);
#pragma unroll
            for (int s = 0; s < Q4K_MAX_TOP_K; ++s)
                if (((need >> s) & 1u) && word_ready(v[s], tag32)) need &= ~(1u << s);
            if (((need >> Q4K_MAX_TOP_K) & 1u) && word_ready(sh, tag32)) need &= ~(1u << Q4K_MAX_TOP_K);
            if (!need) break;
            if (round >= kLayerMaxPolls || sm100::global_timer_ns() - t0 > limit_ns) {
                ok = false;
                break;
            }
        }
        float acc = staged_h ? S.h[idx] : cb.h_mid[o];
#pragma unroll
        for (int s = 0; s < Q4K_MAX_TOP_K; ++s)
            if (s < T && id_valid(S.id[t * T + s], num_experts)) acc = fmaf(S.w[t * T + s], word_value(v[s]), acc);
        if (out1) {
            const float g = cb.shared_mode == Q4K_SHARED_SIGMOID ? 1.0f / (1.0f + expf(-S.g[t])) : 1.0f;
            acc = fmaf(g, word_value(sh), acc);
        }
        cb.y[o] = acc;
    }
    return ok;
}

// TB: tokens per item; KB: kind of the down items (kOne, or kPair when one-row items would
// outnumber the resident CTAs: a CTA then streams a tile of twice the rows with the registers
// the fused gate|up items use).
template <int TB, int KB>
__global__ void __launch_bounds__(kThreads, 3) layer_kernel(const __grid_constant__ LayerParams P) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ FastGroup s_fast[2][kMaxGroups];  // [half][group]: buckets with item offsets
    __shared__ int s_items[2][kMaxGroups + 1];
    __shared__ int s_bad[2][kMaxGroups];
    __shared__ int s_pairs[kTB];
    __shared__ int s_info[6];                    // group, rank, expert, tile, tokens, chunk
    __shared__ int s_chunk_b[2 * kLayerMaxPairs]; // first down item of every (group, bucket, chunk)
    __shared__ int s_n_chunks;
    __shared__ uint64_t s_tag;
    __shared__ uint32_t s_tag32;                 // the tag of this launch's result words
    __shared__ int s_fast_mode;                  // the stamp was meant for this launch: tags suffice
    __shared__ __align__(8) uint64_t s_bar;  // the down tile's copy into shared memory
    __shared__ __align__(8) uint64_t s_xbar; // a gate|up item's activation rows' copy
    __shared__ __align__(8) uint64_t s_abar; // a gate|up item's weight tiles' copy
    __shared__ int s_never;                  // (bounded waits take an abort word; never set)
    __shared__ CombineStage s_cbs;           // the inputs of this CTA's combine

    // (not launched as a programmatic dependent, so earlier kernels of the stream are complete
    // and the wait returns at once); the next kernel may launch early: it can only take space
    // left over once every CTA of this grid has started, which the trigger implies
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // the generation word's, the stamp's and the launch count's loads overlap the bucketing
    const uint64_t gen = threadIdx.x == 0 ? ld_relaxed_u64(P.gen) : 0;
    const uint64_t stamp = threadIdx.x == 0 ? ld_relaxed_u64(P.gen + 1) : 0;
    const uint64_t count = threadIdx.x == 0 ? ld_relaxed_u64(P.gen + 2) : 0;
    {   // bucketing: warp w takes half w >> 1 (gate|up, down), group w & 1
        const int half = warp >> 1, gi = warp & 1;
        if (gi < P.n_groups) {
            const GroupDev& G = half ? P.b[gi] : P.a[gi];
            fast_bucket(G.ids, G.n_pairs, G.num_experts, G.tiles, TB, 0, s_fast[half][gi], &s_bad[half][gi]);
        }
    }
    __syncthreads();
    if (threadIdx.x < 2) {
        const int half = threadIdx.x;
        s_items[half][0] = 0;
        for (int gi = 0; gi < P.n_groups; ++gi) {
            const FastGroup& F = s_fast[half][gi];
            s_items[half][gi + 1] = s_items[half][gi] + F.start[F.U];
        }
        if (half == 0) {
            s_never = 0;
            sm100::mbar_init(&s_bar, 1);
            sm100::mbar_init(&s_xbar, 1);
            sm100::mbar_init(&s_abar, 1);
            sm100::fence_mbar_init();
            const uint64_t tag = next_tag(gen);
            s_tag = tag;
            s_tag32 = word_tag(count + 1);
            s_fast_mode = stamp == launch_stamp(tag, P.shape);
            st_relaxed_u64(P.cta_tag + blockIdx.x, tag);  // this CTA has read the generation
        }
    }
    __syncthreads();
    const uint64_t tag = s_tag;
    const uint32_t tag32 = s_tag32;
    const bool fast = s_fast_mode;
    const int na = s_items[0][P.n_groups], nb = s_items[1][P.n_groups];
    // the caps bound any bucketing (chunks <= pairs); checked all the same
    const bool fits = na <= P.cap_a && nb <= P.cap_b;
    bool ok = fits;
    const int64_t grid = gridDim.x, cta = blockIdx.x;
    const int a0 = (int)(cta * na / grid), a1 = (int)((cta + 1) * na / grid);
    const int b0 = (int)(cta * nb / grid), b1 = (int)((cta + 1) * nb / grid);
    uint8_t* xs = smem + P.x_off;
    float2* meta = reinterpret_cast<float2*>(smem + P.meta_off);
    uint8_t* slot = smem + P.slot_off;                          // the first down tile's copy
    float* raw = reinterpret_cast<float*>(smem + P.raw_off);    // gate|up activation rows
    uint8_t* atile = smem + P.atile_off;                        // gate|up weight tiles: gate, up

    // ---- the CTA's first down tile (its rows are consecutive in the slab) is copied into
    // shared memory with one bulk copy. When the raw activation rows share its space the copy
    // starts after the last gate|up staging, else right away.
    const bool slot_item = ok && P.use_slot && b0 < b1;
    bool slot_issued = false, slot_waited = false;
    auto issue_slot = [&]() {  // all threads
        if (warp == 0) {
            const FastLoc L = fast_locate(s_fast[1], s_items[1], P.b, P.n_groups, TB, b0, nullptr);
            if (lane == 0) {
                const GroupDev& G = P.b[L.gi];
                const int tr = item_tile_rows(G.lg_split, KB);
                const int r0 = L.tile * tr, rows = min(tr, G.n - r0);
                const uint32_t bytes = (uint32_t)((int64_t)rows * G.nb01);
                sm100::fence_proxy_async_smem();  // reads of a shared raw area come first
                sm100::mbar_arrive_expect_tx(&s_bar, bytes);
                sm100::bulk_g2s(slot, G.w + (int64_t)L.e * G.nb02 + (int64_t)r0 * G.nb01, bytes, &s_bar);
            }
        }
        slot_issued = true;
    };
    if (slot_item && a0 == a1) issue_slot();
    // the bulk copies of the gate|up items: bit 0 / 1 = a copy on s_xbar / s_abar not yet waited
    // for (drained before the CTA leaves, also after a wait gave up), bit 2 / 3 = the parity of
    // the phase that barrier completes next
    uint32_t cps = 0;

    int staged = -1;  // (half, group, rank, chunk) of the staged activation rows
    // ---- gate|up + SwiGLU items: activation rows and (use_atile) the weight tiles of both slabs
    // arrive by bulk copy, which keeps them out of the SM's load queue
    auto gate_up_item = [&](auto from_smem, int item, int gi, const GroupDev& G, int e, int tile, int nt,
                            int key) -> bool {
        constexpr bool SM = decltype(from_smem)::value;
        ItemLane<kFused, SM> IL;
        if constexpr (!SM) item_issue<kFused>(G, e, tile, lane, warp, IL);
        if (key != staged) {
            if (P.use_xcopy) {
                if (!__syncthreads_and(mbar_wait_for(&s_xbar, (cps >> 2) & 1u, &s_never, P.wait_ns))) return false;
                cps = (cps ^ 4u) & ~1u;
                stage_rows_smem(raw, nt, G.k, xs, meta);
            } else {
                stage_rows<false>(G, s_pairs, nt, xs, meta);
            }
            staged = key;
        }
        if (slot_item && !slot_issued && item == a1 - 1) {
            __syncthreads();  // the last reads of the raw rows
            issue_slot();
        }
        if constexpr (SM) {
            if (!__syncthreads_and(mbar_wait_for(&s_abar, (cps >> 3) & 1u, &s_never, P.wait_ns))) return false;
            cps = (cps ^ 8u) & ~2u;
            item_issue<kFused, true>(G, e, tile, lane, warp, IL, atile, atile + P.atile_bytes);
        }
        __syncthreads();
        item_compute<kFused, TB>(G, IL, s_pairs, nt, xs, meta, lane, P.act64[gi], tag32);
        if (!fast) {
            __syncthreads();
            publish(P.flag_a + item, tag);
        }
        return true;
    };
    for (int item = a0; ok && item < a1; ++item) {
        if (warp == 0) {
            const FastLoc L = fast_locate(s_fast[0], s_items[0], P.a, P.n_groups, TB, item, s_pairs);
            if (lane == 0) { s_info[0] = L.gi; s_info[1] = L.r; s_info[2] = L.e; s_info[3] = L.tile; s_info[4] = L.nt; s_info[5] = L.chunk; }
        }
        __syncthreads();
        const int gi = s_info[0], r = s_info[1], e = s_info[2], tile = s_info[3], nt = s_info[4], chunk = s_info[5];
        const GroupDev& G = P.a[gi];
        const int key = ((gi * 32 + r) * 32 + chunk) * 2;
        const bool xc = key != staged && P.use_xcopy;  // (uniform) this item's copies
        cps |= (xc ? 1u : 0u) | (P.use_atile ? 2u : 0u);
        if (threadIdx.x == 0) {
            if (xc || P.use_atile) sm100::fence_proxy_async_smem();  // earlier reads of these areas first
            if (xc) {
                sm100::mbar_arrive_expect_tx(&s_xbar, (uint32_t)(nt * G.k * 4));
                for (int t = 0; t < nt; ++t)
                    sm100::bulk_g2s(raw + t * G.k, act_row(G, s_pairs[t]), (uint32_t)(G.k * 4), &s_xbar);
            }
            if (P.use_atile) {
                const int tra = item_tile_rows(G.lg_split, kFused);
                const int r0 = tile * tra, rows = min(tra, G.n - r0);
                const uint32_t bytes = (uint32_t)((int64_t)rows * G.nb01);
                const int64_t src = (int64_t)e * G.nb02 + (int64_t)r0 * G.nb01;
                sm100::mbar_arrive_expect_tx(&s_abar, 2 * bytes);
                sm100::bulk_g2s(atile, G.w + src, bytes, &s_abar);
                sm100::bulk_g2s(atile + P.atile_bytes, G.w2 + src, bytes, &s_abar);
            }
        }
        // a down tile with its own space goes into the copy queue right behind the first item's
        // weight tiles, which are needed first
        if (slot_item && !slot_issued && !P.slot_shares_raw) issue_slot();
        ok = P.use_atile ? gate_up_item(std::true_type{}, item, gi, G, e, tile, nt, key)
                         : gate_up_item(std::false_type{}, item, gi, G, e, tile, nt, key);
    }

    // ---- down items: each reads the activations of its chunk (all their row tiles) as they are
    // written (flag mode: after the gate|up items' flags); the first from its shared-memory copy
    // when there is one. The CTA of a row tile's last down item (the tile's item in the last
    // chunk: items nb - tiles .. nb - 1) combines that tile.
    const bool shared = P.cb.shared_mode != Q4K_SHARED_NONE && P.n_groups > 1;
    const int tr = item_tile_rows(P.b[0].lg_split, KB);
    const int n_tiles = P.b[0].tiles;
    const int first_last = nb - n_tiles;  // first of the items that end a tile
    if (threadIdx.x == 0 && !fast) {  // down items of tile 0 of every chunk (a combine's wait list)
        int nc = 0;
        for (int gi = 0; gi < P.n_groups; ++gi) {
            const FastGroup& F = s_fast[1][gi];
            for (int r = 0; r < F.U; ++r) {
                const int chunks = (F.start[r + 1] - F.start[r]) / P.b[gi].tiles;
                for (int c = 0; c < chunks && nc < 2 * kLayerMaxPairs; ++c)
                    s_chunk_b[nc++] = s_items[1][gi] + F.start[r] + c * P.b[gi].tiles;
            }
        }
        s_n_chunks = nc;
    }
    auto combine_tile = [&](int t) -> bool {  // all threads; the inputs were staged
        const GroupDev& R = P.b[0];
        if (!fast && !wait_tags(P.flag_b, s_n_chunks, tag, P.wait_ns, [t](int j) { return s_chunk_b[j] + t; }))
            return false;
        const bool done = combine_tagged(P.cb, P.out64[0], shared ? P.out64[1] : nullptr, R.num_experts, R.n_pairs,
                                         R.top_k, R.n, t * tr, min(R.n, (t + 1) * tr), s_cbs, tag32, P.wait_ns);
        return __syncthreads_and(done);
    };
    auto down_item = [&](auto& IL, int item, const GroupDev& G, int gi, int r, int nt, int chunk, int tile) -> bool {
        const int key = ((gi * 32 + r) * 32 + chunk) * 2 + 1;
        const bool ends_tile = item >= first_last;
        if (ends_tile) {
            const GroupDev& R = P.b[0];
            combine_stage_issue(P.cb, R.ids, R.n_pairs, R.top_k, R.n, shared, tile * tr,
                                min(R.n, (tile + 1) * tr) - tile * tr, s_cbs);
        }
        if (key != staged) {
            if (!fast) {
                const int first = s_items[0][gi] + s_fast[0][gi].start[r] + chunk * P.a[gi].tiles;
                if (!wait_tags(P.flag_a, P.a[gi].tiles, tag, P.wait_ns, [first](int j) { return first + j; }))
                    return false;
            }
            if (!stage_rows_tagged(P.act64[gi], G.outer, G.inner, G.top_k, s_pairs, nt, G.k, tag32, P.wait_ns, xs, meta))
                return false;
            staged = key;
        }
        __syncthreads();
        item_compute<KB, TB>(G, IL, s_pairs, nt, xs, meta, lane, P.out64[gi], tag32);
        __syncthreads();
        if (!fast) publish(P.flag_b + item, tag);
        if (ends_tile) {
            cp_async_wait_all();
            __syncthreads();
            return combine_tile(tile);
        }
        return true;
    };
    for (int item = b0; ok && item < b1; ++item) {
        if (warp == 0) {
            const FastLoc L = fast_locate(s_fast[1], s_items[1], P.b, P.n_groups, TB, item, s_pairs);
            if (lane == 0) { s_info[0] = L.gi; s_info[1] = L.r; s_info[2] = L.e; s_info[3] = L.tile; s_info[4] = L.nt; s_info[5] = L.chunk; }
        }
        __syncthreads();
        const int gi = s_info[0], r = s_info[1], e = s_info[2], tile = s_info[3], nt = s_info[4], chunk = s_info[5];
        const GroupDev& G = P.b[gi];
        if (slot_issued && item == b0) {
            ok = __syncthreads_and(mbar_wait_for(&s_bar, 0, &s_never, P.wait_ns));
            slot_waited = ok;
            if (!ok) break;
            ItemLane<KB, true> IL;
            item_issue<KB, true>(G, e, tile, lane, warp, IL, slot);
            ok = down_item(IL, item, G, gi, r, nt, chunk, tile);
        } else {
            ItemLane<KB> IL;
            item_issue<KB>(G, e, tile, lane, warp, IL);  // weights do not depend on gate|up
            ok = down_item(IL, item, G, gi, r, nt, chunk, tile);
        }
    }
    // no down item at all (every id out of range, no shared expert): y = h_mid, tiles split
    // over the CTAs
    if (ok && nb == 0) {
        const GroupDev& R = P.b[0];
        for (int t = (int)(cta * n_tiles / grid); ok && t < (int)((cta + 1) * n_tiles / grid); ++t) {
            __syncthreads();
            combine_stage_issue(P.cb, R.ids, R.n_pairs, R.top_k, R.n, shared, t * tr, min(R.n, (t + 1) * tr) - t * tr,
                                s_cbs);
            cp_async_wait_all();
            __syncthreads();
            ok = combine_tile(t);
        }
    }
    // a copy still in flight must land before the CTA leaves (after an abort)
    cp_async_wait_all();
    if (slot_issued && !slot_waited) sm100::mbar_wait(&s_bar, 0, &s_never);
    if (cps & 1u) sm100::mbar_wait(&s_xbar, (cps >> 2) & 1u, &s_never);
    if (cps & 2u) sm100::mbar_wait(&s_abar, (cps >> 3) & 1u, &s_never);

    if (threadIdx.x == 0) {
        if (!fits) raise_flag(P.err_flag, Q4K_ERR_LIMIT);
        else if (!ok) raise_flag(P.err_flag, Q4K_ERR_TIMEOUT);
        if (blockIdx.x == 0)
            for (int half = 0; half < 2; ++half)
                for (int gi = 0; gi < P.n_groups; ++gi)
                    if (s_bad[half][gi]) raise_flag(P.err_flag, Q4K_ERR_EXPERT_ID);
    }
    // ---- advance the generation and the launch count once every CTA has read them, and leave
    // the next launch its stamp (this launch's shapes under the next tag). A launch that saw an
    // id out of range wrote no words for that pair, so it leaves none: the next launch of the
    // same shapes could read those words.
    if (blockIdx.x == 0) {
        const bool all = wait_tags(P.cta_tag, (int)gridDim.x, tag, P.wait_ns, [](int j) { return j; });
        if (threadIdx.x == 0) {
            bool clean = true;
            for (int half = 0; half < 2; ++half)
                for (int gi = 0; gi < P.n_groups; ++gi) clean = clean && !s_bad[half][gi];
            if (all) {
                st_relaxed_u64(P.gen + 1, clean ? launch_stamp(next_tag(tag), P.shape) : 0ull);
                st_relaxed_u64(P.gen + 2, count + 1);
                st_relaxed_u64(P.gen, tag);
            } else {
                raise_flag(P.err_flag, Q4K_ERR_TIMEOUT);
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
// The wide layer kernel: the same layer, items, hand-offs and sums as layer_kernel, for the
// case where every CTA takes at most one gate|up item and at most one down item, both with
// their weight tiles in shared memory (the decode layer). Its CTAs have 256 threads: two groups
// of four warps, h = warp >> 2. In a gate|up item group 0 folds the gate rows and group 1 the
// up rows of the tile; in a down item (tiles of 64 rows) group 0 folds the first 32 rows and
// group 1 the rest. Within a group the lanes are laid out as in item_issue, and each lane
// folds one row of one slab over its blocks in the canonical order, so every sum equals
// layer_kernel's (and the two-launch layer's) bit for bit. Twice the warps per CTA, each with
// half the work: the dot products are bound by the latency of each warp's chain, not by the
// SM's issue rate.
constexpr int kWideThreads = 256;
constexpr int kWideCopyRows = 8;   // rows per bulk copy of a gate|up weight tile

// One lane's fold of its row (wrow: the row's blocks in shared memory; zeros when !row_ok)
// against token 0's staged planes, then the xor reduction over the row's 4*S lanes: the row's
// sum in each of them.
__device__ __forceinline__ float row_fold_smem(const uint8_t* wrow, const GroupDev& G, int lane, const uint8_t* xs,
                                               const float2* meta, bool row_ok) {
    const int S = 1 << G.lg_split;
    const int c = lane & 3, sl = (lane >> 2) & (S - 1);
    const int nb = G.k / kQK;
    const int nbl = sl < nb ? (nb - sl + S - 1) / S : 0;
    float acc = 0.0f;
    for (int i = 0; i < nbl; ++i) {
        const int b = sl + S * i;
        uint4 H = make_uint4(0, 0, 0, 0), Q0 = H, Q1 = H;
        if (row_ok) {
            const uint8_t* p = wrow + (int64_t)b * kBlockBytes;
            H = ldw16<true>(p); Q0 = ldw16<true>(p + 16 + 32 * c); Q1 = ldw16<true>(p + 32 + 32 * c);
        }
        float sa, ma, sb, mb;
        block_scales(H, c, sa, ma, sb, mb);
        const uint4* xp = reinterpret_cast<const uint4*>(xs + (4 * b + c) * kPairBytes);
        const float4 mt = *reinterpret_cast<const float4*>(meta + 8 * b + 2 * c);
        int Sa, Sb;
        dot64(Q0, Q1, xp, Sa, Sb);
        acc = fold_term(acc, block_term(mt, sa, ma, sb, mb, Sa, Sb), i == 0);
    }
    for (int off = 1; off < 4 * S; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    return acc;
}

__global__ void __launch_bounds__(kWideThreads, 3) layer_wide_kernel(const __grid_constant__ LayerParams P) {
    constexpr int NT = kWideThreads;
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ FastGroup s_fast[2][kMaxGroups];
    __shared__ int s_items[2][kMaxGroups + 1];
    __shared__ int s_bad[2][kMaxGroups];
    __shared__ int s_pairs[kTB];
    __shared__ int s_info[6];
    __shared__ int s_chunk_b[2 * kLayerMaxPairs];
    __shared__ int s_n_chunks;
    __shared__ uint64_t s_tag;
    __shared__ uint32_t s_tag32;
    __shared__ int s_fast_mode;
    __shared__ __align__(8) uint64_t s_bar;   // the down tile's copy
    __shared__ __align__(8) uint64_t s_xbar;  // the gate|up item's activation row's copy
    __shared__ __align__(8) uint64_t s_abar;  // the gate|up item's weight tiles' copy
    __shared__ int s_never;
    __shared__ float s_g[32];                 // a gate|up tile's gate sums (group 0 -> group 1)
    __shared__ CombineStage s_cbs;

    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, h = warp >> 2, w4 = warp & 3;
    const uint64_t gen = threadIdx.x == 0 ? ld_relaxed_u64(P.gen) : 0;
    const uint64_t stamp = threadIdx.x == 0 ? ld_relaxed_u64(P.gen + 1) : 0;
    const uint64_t count = threadIdx.x == 0 ? ld_relaxed_u64(P.gen + 2) : 0;
    if (warp < 4) {  // bucketing: warp w takes half w >> 1, group w & 1
        const int half = warp >> 1, gi = warp & 1;
        if (gi < P.n_groups) {
            const GroupDev& G = half ? P.b[gi] : P.a[gi];
            fast_bucket(G.ids, G.n_pairs, G.num_experts, G.tiles, 1, 0, s_fast[half][gi], &s_bad[half][gi]);
        }
    }
    __syncthreads();
    if (threadIdx.x < 2) {
        const int half = threadIdx.x;
        s_items[half][0] = 0;
        for (int gi = 0; gi < P.n_groups; ++gi) {
            const FastGroup& F = s_fast[half][gi];
            s_items[half][gi + 1] = s_items[half][gi] + F.start[F.U];
        }
        if (half == 0) {
            s_never = 0;
            sm100::mbar_init(&s_bar, 1);
            sm100::mbar_init(&s_xbar, 1);
            sm100::mbar_init(&s_abar, 1);
            sm100::fence_mbar_init();
            const uint64_t tag = next_tag(gen);
            s_tag = tag;
            s_tag32 = word_tag(count + 1);
            s_fast_mode = stamp == launch_stamp(tag, P.shape);
            st_relaxed_u64(P.cta_tag + blockIdx.x, tag);
        }
    }
    __syncthreads();
    const uint64_t tag = s_tag;
    const uint32_t tag32 = s_tag32;
    const bool fast = s_fast_mode;
    const int na = s_items[0][P.n_groups], nb = s_items[1][P.n_groups];
    const int64_t grid = gridDim.x, cta = blockIdx.x;
    // at most one item of each half per CTA (the caps bound na and nb; checked all the same)
    const bool fits = na <= P.cap_a && nb <= P.cap_b && na <= grid && nb <= grid;
    bool ok = fits;
    const int a0 = (int)(cta * na / grid), a1 = (int)((cta + 1) * na / grid);
    const int b0 = (int)(cta * nb / grid), b1 = (int)((cta + 1) * nb / grid);
    uint8_t* xs = smem + P.x_off;
    float2* meta = reinterpret_cast<float2*>(smem + P.meta_off);
    uint8_t* slot = smem + P.slot_off;
    float* raw = reinterpret_cast<float*>(smem + P.raw_off);
    uint8_t* atile = smem + P.atile_off;
    const bool has_a = ok && a0 < a1, has_b = ok && b0 < b1;
    bool slot_issued = false, slot_waited = false;
    uint32_t cps = 0;  // bit 0 / 1: the x copy / the weight tiles' copy not yet waited for
    auto issue_slot = [&]() {  // all threads
        if (warp == 0) {
            const FastLoc L = fast_locate(s_fast[1], s_items[1], P.b, P.n_groups, 1, b0, nullptr);
            if (lane == 0) {
                const GroupDev& G = P.b[L.gi];
                const int tr = item_tile_rows(G.lg_split, kPair);
                const int r0 = L.tile * tr, rows = min(tr, G.n - r0);
                const uint32_t bytes = (uint32_t)((int64_t)rows * G.nb01);
                sm100::fence_proxy_async_smem();
                sm100::mbar_arrive_expect_tx(&s_bar, bytes);
                sm100::bulk_g2s(slot, G.w + (int64_t)L.e * G.nb02 + (int64_t)r0 * G.nb01, bytes, &s_bar);
            }
        }
        slot_issued = true;
    };
    if (has_b && !has_a) issue_slot();

    // ---- the gate|up + SwiGLU item
    if (has_a) {
        if (warp == 0) {
            const FastLoc L = fast_locate(s_fast[0], s_items[0], P.a, P.n_groups, 1, a0, s_pairs);
            if (lane == 0) { s_info[0] = L.gi; s_info[2] = L.e; s_info[3] = L.tile; }
        }
        __syncthreads();
        const int gi = s_info[0], e = s_info[2], tile = s_info[3];
        const GroupDev& G = P.a[gi];
        cps = 3u;
        if (threadIdx.x == 0) {
            sm100::mbar_arrive_expect_tx(&s_xbar, (uint32_t)(G.k * 4));
            sm100::bulk_g2s(raw, act_row(G, s_pairs[0]), (uint32_t)(G.k * 4), &s_xbar);
            const int tra = item_tile_rows(G.lg_split, kFused);
            const int r0 = tile * tra, rows = min(tra, G.n - r0);
            const uint32_t bytes = (uint32_t)((int64_t)rows * G.nb01);
            const int64_t src = (int64_t)e * G.nb02 + (int64_t)r0 * G.nb01;
            sm100::mbar_arrive_expect_tx(&s_abar, 2 * bytes);
            // in copies of a few rows, gate and up alternating: the copy engine of an SM then
            // serves its CTAs' tiles side by side rather than one CTA's after another's
            const uint32_t piece = (uint32_t)(kWideCopyRows * G.nb01);
            for (uint32_t o = 0; o < bytes; o += piece) {
                const uint32_t n = min(piece, bytes - o);
                sm100::bulk_g2s(atile + o, G.w + src + o, n, &s_abar);
                sm100::bulk_g2s(atile + P.atile_bytes + o, G.w2 + src + o, n, &s_abar);
            }
        }
        ok = __syncthreads_and(mbar_wait_for(&s_xbar, 0, &s_never, P.wait_ns));
        if (ok) {
            cps &= ~1u;
            stage_row<2, NT>(raw, G.k, xs, meta, threadIdx.x);
            ok = __syncthreads_and(mbar_wait_for(&s_abar, 0, &s_never, P.wait_ns));
        }
        if (ok) {
            cps &= ~2u;
            // the down tile takes the raw row's space (read before the barrier above); its copy
            // starts once this CTA's gate|up tiles are in, so those have HBM to themselves
            // (15.48 against 15.78 us on the Qwen3-like m = 1 layer)
            if (has_b) issue_slot();
            const int lgS = G.lg_split, S = 1 << lgS, rpw = 8 >> lgS;
            const int rt = w4 * rpw + (lane >> (2 + lgS));
            const int row = tile * item_tile_rows(lgS, kFused) + rt;
            const bool row_ok = row < G.n;
            const uint8_t* wrow = atile + (h ? P.atile_bytes : 0) + (int64_t)(row_ok ? rt : 0) * G.nb01;
            const float v = row_fold_smem(wrow, G, lane, xs, meta, row_ok);
            const bool writer = (lane & (4 * S - 1)) == 0;
            if (h == 0 && writer) s_g[rt] = v;
            __syncthreads();
            if (h == 1 && writer && row_ok)
                st_tagged(P.act64[gi] + (int64_t)s_pairs[0] * G.n + row, silu(s_g[rt]) * v, tag32);
            if (!fast) {
                __syncthreads();
                publish<NT>(P.flag_a + a0, tag);
            }
        }
    }

    // ---- the down item; the CTA of a row tile's last down item combines the tile
    const bool shared = P.cb.shared_mode != Q4K_SHARED_NONE && P.n_groups > 1;
    const int tr = item_tile_rows(P.b[0].lg_split, kPair);
    const int n_tiles = P.b[0].tiles;
    if (threadIdx.x == 0 && !fast) {
        int nc = 0;
        for (int gi = 0; gi < P.n_groups; ++gi) {
            const FastGroup& F = s_fast[1][gi];
            for (int r = 0; r < F.U; ++r) {
                const int chunks = (F.start[r + 1] - F.start[r]) / P.b[gi].tiles;
                for (int c = 0; c < chunks && nc < 2 * kLayerMaxPairs; ++c)
                    s_chunk_b[nc++] = s_items[1][gi] + F.start[r] + c * P.b[gi].tiles;
            }
        }
        s_n_chunks = nc;
    }
    auto combine_tile = [&](int t) -> bool {
        const GroupDev& R = P.b[0];
        if (!fast && !wait_tags<NT>(P.flag_b, s_n_chunks, tag, P.wait_ns, [t](int j) { return s_chunk_b[j] + t; }))
            return false;
        const bool done = combine_tagged<NT>(P.cb, P.out64[0], shared ? P.out64[1] : nullptr, R.num_experts,
                                             R.n_pairs, R.top_k, R.n, t * tr, min(R.n, (t + 1) * tr), s_cbs, tag32,
                                             P.wait_ns);
        return __syncthreads_and(done);
    };
    if (ok && has_b) {
        if (warp == 0) {
            const FastLoc L = fast_locate(s_fast[1], s_items[1], P.b, P.n_groups, 1, b0, s_pairs);
            if (lane == 0) { s_info[0] = L.gi; s_info[1] = L.r; s_info[3] = L.tile; s_info[5] = L.chunk; }
        }
        __syncthreads();
        const int gi = s_info[0], r = s_info[1], tile = s_info[3], chunk = s_info[5];
        const GroupDev& G = P.b[gi];
        const bool ends_tile = b0 >= nb - n_tiles;
        if (ends_tile) {
            const GroupDev& R = P.b[0];
            combine_stage_issue<NT>(P.cb, R.ids, R.n_pairs, R.top_k, R.n, shared, tile * tr,
                                    min(R.n, (tile + 1) * tr) - tile * tr, s_cbs);
        }
        if (!fast) {
            const int first = s_items[0][gi] + s_fast[0][gi].start[r] + chunk * P.a[gi].tiles;
            ok = wait_tags<NT>(P.flag_a, P.a[gi].tiles, tag, P.wait_ns, [first](int j) { return first + j; });
        }
        if (ok) ok = stage_rows_tagged<NT>(P.act64[gi], G.outer, G.inner, G.top_k, s_pairs, 1, G.k, tag32, P.wait_ns, xs,
                                           meta);
        if (ok) {
            ok = __syncthreads_and(mbar_wait_for(&s_bar, 0, &s_never, P.wait_ns));
            slot_waited = ok;
        }
        if (ok) {
            const int lgS = G.lg_split, S = 1 << lgS, rpw = 8 >> lgS;
            const int rt = h * (kWarps * rpw) + w4 * rpw + (lane >> (2 + lgS));
            const int row = tile * tr + rt;
            const bool row_ok = row < G.n;
            const float v = row_fold_smem(slot + (int64_t)(row_ok ? rt : 0) * G.nb01, G, lane, xs, meta, row_ok);
            if ((lane & (4 * S - 1)) == 0 && row_ok) st_tagged(P.out64[gi] + (int64_t)s_pairs[0] * G.n + row, v, tag32);
            __syncthreads();
            if (!fast) publish<NT>(P.flag_b + b0, tag);
            if (ends_tile) {
                cp_async_wait_all();
                __syncthreads();
                ok = combine_tile(tile);
            }
        }
    }
    if (ok && nb == 0) {  // no down item at all: y = h_mid, tiles split over the CTAs
        const GroupDev& R = P.b[0];
        for (int t = (int)(cta * n_tiles / grid); ok && t < (int)((cta + 1) * n_tiles / grid); ++t) {
            __syncthreads();
            combine_stage_issue<NT>(P.cb, R.ids, R.n_pairs, R.top_k, R.n, shared, t * tr, min(R.n, (t + 1) * tr) - t * tr,
                                    s_cbs);
            cp_async_wait_all();
            __syncthreads();
            ok = combine_tile(t);
        }
    }
    // copies still in flight land before the CTA leaves (after a wait gave up)
    cp_async_wait_all();
    if (slot_issued && !slot_waited) sm100::mbar_wait(&s_bar, 0, &s_never);
    if (cps & 1u) sm100::mbar_wait(&s_xbar, 0, &s_never);
    if (cps & 2u) sm100::mbar_wait(&s_abar, 0, &s_never);

    if (threadIdx.x == 0) {
        if (!fits) raise_flag(P.err_flag, Q4K_ERR_LIMIT);
        else if (!ok) raise_flag(P.err_flag, Q4K_ERR_TIMEOUT);
        if (blockIdx.x == 0)
            for (int half = 0; half < 2; ++half)
                for (int gi = 0; gi < P.n_groups; ++gi)
                    if (s_bad[half][gi]) raise_flag(P.err_flag, Q4K_ERR_EXPERT_ID);
    }
    if (blockIdx.x == 0) {
        const bool all = wait_tags<NT>(P.cta_tag, (int)gridDim.x, tag, P.wait_ns, [](int j) { return j; });
        if (threadIdx.x == 0) {
            bool clean = true;
            for (int half = 0; half < 2; ++half)
                for (int gi = 0; gi < P.n_groups; ++gi) clean = clean && !s_bad[half][gi];
            if (all) {
                st_relaxed_u64(P.gen + 1, clean ? launch_stamp(next_tag(tag), P.shape) : 0ull);
                st_relaxed_u64(P.gen + 2, count + 1);
                st_relaxed_u64(P.gen, tag);
            } else {
                raise_flag(P.err_flag, Q4K_ERR_TIMEOUT);
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
uint64_t wait_limit_ns() {
    const char* s = getenv("Q4K_WAIT_NS");
    if (s) {
        const long long v = atoll(s);
        if (v > 0) return (uint64_t)v;
    }
    return sm100::kWaitNs;
}

namespace {

struct LayerPlan {
    int lg_a[kMaxGroups], lg_b[kMaxGroups];
    int64_t cap_a, cap_b;
};

// Row splits and the item caps for down items of kind kb (chunks <= pairs per bucket, so
// items <= pairs x tiles).
LayerPlan plan_of(const GemvGroup* gu, const GemvGroup* dn, int n_groups, int kb) {
    LayerPlan L{};
    for (int gi = 0; gi < n_groups; ++gi) {
        L.lg_a[gi] = lg_split_for(gu[gi].k);
        L.lg_b[gi] = gi == 0 ? lg_split_for(dn[0].k) : L.lg_b[0];
        const int ta = item_tile_rows(L.lg_a[gi], kFused), tb = item_tile_rows(L.lg_b[gi], kb);
        L.cap_a += (int64_t)gu[gi].m * gu[gi].top_k * ((gu[gi].n + ta - 1) / ta);
        L.cap_b += (int64_t)dn[gi].m * dn[gi].top_k * ((dn[gi].n + tb - 1) / tb);
    }
    return L;
}

bool g_layer_attr_set[5][64] = {};

// Result words of the single-launch layer: the gate|up outputs of the routed pairs and of the
// shared expert's tokens, then the down outputs of both (64-bit tagged words, row-major).
int64_t result_words(int m, int top_k, int hidden, int inter, int shared_inter) {
    const int64_t pairs = (int64_t)m * top_k;
    return pairs * inter + (int64_t)m * shared_inter + pairs * hidden + (shared_inter > 0 ? (int64_t)m * hidden : 0);
}

// splitmix64's output function on the host (Steele, Lea, Flood 2014), for the shape word.
uint64_t host_mix64(uint64_t z) {
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

}  // namespace

size_t layer_sync_words(int m, int top_k, int hidden, int inter, int shared_inter) {
    if (m < 1 || (int64_t)m * top_k > kLayerMaxPairs || (shared_inter > 0 && m > kLayerMaxPairs)) return 0;
    GemvGroup gu[2] = {}, dn[2] = {};
    gu[0] = GemvGroup{nullptr, nullptr, nullptr, nullptr, 0, 0, nullptr, 1, m, top_k, inter, hidden};
    dn[0] = GemvGroup{nullptr, nullptr, nullptr, nullptr, 0, 0, nullptr, 1, m, top_k, hidden, inter};
    int ng = 1;
    if (shared_inter > 0) {
        gu[1] = GemvGroup{nullptr, nullptr, nullptr, nullptr, 0, 0, nullptr, 1, m, 1, shared_inter, hidden};
        dn[1] = GemvGroup{nullptr, nullptr, nullptr, nullptr, 0, 0, nullptr, 1, m, 1, hidden, shared_inter};
        ng = 2;
    }
    const LayerPlan L = plan_of(gu, dn, ng, kOne);  // one-row down items: the larger cap
    if (L.cap_a + L.cap_b > (1 << 26)) return 0;
    // head, start tags, result words, then the flags
    return kSyncHead + kLayerMaxCtas + (size_t)result_words(m, top_k, hidden, inter, shared_inter) +
           (size_t)L.cap_a + (size_t)L.cap_b;
}

bool layer_one_round(int m, int top_k, int hidden, int inter, int shared_inter) {
    if (m < 1 || top_k < 1) return false;
    GemvGroup gu[2] = {}, dn[2] = {};
    gu[0] = GemvGroup{nullptr, nullptr, nullptr, nullptr, 0, 0, nullptr, 1, m, top_k, inter, hidden};
    dn[0] = GemvGroup{nullptr, nullptr, nullptr, nullptr, 0, 0, nullptr, 1, m, top_k, hidden, inter};
    int ng = 1;
    if (shared_inter > 0) {
        gu[1] = GemvGroup{nullptr, nullptr, nullptr, nullptr, 0, 0, nullptr, 1, m, 1, shared_inter, hidden};
        dn[1] = GemvGroup{nullptr, nullptr, nullptr, nullptr, 0, 0, nullptr, 1, m, 1, hidden, shared_inter};
        ng = 2;
    }
    const int64_t resident = (int64_t)num_sms() * 3;
    const LayerPlan L = plan_of(gu, dn, ng, kPair);
    return L.cap_a <= resident && L.cap_b <= resident;
}

namespace {

// A planned launch: the kernel, its block size, shared memory and grid.
struct LaunchPlan {
    void (*kern)(LayerParams);
    int threads;
    size_t smem;
    int64_t grid;
    bool wide;
};

// Plan a single-launch layer for these groups: P's shapes, shared-memory layout, caps and shape
// word (not its pointers into the workspace, the combine or the error flag) and the kernel the
// launch takes. Sets the kernels' shared-memory attributes on the current device on first use.
// cudaErrorNotSupported where the single launch does not apply.
cudaError_t plan_layer(const GemvGroup* gu, const GemvGroup* dn, int n_groups, bool shared_term, LayerParams& P,
                       LaunchPlan& LP) {
    if (n_groups < 1 || n_groups > kMaxGroups) return cudaErrorNotSupported;
    int64_t max_pairs = 0;
    for (int gi = 0; gi < n_groups; ++gi) max_pairs = std::max<int64_t>(max_pairs, (int64_t)gu[gi].m * gu[gi].top_k);
    if (max_pairs > kLayerMaxPairs) return cudaErrorNotSupported;
    // tokens per item: 1 when every bucket holds about one pair (decode with distinct experts),
    // else up to kTB -- as in the two-launch layer, so both compute alike
    int kmax = 0, tb = 1;
    for (int gi = 0; gi < n_groups; ++gi) {
        kmax = std::max(kmax, std::max(gu[gi].k, dn[gi].k));
        if ((int64_t)gu[gi].m * gu[gi].top_k > gu[gi].num_experts) tb = kTB;
    }
    const int64_t per_tok = (int64_t)(kmax / 64) * kPairBytes + (int64_t)(kmax / 32) * 8;
    while (tb > 1 && per_tok * tb > 150 * 1024) tb >>= 1;
    if (tb != 1 && tb != kTB) tb = 1;
    // paired down items when one-row items would outnumber the CTAs the SMs hold; always for the
    // wide kernel (one token per item, the gate|up tiles, the down tile and the activation row
    // in shared memory, one item of each half per CTA; Q4K_LAYER_WIDE=0: never)
    const int64_t resident = (int64_t)num_sms() * 3;
    const char* wide_env = getenv("Q4K_LAYER_WIDE");
    bool wide_ok = (wide_env == nullptr || atoi(wide_env) != 0) && tb == 1;
    for (int gi = 0; wide_ok && gi < n_groups; ++gi) {
        const int lga = lg_split_for(gu[gi].k), lgb = lg_split_for(dn[0].k);
        const int64_t nb01a = (int64_t)(gu[gi].k / kQK) * kBlockBytes, nb01b = (int64_t)(dn[gi].k / kQK) * kBlockBytes;
        wide_ok = 2 * item_tile_rows(lga, kFused) * nb01a <= 48 * 1024 && item_tile_rows(lgb, kPair) * nb01b <= 48 * 1024 &&
                  (int64_t)gu[gi].k * 4 <= 32 * 1024;
    }
    if (wide_ok) {
        const LayerPlan Lw = plan_of(gu, dn, n_groups, kPair);
        wide_ok = Lw.cap_a <= resident && Lw.cap_b <= resident;
    }
    const int kb = wide_ok || plan_of(gu, dn, n_groups, kOne).cap_b > resident ? kPair : kOne;
    const LayerPlan L = plan_of(gu, dn, n_groups, kb);
    const int m = gu[0].m, top_k = gu[0].top_k, hidden = dn[0].n, inter = gu[0].n;
    const int shared_inter = n_groups > 1 ? gu[1].n : 0;
    P = LayerParams{};
    P.n_groups = n_groups;
    for (int gi = 0; gi < n_groups; ++gi) {
        P.a[gi] = group_dev(gu[gi], L.lg_a[gi], kFused);
        P.b[gi] = group_dev(dn[gi], L.lg_b[gi], kb);
    }
    P.x_off = 0;
    P.meta_off = (int)(((int64_t)(kmax / 64) * kPairBytes * tb + 15) & ~int64_t(15));
    const size_t base_smem = (size_t)P.meta_off + (size_t)(kmax / 32) * 8 * tb;
    // Shared memory beyond the staged planes, each part used where it fits:
    //  - the gate|up item's weight tiles (gate, up) when both fit 48 KB (use_atile);
    //  - the first down tile of the CTA when it fits 48 KB (use_slot);
    //  - the gate|up activation rows when they fit 32 KB (use_xcopy), in the down tile's space
    //    when there is one (its copy then starts after the last gate|up staging).
    int64_t slot_bytes = 0, atile_bytes = 0;
    int ka = 0;
    for (int gi = 0; gi < n_groups; ++gi) {
        slot_bytes = std::max<int64_t>(slot_bytes, (int64_t)item_tile_rows(L.lg_b[gi], kb) * P.b[gi].nb01);
        atile_bytes = std::max<int64_t>(atile_bytes, (int64_t)item_tile_rows(L.lg_a[gi], kFused) * P.a[gi].nb01);
        ka = std::max(ka, gu[gi].k);
    }
    const int64_t raw_bytes = (int64_t)ka * 4 * tb;
    P.use_slot = slot_bytes <= 48 * 1024 ? 1 : 0;
    P.use_xcopy = raw_bytes <= 32 * 1024 ? 1 : 0;
    P.slot_shares_raw = P.use_slot && P.use_xcopy ? 1 : 0;
    P.atile_bytes = (int)atile_bytes;
    auto layout = [&](bool atile) {
        size_t off = (base_smem + 127) & ~size_t(127);
        P.use_atile = atile ? 1 : 0;
        P.atile_off = (int)off;
        if (atile) off += (size_t)(2 * atile_bytes);
        off = (off + 127) & ~size_t(127);
        P.slot_off = P.raw_off = (int)off;
        const int64_t region = std::max<int64_t>(P.use_slot ? slot_bytes : 0, P.use_xcopy ? raw_bytes : 0);
        return off + (size_t)region;
    };
    size_t smem = layout(2 * atile_bytes <= 48 * 1024);
    P.cap_a = (int)L.cap_a;
    P.cap_b = (int)L.cap_b;
    // the shapes that decide which result words a launch writes and reads, and where
    uint64_t shape = host_mix64(0x51A9E0F1A7E2ull);
    for (const int64_t v : {(int64_t)m, (int64_t)top_k, (int64_t)hidden, (int64_t)inter, (int64_t)shared_inter,
                            (int64_t)n_groups, (int64_t)kb, (int64_t)tb, (int64_t)shared_term})
        shape = host_mix64(shape ^ (uint64_t)v);
    P.shape = shape;

    void (*kern)(LayerParams) = tb == 1 ? (kb == kPair ? layer_kernel<1, kPair> : layer_kernel<1, kOne>)
                                        : (kb == kPair ? layer_kernel<kTB, kPair> : layer_kernel<kTB, kOne>);
    bool wide = wide_ok && P.use_atile && P.use_slot && P.use_xcopy;
    int threads = kThreads;
    if (wide) {
        kern = layer_wide_kernel;
        threads = kWideThreads;
    }
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    // the shared-memory attributes are set once per device and kernel
    auto prepare = [&](void (*k)(LayerParams), int kind) -> cudaError_t {
        if (g_layer_attr_set[kind][dev]) return cudaSuccess;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
        if (e == cudaSuccess) g_layer_attr_set[kind][dev] = true;
        return e;
    };
    err = prepare(kern, wide ? 4 : (tb == 1 ? 0 : 1) + (kb == kPair ? 2 : 0));
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (err != cudaSuccess) return err;
    if (wide && (int64_t)per_sm * num_sms() < std::max(L.cap_a, L.cap_b)) {
        // not one item of each half per CTA: the four-warp kernel
        kern = layer_kernel<1, kPair>;
        threads = kThreads;
        wide = false;
        err = prepare(kern, 2);
        if (err != cudaSuccess) return err;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
        if (err != cudaSuccess) return err;
    }
    if (P.use_atile && per_sm < 3 && threads == kThreads) {  // the weight tiles must not cost residency
        smem = layout(false);
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
        if (err != cudaSuccess) return err;
    }
    if (smem > 200 * 1024) return cudaErrorNotSupported;
    if (per_sm < 1) return cudaErrorNotSupported;
    // every CTA must be resident at once (the waits): at most what the SMs hold
    int64_t grid = (int64_t)num_sms() * per_sm;
    grid = std::min<int64_t>(grid, kLayerMaxCtas);
    grid = std::min<int64_t>(grid, std::max<int64_t>(std::max(L.cap_a, L.cap_b), 1));
    LP.kern = kern;
    LP.threads = threads;
    LP.smem = smem;
    LP.grid = grid;
    LP.wide = wide;
    return cudaSuccess;
}

}  // namespace

int layer_kernel_kind(int m, int top_k, int num_experts, int hidden, int inter, int shared_inter) {
    if (layer_sync_words(m, top_k, hidden, inter, shared_inter) == 0) return 0;
    GemvGroup gu[2] = {}, dn[2] = {};
    gu[0] = GemvGroup{nullptr, nullptr, nullptr, nullptr, 0, 0, nullptr, num_experts, m, top_k, inter, hidden};
    dn[0] = GemvGroup{nullptr, nullptr, nullptr, nullptr, 0, 0, nullptr, num_experts, m, top_k, hidden, inter};
    int ng = 1;
    if (shared_inter > 0) {
        gu[1] = GemvGroup{nullptr, nullptr, nullptr, nullptr, 0, 0, nullptr, 1, m, 1, shared_inter, hidden};
        dn[1] = GemvGroup{nullptr, nullptr, nullptr, nullptr, 0, 0, nullptr, 1, m, 1, hidden, shared_inter};
        ng = 2;
    }
    LayerParams P{};
    LaunchPlan LP{};
    const cudaError_t e = plan_layer(gu, dn, ng, shared_inter > 0, P, LP);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return e == cudaErrorNotSupported ? 0 : 1;  // (no device to ask: the kernel is unknown)
    }
    return LP.wide ? 2 : 1;
}

cudaError_t launch_layer_persistent(const GemvGroup* gu, const GemvGroup* dn, int n_groups, const CombineSpec& cb,
                                    uint64_t* sync, size_t sync_words, int* err_flag, cudaStream_t stream) {
    LayerParams P{};
    LaunchPlan LP{};
    cudaError_t err = plan_layer(gu, dn, n_groups, cb.shared_mode != Q4K_SHARED_NONE, P, LP);
    if (err != cudaSuccess) return err;
    const int m = gu[0].m, top_k = gu[0].top_k, hidden = dn[0].n, inter = gu[0].n;
    const int shared_inter = n_groups > 1 ? gu[1].n : 0;
    const int64_t n_results = result_words(m, top_k, hidden, inter, shared_inter);
    if (sync == nullptr || sync_words < kSyncHead + kLayerMaxCtas + (size_t)(n_results + P.cap_a + P.cap_b))
        return cudaErrorNotSupported;
    P.cb = cb;
    P.gen = sync;
    P.cta_tag = sync + kSyncHead;
    uint64_t* words = P.cta_tag + kLayerMaxCtas;  // 16-byte aligned (even word offset)
    P.act64[0] = words;
    P.act64[1] = P.act64[0] + (int64_t)m * top_k * inter;
    P.out64[0] = P.act64[1] + (int64_t)m * shared_inter;
    P.out64[1] = n_groups > 1 ? P.out64[0] + (int64_t)m * top_k * hidden : nullptr;
    P.flag_a = words + n_results;
    P.flag_b = P.flag_a + P.cap_a;
    P.err_flag = err_flag;
    P.wait_ns = wait_limit_ns();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)LP.grid);
    cfg.blockDim = dim3(LP.threads);
    cfg.dynamicSmemBytes = LP.smem;
    cfg.stream = stream;
    // A cooperative launch: the driver starts the grid only with every CTA resident at once,
    // which the waits between CTAs need (the grid is at most what the SMs hold). Not a
    // programmatic dependent: its CTAs could then be placed beside the previous kernel's last
    // CTAs on SMs configured for a smaller shared-memory share.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, LP.kern, P);
    if (e == cudaErrorCooperativeLaunchTooLarge) {
        // fewer CTAs fit than the occupancy query said (e.g. SMs held by another client): the
        // caller runs the two-launch layer, which gives the same bits
        cudaGetLastError();
        return cudaErrorNotSupported;
    }
    return e;
}

}  // namespace q4k

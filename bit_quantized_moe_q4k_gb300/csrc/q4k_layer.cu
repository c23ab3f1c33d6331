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
// starts its down item as soon as the gate|up items of that bucket chunk have landed; and the
// last down item of a row tile combines that tile.
//
// Hand-off between CTAs without zero-initialised state: every item, when its rows are
// written, stores a 64-bit tag into its own flag word; a consumer waits until the flags it
// needs hold the tag. The tag of a launch is next_tag(generation word); the generation word is
// advanced to the tag at the end of the launch (by CTA 0, once every CTA has recorded that it
// read the old value), so stale flags of earlier launches never match and nothing needs
// clearing -- also not on the first call on fresh memory. The combine's per-tile counters come
// in two sets used by alternate launches: a launch zeroes the set the next one uses and stamps
// its header with that launch's tag; a launch whose set is not stamped so (the first on this
// memory, a call of another shape) polls the down items' flags instead. Every wait is bounded
// in time; one that gives up raises Q4K_ERR_TIMEOUT. The waits need every CTA of the grid
// resident at once: the grid is capped at what the SMs hold, it is an ordinary launch (it
// starts on SMs the previous kernel has left), and CTAs never wait on a CTA that
// is itself waiting (gate|up items never wait; down items wait only on gate|up items; the
// combine waits only on down items).
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
    uint64_t* gen;            // generation word
    uint64_t* cnt_hdr;        // [2] tag for which counter set s is zero (set by the previous launch)
    unsigned* cnt;            // [2][nt_max] per combine tile: down items done
    int nt_max;
    uint64_t* cta_tag;        // [kLayerMaxCtas] tag each CTA read
    uint64_t* flag_a;         // [cap_a] one per gate|up item
    uint64_t* flag_b;         // [cap_b] one per down item
    int cap_a, cap_b;
    int* err_flag;
    uint64_t wait_ns;         // limit of every wait
};

// A counter set's header: the tag of the launch it was prepared for, bound to the sets' size
// (which moves with hidden), so a call of another shape never takes words laid out for
// another as its zeroed counters.
__device__ __forceinline__ uint64_t set_stamp(uint64_t tag, int nt_max) {
    return tag ^ ((uint64_t)(unsigned)nt_max * 0x9E3779B97F4A7C15ull);
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Block-wide: wait until flags[index(j)] == tag for all j < n. Each thread owns j = tid,
// tid + kThreads, ...; it re-reads only those it has not yet seen set (up to 8 loads per
// round). The reads are acquire loads, so every flag was acquired before the barrier that
// ends the wait, and what any thread of the block does after it is ordered after the
// flags' releases. True when all are set; false once the wait has run for limit_ns or
// kLayerMaxPolls rounds. Uniform over the block.
template <class Index>
__device__ __forceinline__ bool wait_tags(const uint64_t* flags, int n, uint64_t tag, uint64_t limit_ns, Index index) {
    int j = threadIdx.x;
    const uint64_t t0 = sm100::global_timer_ns();
    for (uint32_t round = 0;; ++round) {
        uint64_t v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int jj = j + u * kThreads;
            v[u] = jj < n ? ld_acquire_u64(flags + index(jj)) : tag;
        }
        int seen = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (v[u] != tag) break;
            ++seen;
        }
        j += seen * kThreads;
        if (__syncthreads_and(j >= n)) return true;
        const bool late = round >= kLayerMaxPolls || sm100::global_timer_ns() - t0 > limit_ns;
        if (__syncthreads_or(late)) return false;
        __nanosleep(32);
    }
}

// Publish an item: its rows were written by this block's threads (the caller synchronised
// the block); one thread stores the tag with release order at GPU scope, which makes those
// rows visible first. It is a thread of the last warp: warp 0 locates the next item.
__device__ __forceinline__ void publish(uint64_t* flag, uint64_t tag) {
    if (threadIdx.x == kThreads - 32) asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(flag), "l"(tag) : "memory");
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
    __shared__ int s_set, s_cnt_ok, s_per_tile, s_last;  // counter set, it is valid, items per tile
    __shared__ __align__(8) uint64_t s_bar;  // the down tile's copy into shared memory
    __shared__ __align__(8) uint64_t s_xbar; // a gate|up item's activation rows' copy
    __shared__ __align__(8) uint64_t s_abar; // a gate|up item's weight tiles' copy
    __shared__ int s_never;                  // (bounded waits take an abort word; never set)

    // (launched as an ordinary launch, so earlier kernels of the stream are complete and the
    // wait returns at once); the next kernel may launch early: it can only take space left
    // over once every CTA of this grid has started, which the trigger implies
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // the generation word's load overlaps the bucketing (its value is used after it)
    const uint64_t gen = threadIdx.x == 0 ? ld_relaxed_u64(P.gen) : 0;
    const uint64_t hdr0 = threadIdx.x == 0 ? ld_relaxed_u64(P.cnt_hdr) : 0;
    const uint64_t hdr1 = threadIdx.x == 0 ? ld_relaxed_u64(P.cnt_hdr + 1) : 0;
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
            // the previous launch zeroed this launch's counter set and stamped it with this tag
            // (else: the first call on this memory, or a call of another shape) -> poll instead
            s_set = (int)(tag & 1ull);
            s_cnt_ok = ((tag & 1ull) ? hdr1 : hdr0) == set_stamp(tag, P.nt_max) && P.b[0].tiles <= P.nt_max;
            st_relaxed_u64(P.cta_tag + blockIdx.x, tag);  // this CTA has read the generation
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {  // down items per combine tile: every chunk has one on each tile
        int per_tile = 0;
        for (int gi = 0; gi < P.n_groups; ++gi) per_tile += (s_items[1][gi + 1] - s_items[1][gi]) / P.b[gi].tiles;
        s_per_tile = per_tile;  // read after the barriers of the items below
    }
    const uint64_t tag = s_tag;
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
    if (slot_item && (a0 == a1 || !P.slot_shares_raw)) issue_slot();
    // the bulk copies of the gate|up items: bit 0 / 1 = a copy on s_xbar / s_abar not yet waited
    // for (drained before the CTA leaves, also after a wait gave up), bit 2 / 3 = the parity of
    // the phase that barrier completes next
    uint32_t cps = 0;

    int staged = -1;  // (half, group, rank, chunk) of the staged activation rows
    // ---- gate|up + SwiGLU items: activation rows and (use_atile) the weight tiles of both slabs
    // arrive by bulk copy, which keeps them out of the SM's load queue
    auto gate_up_item = [&](auto from_smem, int item, const GroupDev& G, int e, int tile, int nt, int key) -> bool {
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
        item_compute<kFused, TB>(G, IL, s_pairs, nt, xs, meta, lane);
        __syncthreads();
        publish(P.flag_a + item, tag);
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
        ok = P.use_atile ? gate_up_item(std::true_type{}, item, G, e, tile, nt, key)
                         : gate_up_item(std::false_type{}, item, G, e, tile, nt, key);
    }

    // ---- down items: each waits for the gate|up items of its chunk (all their row tiles)
    // (the first from its shared-memory copy when there is one)
    const bool shared = P.cb.shared_mode != Q4K_SHARED_NONE && P.n_groups > 1;
    const int tr = item_tile_rows(P.b[0].lg_split, KB);
    auto combine_tile = [&](int t) {
        const GroupDev& R = P.b[0];
        combine_span(P.cb, R.out, R.ids, R.num_experts, R.n_pairs, R.top_k, R.n, shared ? P.b[1].out : nullptr, t * tr,
                     min(R.n, (t + 1) * tr), threadIdx.x, kThreads);
    };
    auto down_item = [&](auto& IL, int item, const GroupDev& G, int gi, int r, int nt, int chunk, int tile) -> bool {
        const int key = ((gi * 32 + r) * 32 + chunk) * 2 + 1;
        if (key != staged) {
            const int first = s_items[0][gi] + s_fast[0][gi].start[r] + chunk * P.a[gi].tiles;
            if (!wait_tags(P.flag_a, P.a[gi].tiles, tag, P.wait_ns, [first](int j) { return first + j; })) return false;
            stage_rows<true>(G, s_pairs, nt, xs, meta);
            staged = key;
        }
        __syncthreads();
        item_compute<KB, TB>(G, IL, s_pairs, nt, xs, meta, lane);
        __syncthreads();
        if (s_cnt_ok) {  // the last down item of the tile combines it
            // the counter's release makes this item's rows visible (no flag: only the combine
            // without counters reads the down flags); its acquire, passed on to the block by the
            // barrier, orders the reads of the other items' rows (from L2) after their releases
            if (threadIdx.x == kThreads - 32)
                s_last = atom_add_acq_rel(P.cnt + s_set * P.nt_max + tile, 1u) + 1u == (unsigned)s_per_tile;
            __syncthreads();
            if (s_last) combine_tile(tile);
        } else {
            publish(P.flag_b + item, tag);
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
    // a copy still in flight must land before the CTA leaves (after an abort)
    if (slot_issued && !slot_waited) sm100::mbar_wait(&s_bar, 0, &s_never);
    if (cps & 1u) sm100::mbar_wait(&s_xbar, (cps >> 2) & 1u, &s_never);
    if (cps & 2u) sm100::mbar_wait(&s_abar, (cps >> 3) & 1u, &s_never);

    // ---- combine (without valid counters): row tiles of the routed down group, each by a
    // designated CTA after its down items' flags
    if (threadIdx.x == 0 && !s_cnt_ok) {  // down items of tile 0 of every chunk (the combine's wait list)
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
    __syncthreads();
    const int n_tiles = P.b[0].tiles;
    const int t0 = (int)(cta * n_tiles / grid), t1 = (int)((cta + 1) * n_tiles / grid);
    for (int t = t0; ok && !s_cnt_ok && t < t1; ++t) {
        ok = wait_tags(P.flag_b, s_n_chunks, tag, P.wait_ns, [t](int j) { return s_chunk_b[j] + t; });
        if (!ok) break;
        combine_tile(t);
    }

    if (threadIdx.x == 0) {
        if (!fits) raise_flag(P.err_flag, Q4K_ERR_LIMIT);
        else if (!ok) raise_flag(P.err_flag, Q4K_ERR_TIMEOUT);
        if (blockIdx.x == 0)
            for (int half = 0; half < 2; ++half)
                for (int gi = 0; gi < P.n_groups; ++gi)
                    if (s_bad[half][gi]) raise_flag(P.err_flag, Q4K_ERR_EXPERT_ID);
    }
    // ---- advance the generation once every CTA has read it, and prepare the next launch's
    // counter set (the one this launch does not use): zero it, then stamp it with its tag
    if (blockIdx.x == 0) {
        const bool all = wait_tags(P.cta_tag, (int)gridDim.x, tag, P.wait_ns, [](int j) { return j; });
        if (all) {
            unsigned* next = P.cnt + (s_set ^ 1) * P.nt_max;
            for (int i = threadIdx.x; i < P.nt_max; i += kThreads) next[i] = 0u;
            __syncthreads();
        }
        if (threadIdx.x == 0) {
            if (all) {
                __threadfence();
                st_relaxed_u64(P.cnt_hdr + (s_set ^ 1), set_stamp(next_tag(tag), P.nt_max));
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

bool g_layer_attr_set[4][64] = {};

// Combine tiles of the smallest row tile (8 rows), whatever the down items' kind.
int combine_tiles_max(int hidden) { return (hidden + 7) / 8; }

// Words before the start tags: the generation word, two counter-set headers and two sets of
// u32 counters. They depend on hidden only, so they stay in place when m changes.
size_t sync_head_words(int hidden) { return 3 + (size_t)(combine_tiles_max(hidden) + 1) / 2 * 2; }

}  // namespace

size_t layer_sync_head_words(int hidden) { return sync_head_words(hidden); }

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
    return sync_head_words(hidden) + kLayerMaxCtas + (size_t)L.cap_a + (size_t)L.cap_b;
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

cudaError_t launch_layer_persistent(const GemvGroup* gu, const GemvGroup* dn, int n_groups, const CombineSpec& cb,
                                    uint64_t* sync, size_t sync_words, int* err_flag, cudaStream_t stream) {
    if (n_groups < 1 || n_groups > kMaxGroups) return cudaErrorNotSupported;
    int64_t max_pairs = 0;
    for (int gi = 0; gi < n_groups; ++gi) max_pairs = std::max<int64_t>(max_pairs, (int64_t)gu[gi].m * gu[gi].top_k);
    if (max_pairs > kLayerMaxPairs) return cudaErrorNotSupported;
    // paired down items when one-row items would outnumber the CTAs the SMs hold
    const int64_t resident = (int64_t)num_sms() * 3;
    const int kb = plan_of(gu, dn, n_groups, kOne).cap_b > resident ? kPair : kOne;
    const LayerPlan L = plan_of(gu, dn, n_groups, kb);
    const size_t head = sync_head_words(dn[0].n);
    if (sync == nullptr || sync_words < head + kLayerMaxCtas + (size_t)(L.cap_a + L.cap_b)) return cudaErrorNotSupported;
    LayerParams P{};
    P.n_groups = n_groups;
    int kmax = 0, tb = 1;
    for (int gi = 0; gi < n_groups; ++gi) {
        P.a[gi] = group_dev(gu[gi], L.lg_a[gi], kFused);
        P.b[gi] = group_dev(dn[gi], L.lg_b[gi], kb);
        kmax = std::max(kmax, std::max(gu[gi].k, dn[gi].k));
        // tokens per item: 1 when every bucket holds about one pair (decode with distinct
        // experts), else up to kTB -- as in the two-launch layer, so both compute alike
        if ((int64_t)gu[gi].m * gu[gi].top_k > gu[gi].num_experts) tb = kTB;
    }
    const int64_t per_tok = (int64_t)(kmax / 64) * kPairBytes + (int64_t)(kmax / 32) * 8;
    while (tb > 1 && per_tok * tb > 150 * 1024) tb >>= 1;
    if (tb != 1 && tb != kTB) tb = 1;
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
    P.cb = cb;
    P.gen = sync;
    P.cnt_hdr = sync + 1;
    P.cnt = reinterpret_cast<unsigned*>(sync + 3);
    P.nt_max = combine_tiles_max(dn[0].n);
    P.cta_tag = sync + head;
    P.flag_a = P.cta_tag + kLayerMaxCtas;
    P.flag_b = P.flag_a + L.cap_a;
    P.cap_a = (int)L.cap_a;
    P.cap_b = (int)L.cap_b;
    P.err_flag = err_flag;
    P.wait_ns = wait_limit_ns();

    void (*kern)(LayerParams) = tb == 1 ? (kb == kPair ? layer_kernel<1, kPair> : layer_kernel<1, kOne>)
                                        : (kb == kPair ? layer_kernel<kTB, kPair> : layer_kernel<kTB, kOne>);
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const int kind = (tb == 1 ? 0 : 1) + (kb == kPair ? 2 : 0);
    if (!g_layer_attr_set[kind][dev]) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
        if (err != cudaSuccess) return err;
        g_layer_attr_set[kind][dev] = true;
    }
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (err != cudaSuccess) return err;
    if (P.use_atile && per_sm < 3) {  // the weight tiles must not cost residency
        smem = layout(false);
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
        if (err != cudaSuccess) return err;
    }
    if (smem > 200 * 1024) return cudaErrorNotSupported;
    if (per_sm < 1) return cudaErrorNotSupported;
    // every CTA must be resident at once (the waits): at most what the SMs hold
    int64_t grid = (int64_t)num_sms() * per_sm;
    grid = std::min<int64_t>(grid, kLayerMaxCtas);
    grid = std::min<int64_t>(grid, std::max<int64_t>(std::max(L.cap_a, L.cap_b), 1));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    // an ordinary launch: it starts on idle SMs. As a programmatic dependent its CTAs could be
    // placed beside the previous kernel's last CTAs on SMs configured for a smaller shared-memory
    // share, which then hold fewer of them than the grid needs resident at once.
    return cudaLaunchKernelEx(&cfg, kern, P);
}

}  // namespace q4k

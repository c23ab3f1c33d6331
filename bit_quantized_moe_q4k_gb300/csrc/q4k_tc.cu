// q4k_tc.cu -- tensor-core grouped GEMM (tcgen05) for experts whose bucket holds many tokens.
//
// Same result as the id-GEMV for those experts (ferrum-kernels q4_k_moe_id_gemv_batched.rs:
// out[p, r] = W_{ids[p]}[r, :] . x_p; with two slabs, silu(gate) * up), computed as a dense
// contraction per (expert, 128-row tile, chunk of 32 tokens of the expert's bucket):
//   D[r, t] = sum_k A[r, k] * B[t, k]
// with A in tensor memory and B in shared memory (tcgen05.mma, kind::f16, fp32 accumulation).
// When the batch averages at least two chunks per expert, a work item takes two chunks of one
// row tile, and each block's A serves the MMAs of both.
//
// Exactness of the operands. Q4_K gives per 32-weight sub-block j of a 256-weight block
//   sum_k w_k x_k = d * sum_j sc_j sum_{k in j} q_k x_k  -  dmin * sum_j m_j sum_{k in j} x_k.
// A holds the integers sc_j * q_k (<= 945, exact in fp16). x is split into two fp16 parts,
// x = hi + lo with hi = fp16(x), lo = fp16(x - hi), and both are multiplied by the same A
// (the 32 tokens' hi rows and their lo rows side by side in one N = 64 operand, so one MMA
// per k step forms both; the epilogue adds the two halves), so the product carries x to ~2^-22
// instead of fp16's 2^-11 (which alone put FFN outputs at the edge of the 1e-3 acceptance).
// A second, 16-deep MMA per block computes sum_j m_j * sx_j
// with sx_j = sum_{k in j} x_k split into two fp16 halves (hi + lo), i.e. to ~2^-22. The
// per-block factors d and dmin are applied in fp32 by the epilogue, which reads each block's
// two partial accumulators from tensor memory (double-buffered, so the next block's MMAs
// run meanwhile).
//
// Roles (10 warps): warps 0-7 dequantize and run the epilogue, two warps per TMEM lane
// quarter (thread = weight row = TMEM lane): warp w < 4 takes the 64-weight groups 0-1 of
// the block and tokens 0-15 of the epilogue, warp w + 4 groups 2-3 and tokens 16-31; warp 8
// issues the bulk copies (raw Q4_K rows of the tile, and the prepared B image of the
// block); warp 9 owns tensor memory and issues the MMAs. Raw rows -> registers -> A:
// dequantization writes each row's 256 weights as 128 fp16-pair columns with tcgen05.st
// (the A operand never touches shared memory). Pipelines on mbarriers; every wait is
// bounded and an abort flag lets all roles leave together.
//
// The B image of a (chunk, block) is built once by tc_prep_kernel in the workspace: the 32
// tokens' x in fp16, in the k order of the A columns, already laid out as the 128-byte
// swizzled K-major smem tile, plus the sx hi/lo row of the min-term MMA.
#include <cuda.h>
#include <cuda_fp16.h>

#include "q4k_bucket.cuh"
#include "q4k_internal.cuh"
#include "q4k_sm100.cuh"
#include "q4k_sync.cuh"

namespace q4k {
using namespace sm100;

constexpr int kTcThreads = 320;
constexpr int kTcWorkers = 256;               // dequant + epilogue threads (warps 0-7)
constexpr int kTcCopyWarp = 8, kTcMmaWarp = 9;
constexpr int kTcRows = 128;                  // M (TMEM lanes)
constexpr int kTcTok = 32;                    // N (tokens per chunk)
// One block's B image: 4 K-panels of 64 rows x 128 B, rows 0-31 the 32 tokens' x rounded to
// fp16 and rows 32-63 their residuals x - fp16(x); then the min-term operand.
constexpr int kPanel = 2 * kTcTok * 128;       // one K-panel: 64 rows x 128 B
constexpr int kImgLoRow = kTcTok;              // first residual row of a panel
constexpr int kImgB2 = kTcTok * 128;           // min-term operand [32 tokens x 128 B]
constexpr int kImgMin = 4 * kPanel;            // offset of the min-term operand
constexpr int kImgBlock = 4 * kPanel + kImgB2; // bytes of one block's B image
constexpr int kRawStage = kTcRows * kBlockBytes;
constexpr int kNRaw = 4;   // raw Q4_K row stages in shared memory (copies run this far ahead)
constexpr int kNImg = 3;   // activation image stages in shared memory
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns: A stages (128 each), min-term A stages (16 each), D1 stages (64
// each: 32 tokens' fp16 part, then their residual part), D2 stages (32 each: min term)
constexpr uint32_t kColA = 0, kColA2 = 256, kColD1 = 288, kColD2 = 416;

struct TcGroup {
    const uint8_t* w;    // slab [E][n][k/256] blocks
    const uint8_t* w2;   // second slab (up) for silu(gate)*up, or null
    const int32_t* ids;  // or null: every pair uses expert 0
    const float* a;
    int64_t outer, inner;
    float* out;
    uint8_t* img;        // B images [max_chunks][nb][kImgBlock]
    int64_t nb01, nb02;
    int num_experts, n_pairs, top_k, n, k, tiles;
};

struct TcParams {
    CUtensorMap tmap[2][2];  // [group][slab]: the slab as a 2-D byte tensor [E*n rows, nb01 bytes]
    TcGroup g[2];
    int n_groups;
    int tc_min;       // experts with at least this many pairs take the tensor-core path
    int hist_off[2];  // int offsets of each group's tables in shared memory
    int tab_off;      // byte offset of the tables
    int* err_flag;
    uint64_t wait_ns; // limit of the pipeline waits (the drains after an abort keep their own)
};

// Per-CTA bucketing for the tensor-core path: cnt[e] pairs per expert and start[e] = first
// chunk id of expert e (exclusive prefix of ceil(cnt/32) over experts with cnt >= tc_min).
// Returns the number of chunks.
__device__ __forceinline__ int tc_chunks(const TcGroup& G, int tc_min, int* cnt, int* start, int* s_warp,
                                         int* s_bad) {
    if (G.ids) {
        block_histogram(G.ids, G.n_pairs, G.num_experts, cnt, s_bad);
    } else {
        if (threadIdx.x == 0) { cnt[0] = G.n_pairs; *s_bad = 0; }
        __syncthreads();
    }
    for (int e = threadIdx.x; e < G.num_experts; e += blockDim.x)
        start[e] = cnt[e] >= tc_min ? (cnt[e] + kTcTok - 1) / kTcTok : 0;
    __syncthreads();
    return block_exclusive_scan(start, G.num_experts, s_warp);
}

// chunk id q -> expert (last e with start[e] <= q; it has chunks)
__device__ __forceinline__ int tc_expert_of(const int* start, int num_experts, int q) {
    int lo = 0, hi = num_experts - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (start[mid] <= q) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ void tc_gather(const TcGroup& G, int e, int chunk, int nt, int* s_pairs) {
    const int lane = threadIdx.x & 31;
    if (G.ids) {
        warp_gather_bucket(G.ids, G.n_pairs, e, chunk * kTcTok, nt, s_pairs);
    } else if (lane < nt) {
        s_pairs[lane] = chunk * kTcTok + lane;
    }
}

// ------------------------------------------------------------------------------------------
// B images: grid (max chunks, groups, block slices), 128 threads. CTA z builds the blocks
// b = z, z + gridDim.z, ... of its chunk; warp w builds tokens t = w, w+4, ...
__global__ void __launch_bounds__(128)
tc_prep_kernel(const __grid_constant__ TcParams P) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int s_warp[33];
    __shared__ int s_bad;
    __shared__ int s_pairs[kTcTok];
    __shared__ int s_info[3];
    const int gi = blockIdx.y;
    const TcGroup& G = P.g[gi];
    int* cnt = reinterpret_cast<int*>(smem);
    int* start = cnt + G.num_experts;
    // the ids and activations may be the previous kernel's output
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int total = tc_chunks(G, P.tc_min, cnt, start, s_warp, &s_bad);
    const int q = blockIdx.x;
    if (q >= total) return;
    if (threadIdx.x == 0) {
        const int e = tc_expert_of(start, G.num_experts, q);
        s_info[0] = e;
        s_info[1] = q - start[e];
        s_info[2] = min(kTcTok, cnt[e] - (q - start[e]) * kTcTok);
    }
    __syncthreads();
    const int e = s_info[0], chunk = s_info[1], nt = s_info[2];
    if (threadIdx.x < 32) tc_gather(G, e, chunk, nt, s_pairs);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c4 = lane >> 3, ip = lane & 7;
    const int nb = G.k / kQK;
    uint8_t* img0 = G.img + (int64_t)q * nb * kImgBlock;
    for (int b = blockIdx.z; b < nb; b += gridDim.z) {
        uint8_t* img = img0 + (int64_t)b * kImgBlock;
        for (int t = warp; t < kTcTok; t += 4) {
            float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
            if (t < nt) {
                const int p = s_pairs[t];
                const float* row = G.a + (int64_t)(p / G.top_k) * G.outer + (int64_t)(p % G.top_k) * G.inner +
                                   (int64_t)b * kQK + 64 * c4 + 4 * ip;
                lo = *reinterpret_cast<const float4*>(row);
                hi = *reinterpret_cast<const float4*>(row + 32);
            }
            // k order of the A columns: elements 4i'+{0,2,1,3} then 32+4i'+{0,2,1,3} of group c4
            const float xv[8] = {lo.x, lo.z, lo.y, lo.w, hi.x, hi.z, hi.y, hi.w};
            uint32_t hw8[4], lw8[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __half a = __float2half_rn(xv[2 * i]), b = __float2half_rn(xv[2 * i + 1]);
                const __half ra = __float2half_rn(xv[2 * i] - __half2float(a));
                const __half rb = __float2half_rn(xv[2 * i + 1] - __half2float(b));
                hw8[i] = (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
                lw8[i] = (uint32_t)__half_as_ushort(ra) | ((uint32_t)__half_as_ushort(rb) << 16);
            }
            // 128-byte swizzle: 16-byte chunk ip of row rr sits at chunk ip ^ (rr & 7); rows t and
            // 32 + t share the pattern
            const int off = c4 * kPanel + t * 128 + ((ip ^ (t & 7)) << 4);
            *reinterpret_cast<uint4*>(img + off) = make_uint4(hw8[0], hw8[1], hw8[2], hw8[3]);
            *reinterpret_cast<uint4*>(img + off + kImgLoRow * 128) = make_uint4(lw8[0], lw8[1], lw8[2], lw8[3]);
            // sub-block sums (fp32) of sub-blocks 2*c4 (lo) and 2*c4+1 (hi) over the 8 lanes of c4
            float sl = (lo.x + lo.y) + (lo.z + lo.w), sh = (hi.x + hi.y) + (hi.z + hi.w);
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) {
                sl += __shfl_xor_sync(0xffffffffu, sl, off);
                sh += __shfl_xor_sync(0xffffffffu, sh, off);
            }
            // lane 0 gathers sx_0..7 and writes the min-term row: [hi(sx_0..7) | lo(sx_0..7)]
            float sx[8];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                sx[2 * c] = __shfl_sync(0xffffffffu, sl, 8 * c);
                sx[2 * c + 1] = __shfl_sync(0xffffffffu, sh, 8 * c);
            }
            if (lane == 0) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const __half a0 = __float2half_rn(sx[2 * i]), a1 = __float2half_rn(sx[2 * i + 1]);
                    const __half b0 = __float2half_rn(sx[2 * i] - __half2float(a0));
                    const __half b1 = __float2half_rn(sx[2 * i + 1] - __half2float(a1));
                    hw[i] = (uint32_t)__half_as_ushort(a0) | ((uint32_t)__half_as_ushort(a1) << 16);
                    lw[i] = (uint32_t)__half_as_ushort(b0) | ((uint32_t)__half_as_ushort(b1) << 16);
                }
                uint8_t* r2 = img + kImgMin + t * 128;
                *reinterpret_cast<uint4*>(r2 + ((0 ^ (t & 7)) << 4)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(r2 + ((1 ^ (t & 7)) << 4)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

__device__ __forceinline__ __half2 hfma2_bits(uint32_t a, __half2 b, __half2 c) {
    return __hfma2(*reinterpret_cast<__half2*>(&a), b, c);
}

// item -> (expert, tile, first chunk, chunks, tokens of each): an item is a row tile of one
// expert and CPI consecutive 32-token chunks of its bucket (CPI = 2: a pair, the last pair of an
// odd count holding one, so each block is dequantized once for up to 64 tokens). Items of expert
// e are [pstart[e]*tiles, (pstart[e] + groups_e)*tiles), chunk group fastest, so the groups of one
// row tile run together and share its weight reads in L2.
struct TcItem { int e, tile, c0, nch, nt0, nt1; };
template <int CPI>
__device__ __forceinline__ TcItem tc_item(const TcGroup& G, const int* cnt, const int* pstart, int item) {
    int lo = 0, hi = G.num_experts - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pstart[mid] * G.tiles <= item) lo = mid; else hi = mid - 1;
    }
    TcItem it;
    it.e = lo;
    const int chunks_e = (cnt[lo] + kTcTok - 1) / kTcTok;
    const int pairs_e = CPI == 1 ? chunks_e : (chunks_e + 1) / 2;
    const int local = item - pstart[lo] * G.tiles;
    it.tile = local / pairs_e;
    it.c0 = CPI * (local % pairs_e);
    it.nch = CPI == 1 ? 1 : min(2, chunks_e - it.c0);
    it.nt0 = min(kTcTok, cnt[lo] - it.c0 * kTcTok);
    it.nt1 = it.nch > 1 ? min(kTcTok, cnt[lo] - (it.c0 + 1) * kTcTok) : 0;
    return it;
}

// Persistent: grid = (SMs, groups); each CTA walks items grid-stride. A global step counter
// (one step = one Q4_K block of one slab) carries the A stage index and mbarrier parity
// across items, an image counter (one per step and chunk) the B stages; tensor memory is
// allocated once per CTA. The two accumulator slots (D1, D2) serve the two chunks of a pair
// item, or alternate between the steps of a one-chunk item (double buffering); every role
// counts the uses of each slot the same way.
template <bool FUSED, int CPI>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_gemm_kernel(const __grid_constant__ TcParams P) {
    static_assert(CPI == 1 || CPI == 2, "one or two chunks per item");
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* bimg = smem;                          // kNImg x kImgBlock (1024-byte aligned stages)
    uint8_t* raw = smem + kNImg * kImgBlock;       // kNRaw x kRawStage
    int* tabs = reinterpret_cast<int*>(smem + P.tab_off);
    __shared__ __align__(8) uint64_t bar_raw_full[kNRaw], bar_raw_empty[kNRaw], bar_a_full[2], bar_a_empty[2];
    __shared__ __align__(8) uint64_t bar_b_full[kNImg], bar_b_empty[kNImg], bar_d_full[2], bar_d_empty[2], bar_drain;
    __shared__ uint32_t s_tmem;
    __shared__ int s_warp[33];
    __shared__ int s_bad;
    __shared__ int s_pairs_w[8][CPI * kTcTok];  // each worker warp keeps its own copy (no cross-warp barrier)
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gi = blockIdx.y;
    const TcGroup& G = P.g[gi];
    int* cnt = tabs + P.hist_off[gi];
    int* start = cnt + G.num_experts;     // first chunk of each expert (its B images)
    int* pstart = CPI == 1 ? start : start + G.num_experts;  // first chunk group of each expert (its items)
    int groups = tc_chunks(G, P.tc_min, cnt, start, s_warp, &s_bad);
    if constexpr (CPI == 2) {
        for (int e = tid; e < G.num_experts; e += blockDim.x)
            pstart[e] = cnt[e] >= P.tc_min ? ((cnt[e] + kTcTok - 1) / kTcTok + 1) / 2 : 0;
        __syncthreads();
        groups = block_exclusive_scan(pstart, G.num_experts, s_warp);
    }
    const int total_items = groups * G.tiles;
    if ((int)blockIdx.x >= total_items) return;  // uniform per CTA: before any allocation

    if (warp == kTcMmaWarp) {
        tmem_alloc(&s_tmem, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < kNRaw; ++i) {
            mbar_init(&bar_raw_full[i], 1);
            mbar_init(&bar_raw_empty[i], kTcWorkers);
        }
        for (int i = 0; i < kNImg; ++i) {
            mbar_init(&bar_b_full[i], 1);
            mbar_init(&bar_b_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_a_full[i], kTcWorkers);
            mbar_init(&bar_a_empty[i], 1);
            mbar_init(&bar_d_full[i], 1);
            mbar_init(&bar_d_empty[i], kTcWorkers);
        }
        mbar_init(&bar_drain, 1);
        fence_mbar_init();
        s_abort = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int nb = G.k / kQK;
    const int nslab = FUSED ? 2 : 1;
    const int steps = nslab * nb;

    if (warp == kTcCopyWarp) {
        // ---------------- copy producer: raw rows of the tile and the block's B image
        int raw_issued = 0, b_issued = 0;
        bool ok = true;
        if constexpr (CPI == 1) {
        int gs = 0;  // global step
        for (int item = blockIdx.x; item < total_items && ok; item += gridDim.x) {
            const TcItem it = tc_item<CPI>(G, cnt, pstart, item);
            const int row0 = it.tile * kTcRows;
            const uint8_t* img = G.img + (int64_t)(start[it.e] + it.c0) * nb * kImgBlock;
            for (int s = 0; s < steps; ++s, ++gs) {
                const int rst = gs % kNRaw;
                const uint32_t rph = (gs / kNRaw) & 1;
                const int bst = gs % kNImg;
                const uint32_t bph = (gs / kNImg) & 1;
                const int slab = s / nb, b = s % nb;
                int okl = 1;
                if (lane == 0) {
                    okl = mbar_wait_for(&bar_raw_empty[rst], rph ^ 1, &s_abort, P.wait_ns);
                    if (okl) {
                        // one tensor load: 128 rows x 144 bytes of block b (rows past the slab read as zero)
                        mbar_arrive_expect_tx(&bar_raw_full[rst], kRawStage);
                        tma_load_2d(raw + rst * kRawStage, &P.tmap[gi][slab], b * kBlockBytes, it.e * G.n + row0,
                                    &bar_raw_full[rst]);
                    }
                }
                if (!__shfl_sync(0xffffffffu, okl, 0)) { ok = false; break; }
                raw_issued = gs + 1;
                if (lane == 0) {
                    okl = mbar_wait_for(&bar_b_empty[bst], bph ^ 1, &s_abort, P.wait_ns);
                    if (okl) {
                        mbar_arrive_expect_tx(&bar_b_full[bst], kImgBlock);
                        bulk_g2s(bimg + bst * kImgBlock, img + (int64_t)b * kImgBlock, kImgBlock, &bar_b_full[bst]);
                    }
                }
                if (!__shfl_sync(0xffffffffu, okl, 0)) { ok = false; break; }
                b_issued = gs + 1;
            }
        }
        } else {
        int gs = 0, gimg = 0;  // global step, global image
        for (int item = blockIdx.x; item < total_items && ok; item += gridDim.x) {
            const TcItem it = tc_item<CPI>(G, cnt, pstart, item);
            const int row0 = it.tile * kTcRows;
            const uint8_t* img = G.img + (int64_t)(start[it.e] + it.c0) * nb * kImgBlock;
            for (int s = 0; s < steps && ok; ++s, ++gs) {
                const int rst = gs % kNRaw;
                const uint32_t rph = (gs / kNRaw) & 1;
                const int slab = s / nb, b = s % nb;
                int okl = 1;
                if (lane == 0) {
                    okl = mbar_wait_for(&bar_raw_empty[rst], rph ^ 1, &s_abort, P.wait_ns);
                    if (okl) {
                        // one tensor load: 128 rows x 144 bytes of block b (rows past the slab read as zero)
                        mbar_arrive_expect_tx(&bar_raw_full[rst], kRawStage);
                        tma_load_2d(raw + rst * kRawStage, &P.tmap[gi][slab], b * kBlockBytes, it.e * G.n + row0,
                                    &bar_raw_full[rst]);
                    }
                }
                if (!__shfl_sync(0xffffffffu, okl, 0)) { ok = false; break; }
                raw_issued = gs + 1;
                for (int c = 0; c < it.nch; ++c, ++gimg) {  // the block's B image of each chunk
                    const int bst = gimg % kNImg;
                    const uint32_t bph = (gimg / kNImg) & 1;
                    if (lane == 0) {
                        okl = mbar_wait_for(&bar_b_empty[bst], bph ^ 1, &s_abort, P.wait_ns);
                        if (okl) {
                            mbar_arrive_expect_tx(&bar_b_full[bst], kImgBlock);
                            bulk_g2s(bimg + bst * kImgBlock, img + ((int64_t)c * nb + b) * kImgBlock, kImgBlock,
                                     &bar_b_full[bst]);
                        }
                    }
                    if (!__shfl_sync(0xffffffffu, okl, 0)) { ok = false; break; }
                    b_issued = gimg + 1;
                }
            }
        }
        }
        if (!ok && lane == 0) {
            // let the copies already issued land before the CTA leaves (bounded)
            volatile int never = 0;
            for (int g = max(0, raw_issued - kNRaw); g < raw_issued; ++g)
                mbar_wait(&bar_raw_full[g % kNRaw], (g / kNRaw) & 1, &never);
            for (int g = max(0, b_issued - kNImg); g < b_issued; ++g)
                mbar_wait(&bar_b_full[g % kNImg], (g / kNImg) & 1, &never);
        }
    } else if (warp == kTcMmaWarp) {
        // ---------------- MMA issuer: the whole warp runs the loop on warp-uniform values and
        // waits on the barriers; one elected lane issues each MMA and commit. (Issued by a lone
        // lane with per-instruction operand arithmetic, the same MMAs took about 1.7x as long.)
        const uint32_t idesc = idesc_f16_f32(kTcRows, 2 * kTcTok);   // fp16 part | residual
        const uint32_t idesc_min = idesc_f16_f32(kTcRows, kTcTok);
        const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
        const uint32_t bimg_addr = __shfl_sync(0xffffffffu, smem_u32(bimg), 0);
        bool ok = true;
        int issued = 0;
        // One chunk per item keeps its own loop (stage = step parity for A, B and D alike): run
        // through the pair loop below, the same one-chunk items took measurably longer.
        if constexpr (CPI == 1) {
        int gs = 0;
        for (int item = blockIdx.x; item < total_items && ok; item += gridDim.x) {
            for (int s = 0; s < steps; ++s, ++gs) {
                const int st = gs & 1;
                const uint32_t ph = (gs >> 1) & 1;
                const int bst = gs % kNImg;
                const uint32_t bph = (gs / kNImg) & 1;
                const bool got = mbar_wait_for(&bar_a_full[st], ph, &s_abort, P.wait_ns) &&
                                 mbar_wait_for(&bar_b_full[bst], bph, &s_abort, P.wait_ns) &&
                                 mbar_wait_for(&bar_d_empty[st], ph ^ 1, &s_abort, P.wait_ns);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // one descriptor per step; the k steps add constant offsets to its address field
                const uint64_t bdesc = desc_sw128_kmajor(bimg_addr + bst * kImgBlock);
                const uint32_t a0 = tm + kColA + st * 128, d1 = tm + kColD1 + st * 64;
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * kPanel + (kk & 3) * 32;
                    mma_f16_ts_elect(d1, a0 + 8 * kk, bdesc + (koff >> 4), idesc, kk > 0);
                }
                mma_f16_ts_elect(tm + kColD2 + st * 32, tm + kColA2 + st * 16, bdesc + (kImgMin >> 4), idesc_min, 0);
                mma_commit_elect(&bar_a_empty[st]);
                mma_commit_elect(&bar_b_empty[bst]);
                mma_commit_elect(&bar_d_full[st]);
                issued = gs + 1;
            }
        }
        } else {
        int gs = 0, gimg = 0;
        int rr = 0, use0 = 0, use1 = 0;  // slot of the next one-chunk step; uses of each slot
        for (int item = blockIdx.x; item < total_items && ok; item += gridDim.x) {
            const TcItem it = tc_item<CPI>(G, cnt, pstart, item);
            for (int s = 0; s < steps && ok; ++s, ++gs) {
                const int st = gs & 1;
                const uint32_t ph = (gs >> 1) & 1;
                if (!__all_sync(0xffffffffu, mbar_wait_for(&bar_a_full[st], ph, &s_abort, P.wait_ns))) {
                    ok = false;
                    break;
                }
                const uint32_t a0 = tm + kColA + st * 128;
                for (int c = 0; c < it.nch; ++c, ++gimg) {
                    const int slot = it.nch == 2 ? c : rr;
                    const int bst = gimg % kNImg;
                    const uint32_t bph = (gimg / kNImg) & 1;
                    const bool got = mbar_wait_for(&bar_b_full[bst], bph, &s_abort, P.wait_ns) &&
                                     mbar_wait_for(&bar_d_empty[slot], ((slot ? use1 : use0) & 1) ^ 1, &s_abort,
                                                   P.wait_ns);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // one descriptor per image; the k steps add constant offsets to its address field
                    const uint64_t bdesc = desc_sw128_kmajor(bimg_addr + bst * kImgBlock);
                    const uint32_t d1 = tm + kColD1 + slot * 64;
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk) {
                        const uint32_t koff = (kk >> 2) * kPanel + (kk & 3) * 32;
                        mma_f16_ts_elect(d1, a0 + 8 * kk, bdesc + (koff >> 4), idesc, kk > 0);
                    }
                    mma_f16_ts_elect(tm + kColD2 + slot * 32, tm + kColA2 + st * 16, bdesc + (kImgMin >> 4),
                                     idesc_min, 0);
                    mma_commit_elect(&bar_b_empty[bst]);
                    mma_commit_elect(&bar_d_full[slot]);
                    if (slot) ++use1; else ++use0;
                    issued = 1;
                }
                if (!ok) break;
                if (it.nch == 1) rr ^= 1;
                mma_commit_elect(&bar_a_empty[st]);
            }
        }
        }
        if (!ok) {
            if (lane == 0) {
                s_abort = 1;
                raise_flag(P.err_flag, Q4K_ERR_TIMEOUT);
            }
            if (issued > 0) {  // outstanding MMAs finish before tensor memory is freed
                volatile int never = 0;
                mma_commit_elect(&bar_drain);
                mbar_wait(&bar_drain, 0, &never);
            }
        }
        __syncwarp();
    } else {
        // ---------------- dequantize (thread = row = TMEM lane) and epilogue
        const int quarter = warp & 3, half = warp >> 2;
        const int r = 32 * quarter + lane;  // 0..127
        const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
        constexpr int kHalfTok = kTcTok / 2;
        int gs = 0;
        int rr = 0, use0 = 0, use1 = 0;  // the same slot bookkeeping as the MMA issuer
        bool ok = true;
        for (int item = blockIdx.x; item < total_items && ok; item += gridDim.x) {
            const TcItem it = tc_item<CPI>(G, cnt, pstart, item);
            const int row0 = it.tile * kTcRows;
            const int rows_valid = min(kTcRows, G.n - row0);
            const int ntc[2] = {it.nt0, it.nt1};
            int* s_pairs = s_pairs_w[warp];  // chunk c's pairs at s_pairs[32 c ..]
            __syncwarp();  // this warp's previous outputs are written
            tc_gather(G, it.e, it.c0, it.nt0, s_pairs);
            if (CPI > 1 && it.nch > 1) tc_gather(G, it.e, it.c0 + 1, it.nt1, s_pairs + (CPI - 1) * kTcTok);
            __syncwarp();
            float acc[2][kHalfTok], accg[2][kHalfTok];
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int t = 0; t < kHalfTok; ++t) { acc[c][t] = 0.f; accg[c][t] = 0.f; }
            float d_prev = 0.f, dmin_prev = 0.f;
            for (int s = 0; s <= steps; ++s) {
                const int g_cur = gs + s;
                const int st = g_cur & 1;
                const uint32_t ph = (g_cur >> 1) & 1;
                float d_cur = 0.f, dmin_cur = 0.f;
                if (s < steps) {
                    const int rst = g_cur % kNRaw;
                    const uint32_t rph = (g_cur / kNRaw) & 1;
                    if (!mbar_wait_for(&bar_raw_full[rst], rph, &s_abort, P.wait_ns)) { ok = false; break; }
                    // this half's code bytes: 64-weight groups 2*half, 2*half + 1 (bytes 64*half ..)
                    const uint4* rp = reinterpret_cast<const uint4*>(raw + rst * kRawStage + r * kBlockBytes);
                    const uint4 h = rp[0];
                    uint4 hq[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) hq[i] = rp[1 + 4 * half + i];
                    mbar_arrive(&bar_raw_empty[rst]);
                    d_cur = __half2float(__ushort_as_half((unsigned short)(h.x & 0xFFFFu)));
                    dmin_cur = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
                    int sc[8], mn[8];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const unsigned y = (h.y >> (8 * j)) & 0xFFu, z = (h.z >> (8 * j)) & 0xFFu;
                        const unsigned w = (h.w >> (8 * j)) & 0xFFu;
                        sc[j] = y & 63u;
                        mn[j] = z & 63u;
                        sc[j + 4] = (w & 15u) | ((y >> 6) << 4);
                        mn[j + 4] = (w >> 4) | ((z >> 6) << 4);
                    }
                    if (!mbar_wait_for(&bar_a_empty[st], ph ^ 1, &s_abort, P.wait_ns)) { ok = false; break; }
                    tc_fence_after();
                    // A columns: code word i -> columns 4i..4i+3 = low nibbles of bytes (0,2), (1,3),
                    // high nibbles of bytes (0,2), (1,3), each the exact fp16 pair sc_j * q
#pragma unroll
                    for (int gl = 0; gl < 2; ++gl) {  // 32 columns = 8 code words = 64-weight group g
                        const int g = 2 * half + gl;
                        // sub-blocks 2g (low nibbles) and 2g + 1 (high nibbles)
                        const int sca = half ? sc[4 + 2 * gl] : sc[2 * gl];
                        const int scb = half ? sc[5 + 2 * gl] : sc[1 + 2 * gl];
                        const __half2 klo = __half2half2(__int2half_rn(sca));
                        const __half2 clo = __half2half2(__int2half_rn(-1024 * sca));
                        const __half2 khi = __half2half2(__float2half_rn((float)scb * 0.0625f));
                        const __half2 chi = __half2half2(__int2half_rn(-64 * scb));
                        uint32_t col[32];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint4 qv = hq[2 * gl + (i >> 2)];
                            const uint32_t wq = (i & 3) == 0 ? qv.x : (i & 3) == 1 ? qv.y : (i & 3) == 2 ? qv.z : qv.w;
                            const uint32_t w8 = wq >> 8;
                            col[4 * i + 0] = h2_bits(hfma2_bits((wq & 0x000F000Fu) | 0x64006400u, klo, clo));
                            col[4 * i + 1] = h2_bits(hfma2_bits((w8 & 0x000F000Fu) | 0x64006400u, klo, clo));
                            col[4 * i + 2] = h2_bits(hfma2_bits((wq & 0x00F000F0u) | 0x64006400u, khi, chi));
                            col[4 * i + 3] = h2_bits(hfma2_bits((w8 & 0x00F000F0u) | 0x64006400u, khi, chi));
                        }
                        tmem_st32(tmem + lane_base + kColA + st * 128 + 32 * g, col);
                    }
                    if (half == 0) {
                        uint32_t a2[8];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const __half2 mm = __halves2half2(__int2half_rn(mn[2 * i]), __int2half_rn(mn[2 * i + 1]));
                            a2[i] = a2[i + 4] = h2_bits(mm);
                        }
                        tmem_st8(tmem + lane_base + kColA2 + st * 16, a2);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&bar_a_full[st]);
                }
                if (CPI == 1 && s >= 1) {
                    // epilogue of step s-1 for this half's tokens: acc += d * (D1 hi + D1 lo) - dmin * D2
                    const int pg = g_cur - 1;
                    const int ps = pg & 1;
                    const uint32_t pph = (pg >> 1) & 1;
                    if (!mbar_wait_for(&bar_d_full[ps], pph, &s_abort, P.wait_ns)) { ok = false; break; }
                    // a chunk of at most 16 tokens leaves the second half's columns unused: its
                    // warps only hand the accumulators back (uniform per item)
                    if (kHalfTok * half < it.nt0) {
                        tc_fence_after();
                        uint32_t d1[kHalfTok], d2[kHalfTok], d3[kHalfTok];
                        tmem_ld16(tmem + lane_base + kColD1 + ps * 64 + kHalfTok * half, d1);
                        tmem_ld16(tmem + lane_base + kColD1 + ps * 64 + kTcTok + kHalfTok * half, d3);
                        tmem_ld16(tmem + lane_base + kColD2 + ps * 32 + kHalfTok * half, d2);
                        tmem_wait_ld();
                        tc_fence_before();
                        mbar_arrive(&bar_d_empty[ps]);
#pragma unroll
                        for (int t = 0; t < kHalfTok; ++t)
                            acc[0][t] = fmaf(d_prev, __uint_as_float(d1[t]) + __uint_as_float(d3[t]),
                                             fmaf(-dmin_prev, __uint_as_float(d2[t]), acc[0][t]));
                    } else {
                        mbar_arrive(&bar_d_empty[ps]);
                    }
                    if (FUSED && s - 1 == nb - 1) {  // the gate slab is complete
#pragma unroll
                        for (int t = 0; t < kHalfTok; ++t) { accg[0][t] = acc[0][t]; acc[0][t] = 0.f; }
                    }
                }
                if (CPI == 2 && s >= 1) {
                    // epilogue of step s-1 for this half's tokens of each chunk:
                    // acc += d * (D1 hi + D1 lo) - dmin * D2
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        if (c >= it.nch) break;
                        const int slot = it.nch == 2 ? c : rr;
                        if (!mbar_wait_for(&bar_d_full[slot], (slot ? use1 : use0) & 1, &s_abort, P.wait_ns)) {
                            ok = false;
                            break;
                        }
                        // a chunk of at most 16 tokens leaves the second half's columns unused:
                        // its warps only hand the accumulators back (uniform per item)
                        if (kHalfTok * half < ntc[c]) {
                            tc_fence_after();
                            uint32_t d1[kHalfTok], d2[kHalfTok], d3[kHalfTok];
                            tmem_ld16(tmem + lane_base + kColD1 + slot * 64 + kHalfTok * half, d1);
                            tmem_ld16(tmem + lane_base + kColD1 + slot * 64 + kTcTok + kHalfTok * half, d3);
                            tmem_ld16(tmem + lane_base + kColD2 + slot * 32 + kHalfTok * half, d2);
                            tmem_wait_ld();
                            tc_fence_before();
                            mbar_arrive(&bar_d_empty[slot]);
#pragma unroll
                            for (int t = 0; t < kHalfTok; ++t)
                                acc[c][t] = fmaf(d_prev, __uint_as_float(d1[t]) + __uint_as_float(d3[t]),
                                                 fmaf(-dmin_prev, __uint_as_float(d2[t]), acc[c][t]));
                        } else {
                            mbar_arrive(&bar_d_empty[slot]);
                        }
                        if (slot) ++use1; else ++use0;
                    }
                    if (!ok) break;
                    if (it.nch == 1) rr ^= 1;
                    if (FUSED && s - 1 == nb - 1) {  // the gate slab is complete
#pragma unroll
                        for (int c = 0; c < 2; ++c)
#pragma unroll
                            for (int t = 0; t < kHalfTok; ++t) { accg[c][t] = acc[c][t]; acc[c][t] = 0.f; }
                    }
                }
                d_prev = d_cur;
                dmin_prev = dmin_cur;
            }
            if (!ok) break;
            gs += steps;
            if (r < rows_valid) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
#pragma unroll
                    for (int j = 0; j < kHalfTok; ++j) {
                        const int t = kHalfTok * half + j;
                        if (c < it.nch && t < ntc[c]) {
                            float v = acc[c][j];
                            if (FUSED) v = (accg[c][j] / (1.0f + __expf(-accg[c][j]))) * acc[c][j];
                            G.out[(int64_t)s_pairs[kTcTok * c + t] * G.n + row0 + r] = v;
                        }
                    }
                }
            }
        }
        if (!ok) {
            s_abort = 1;
            raise_flag(P.err_flag, Q4K_ERR_TIMEOUT);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kTcMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------------------------------
int64_t tc_max_chunks(int n_pairs, int tc_min) {
    // sum over experts with >= tc_min pairs of ceil(cnt/32) <= n_pairs/32 + n_pairs/tc_min
    return (int64_t)n_pairs / kTcTok + (int64_t)n_pairs / tc_min + 1;
}

size_t tc_image_bytes(int n_pairs, int k, int tc_min) {
    return (size_t)tc_max_chunks(n_pairs, tc_min) * (size_t)(k / kQK) * kImgBlock;
}

static bool g_tc_attr_set[4][64] = {};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// The slab as a 2-D uint8 tensor: rows = num_experts * n, row length = nb01 bytes; one box is
// one Q4_K block (144 bytes) of 128 consecutive rows.
static cudaError_t encode_slab_map(CUtensorMap* map, const uint8_t* w, int num_experts, int n, int64_t nb01) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)nb01, (cuuint64_t)num_experts * (cuuint64_t)n};
    const cuuint64_t strides[1] = {(cuuint64_t)nb01};
    const cuuint32_t box[2] = {(cuuint32_t)kBlockBytes, (cuuint32_t)kTcRows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Whether a launch works on chunk pairs: the routed batch averages at least two 32-token chunks
// per expert (every group).
static bool tc_pairs(const GemvGroup* groups, int n_groups) {
    bool pairs = true;
    for (int gi = 0; gi < n_groups; ++gi)
        pairs = pairs && (int64_t)groups[gi].m * groups[gi].top_k >= (int64_t)2 * kTcTok * groups[gi].num_experts;
    return pairs;
}

bool tc_fits(const GemvGroup* groups, int n_groups) {
    int ints = 0;
    const int per_expert = tc_pairs(groups, n_groups) ? 3 : 2;  // cnt, start[, pstart]
    for (int gi = 0; gi < n_groups; ++gi) ints += per_expert * groups[gi].num_experts;
    return 1024 + (size_t)(kNImg * kImgBlock + kNRaw * kRawStage) + (size_t)ints * 4 <= 200 * 1024;
}

cudaError_t launch_tc(const GemvGroup* groups, int n_groups, bool fused, int tc_min, uint8_t* const* img,
                      int* err_flag, cudaStream_t stream, bool pdl) {
    TcParams P{};
    P.n_groups = n_groups;
    P.tc_min = tc_min;
    P.err_flag = err_flag;
    P.wait_ns = wait_limit_ns();
    // two 32-token chunks per item (one dequantization of each block for both) when the
    // routed batch averages at least two chunks per expert; else one
    const bool pairs = tc_pairs(groups, n_groups);
    int ints = 0;
    int64_t max_chunks = 0;
    int max_tiles = 0;
    for (int gi = 0; gi < n_groups; ++gi) {
        const GemvGroup& S = groups[gi];
        TcGroup& G = P.g[gi];
        G.w = S.w; G.w2 = S.w2; G.ids = S.ids; G.a = S.a; G.out = S.out; G.img = img[gi];
        G.outer = S.outer; G.inner = S.inner;
        G.nb01 = (int64_t)(S.k / kQK) * kBlockBytes;
        G.nb02 = (int64_t)S.n * G.nb01;
        G.num_experts = S.num_experts; G.n_pairs = S.m * S.top_k; G.top_k = S.top_k; G.n = S.n; G.k = S.k;
        G.tiles = (S.n + kTcRows - 1) / kTcRows;
        P.hist_off[gi] = ints;
        ints += (pairs ? 3 : 2) * S.num_experts;  // cnt, start (chunks)[, pstart (chunk pairs)]
        cudaError_t me = encode_slab_map(&P.tmap[gi][0], S.w, S.num_experts, S.n, G.nb01);
        if (me == cudaSuccess && fused) me = encode_slab_map(&P.tmap[gi][1], S.w2, S.num_experts, S.n, G.nb01);
        if (me != cudaSuccess) return me;
        const int64_t mc = tc_max_chunks(G.n_pairs, tc_min);
        max_chunks = mc > max_chunks ? mc : max_chunks;
        max_tiles = G.tiles > max_tiles ? G.tiles : max_tiles;
    }
    if (max_chunks == 0) return cudaSuccess;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    // prep: B images
    {
        const size_t smem = (size_t)ints * 4;
        cudaLaunchConfig_t cfg = {};
        int kmax = 0;
        for (int gi = 0; gi < n_groups; ++gi) kmax = groups[gi].k > kmax ? groups[gi].k : kmax;
        const int slices = kmax / kQK < 16 ? kmax / kQK : 16;
        cfg.gridDim = dim3((unsigned)max_chunks, n_groups, (unsigned)slices);
        cfg.blockDim = dim3(128);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        err = cudaLaunchKernelEx(&cfg, tc_prep_kernel, P);
        if (err != cudaSuccess) return err;
    }
    P.tab_off = kNImg * kImgBlock + kNRaw * kRawStage;
    // every CTA holds all 512 tensor-memory columns: ask for enough shared memory that only
    // one CTA fits on an SM
    size_t smem = 1024 + (size_t)P.tab_off + (size_t)ints * 4;
    if (smem < 120 * 1024) smem = 120 * 1024;
    if (smem > 200 * 1024) return cudaErrorInvalidValue;
    void (*kern)(TcParams) = fused ? (pairs ? tc_gemm_kernel<true, 2> : tc_gemm_kernel<true, 1>)
                                   : (pairs ? tc_gemm_kernel<false, 2> : tc_gemm_kernel<false, 1>);
    const int kind = (fused ? 1 : 0) + (pairs ? 2 : 0);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!g_tc_attr_set[kind][dev]) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (err != cudaSuccess) return err;
        g_tc_attr_set[kind][dev] = true;
    }
    if (smem > 200 * 1024) return cudaErrorInvalidValue;
    int64_t grid = (int64_t)max_chunks * max_tiles;
    if (grid > num_sms()) grid = num_sms();
    kern<<<dim3((unsigned)grid, n_groups), kTcThreads, smem, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace q4k

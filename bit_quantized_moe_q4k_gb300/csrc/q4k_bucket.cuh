// q4k_bucket.cuh -- block-level building blocks of the pair bucketing.
//
// A (token, slot) pair p = token*top_k + slot belongs to the bucket of expert ids[p]
// (moeflux expert_forward.rs, `encode_moe_batched_permute_fuse` and the map0 step of
// `encode_moe_gather_id_fuse`: bucket the pairs by expert and process each bucket once).
// Buckets are ordered by expert id and each bucket lists its pairs in increasing
// pair index, which makes the result unique.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace q4k {

__device__ __forceinline__ bool id_valid(int32_t e, int num_experts) {
    return e >= 0 && e < num_experts;
}

// Exclusive prefix sum of s[0..n) in place, any n >= 0, called by every thread of the
// block. Thread t owns the contiguous range [t*per, (t+1)*per). s_warp: 33 ints of
// scratch. Returns the total. Ends with a barrier.
__device__ __forceinline__ int block_exclusive_scan(int* s, int n, int* s_warp) {
    const int nt = blockDim.x, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = (nt + 31) >> 5;
    const int per = (n + nt - 1) / nt;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int local = 0;
    for (int i = lo; i < hi; ++i) local += s[i];
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? s_warp[lane] : 0;
        int wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += y;
        }
        if (lane < nwarps) s_warp[lane] = wi - w;  // exclusive warp offsets
        if (lane == 31) s_warp[32] = wi;           // total (nwarps <= 32)
    }
    __syncthreads();
    int run = s_warp[warp] + incl - local;
    const int total = s_warp[32];
    for (int i = lo; i < hi; ++i) {
        const int v = s[i];
        s[i] = run;
        run += v;
    }
    __syncthreads();
    return total;
}

// s_cnt[e] = #{p < n_pairs : ids[p] == e} for e < num_experts; *s_bad = out-of-range ids.
// Called by every thread; ends with a barrier.
__device__ __forceinline__ void block_histogram(const int32_t* ids, int n_pairs, int num_experts,
                                                int* s_cnt, int* s_bad) {
    for (int e = threadIdx.x; e < num_experts; e += blockDim.x) s_cnt[e] = 0;
    if (threadIdx.x == 0) *s_bad = 0;
    __syncthreads();
    for (int p = threadIdx.x; p < n_pairs; p += blockDim.x) {
        int32_t e = ids[p];
        if (id_valid(e, num_experts)) atomicAdd(&s_cnt[e], 1);
        else atomicAdd(s_bad, 1);
    }
    __syncthreads();
}

// One warp: write the pairs p with ids[p] == e, in increasing order, skipping the first
// `skip` of them and keeping at most `keep`, to out[0..). Returns the number written.
__device__ __forceinline__ int warp_gather_bucket(const int32_t* ids, int n_pairs, int32_t e, int skip,
                                                  int keep, int* out) {
    const int lane = threadIdx.x & 31;
    int seen = 0, written = 0;
    for (int base = 0; base < n_pairs && written < keep; base += 32) {
        int p = base + lane;
        bool hit = p < n_pairs && ids[p] == e;
        unsigned mask = __ballot_sync(0xffffffffu, hit);
        int rank = seen + __popc(mask & ((1u << lane) - 1u));
        if (hit && rank >= skip && rank - skip < keep) out[rank - skip] = p;
        seen += __popc(mask);
        written = min(max(seen - skip, 0), keep);
    }
    return written;
}

}  // namespace q4k

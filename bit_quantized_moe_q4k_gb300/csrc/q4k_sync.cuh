// q4k_sync.cuh -- hand-off between the CTAs of one launch without zero-initialised state,
// used by the single-launch layer kernel (q4k_layer.cu) and the tensor-core kernel's bounded
// waits (q4k_tc.cu).
//
// A launch's tag is next_tag(generation word). A CTA that finishes a piece of work stores the
// tag into that piece's flag word (release); a CTA that needs the piece waits until the word
// holds the tag (acquire). The generation word is advanced to the tag by one CTA of the launch
// once every CTA has recorded the value it read, so flags left by earlier launches (or any
// other contents of the memory) never match, and nothing has to be cleared between calls.
// Every wait is bounded in time; the limit is a launch argument.
#pragma once

#include <stdint.h>

#include "q4k_sm100.cuh"

namespace q4k {

// splitmix64's output function (Steele, Lea, Flood 2014): a bijective 64-bit mixer.
__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// The tag of the launch after the one whose generation word is g: a hash of g whose lowest
// bit flips at every launch (consecutive launches use different counter sets).
__device__ __forceinline__ uint64_t next_tag(uint64_t g) { return (mix64(g) & ~1ull) | ((g & 1ull) ^ 1ull); }

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Wait for the mbarrier phase with the given parity. Gives up (false) after limit_ns of wall
// time or once *abort is set. Below a millisecond the waits poll without suspending the
// thread (try_wait may suspend it for longer than such a limit), so a short limit holds.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              uint64_t limit_ns) {
    const bool short_limit = limit_ns < 1000000ull;
    auto try_once = [&]() { return short_limit ? sm100::mbar_test_wait(bar, parity) : sm100::mbar_try_wait(bar, parity); };
    if (try_once()) return true;
    const uint64_t t0 = sm100::global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (try_once()) return true;
        if (*abort) return false;
        if (((i & 15) == 0 || short_limit) && sm100::global_timer_ns() - t0 > limit_ns) return false;
    }
}

}  // namespace q4k

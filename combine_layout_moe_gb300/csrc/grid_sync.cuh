// Grid-wide barrier for cooperative launches, and the acquire / release
// accesses it is built from (sm_90 and later).
#pragma once

#include <cstdint>

#include "common.cuh"
#include "tma.cuh"

namespace moe {

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned atom_add_release_u32(unsigned *p, unsigned v)
{
    unsigned old;
    asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
                 : "memory");
    return old;
}

// Sense-reversing barrier across the co-resident CTAs of a cooperative launch.
// bar[0] counts arrivals and must be zero when a launch starts; bar[1] is the
// generation.  Arrival is a release (it publishes what this CTA wrote before
// its __syncthreads) and the wait an acquire.  The last CTA to arrive resets
// the count and bumps the generation, so every launch leaves the count at zero
// again.  The wait gives up after MBAR_TIMEOUT_NS and reports
// MOE_ERRBIT_TIMEOUT.  Returns whether the barrier completed.
__device__ __forceinline__ bool grid_barrier(unsigned *bar, uint32_t *err_word)
{
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned *count = bar, *gen = bar + 1;
        const unsigned g = ld_acquire_u32(gen);  // before arriving: cannot have moved yet
        int done = 1;
        if (atom_add_release_u32(count, 1u) == gridDim.x - 1) {
            atomicExch(count, 0u);
            atom_add_release_u32(gen, 1u);
        } else {
            const uint64_t t0 = global_ns();
            while (ld_acquire_u32(gen) == g) {
                if (global_ns() - t0 > MBAR_TIMEOUT_NS) {
                    done = 0;
                    report(err_word, MOE_ERRBIT_TIMEOUT);
                    break;
                }
            }
        }
        ok = done;
    }
    __syncthreads();
    return ok != 0;
}

}  // namespace moe

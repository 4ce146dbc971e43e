// Device helpers shared by the layout, dispatch and combine kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "moe_ep.h"

namespace moe {

constexpr unsigned FULL_MASK = 0xffffffffu;

// 16-byte read-only load that bypasses L1 allocation: every payload byte is
// read exactly once, so keeping it in L1 only evicts useful lines.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ int32_t ld_nc_s32(const int32_t *p)
{
    int32_t v;
    asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_nc_f32(const float *p)
{
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void *p, uint4 v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_v2(void *p, uint2 v)
{
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ unsigned lanemask_lt()
{
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ void report(uint32_t *err_word, uint32_t bit)
{
    if (err_word != nullptr)
        atomicOr(err_word, bit);
}

// Programmatic dependent launch.  Every kernel waits for the grid before it in
// the stream to finish (and its writes to be visible) before its first global
// memory access, then lets the next grid in the stream launch early: that
// grid's CTAs become resident and park in their own wait, so the launch gap
// between back-to-back kernels is hidden.  Both are no-ops for a kernel
// launched without the programmatic-serialisation attribute.
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// bf16 pair (packed in a 32-bit word, low half first) widened to two floats.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

}  // namespace moe

// Dispatch -> identity expert -> combine in one persistent kernel, with
// Data-as-Flag readiness (sm_103a).
//
// UBEP, section 3.4 (Data-as-Flag: readiness travels with the data instead of
// a global barrier), section 3.2 (kernel decomposition: consumers start on a
// piece of work as soon as its inputs are signalled) and section 6 (without
// an atomic 512-byte write, fall back to explicit fences or acknowledgements).
// A GPU has no 512-byte atomic store, so every row chunk gets its own 32-bit
// sequence word: the producer stores the chunk, fences, then writes the word;
// the consumer waits for the word with acquire loads, then reads the chunk.
// Words carry the caller's epoch, so they never need a reset between calls
// (UBEP's sentinel-polling variant needs one).
//
// Structure: one cooperative launch (every warp is resident).  Units are
// (token t, chunk c of DC_CHUNK bytes of the row).  Each warp first produces
// its contiguous range of units -- load x[t] chunk c, store it to the k
// destination rows, publish the k sequence words -- and only then consumes its
// range: for j = 0..k-1 wait for word (slot_of[t,j], c), read that row chunk
// from L2 and fold it into fp32 accumulators (one fused multiply-add per slot
// in slot order, starting from +0), then store out[t] chunk c.  Producing never
// waits and every producer is resident, so every wait ends; each wait is
// still bounded by the caller's limit and reports MOE_ERRBIT_TIMEOUT.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"
#include "tma.cuh"

namespace moe {

constexpr int DC_THREADS = 256;
constexpr int DC_U = 4;                 // 16-byte vectors per lane per unit
constexpr int DC_CHUNK = 32 * DC_U * 16;  // bytes of a row per unit (2 KB)

__device__ __forceinline__ void st_relaxed_u32(uint32_t *p, uint32_t v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_word(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// 16-byte load that bypasses L1: the data was written by other SMs during
// this kernel and is read after an acquire.
__device__ __forceinline__ uint4 ld_cg_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__global__ void __launch_bounds__(DC_THREADS)
    dispatch_combine_flagged_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ slot_of,
                                    const float *__restrict__ topk_w, uint4 *recv, void *__restrict__ out,
                                    int out_f32, int T, int k, int C, int nchunks, int64_t units,
                                    uint32_t *seq, uint32_t epoch, uint64_t spin_limit_ns,
                                    int64_t skip_pair, uint32_t *err_word)
{
    wait_prior_grid();
    allow_next_grid();
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (DC_THREADS / 32);
    const int64_t gw = (int64_t)blockIdx.x * (DC_THREADS / 32) + (threadIdx.x >> 5);
    const int64_t u0 = units * gw / nw, u1 = units * (gw + 1) / nw;
    const int N = T * k;

    // ---- produce: x[t] chunk c -> k rows; then every lane fences (its row
    //      stores are visible GPU-wide) and lane j publishes row j's word
    for (int64_t u = u0; u < u1; ++u) {
        const int64_t t = u / nchunks;
        const int c = (int)(u - t * nchunks);
        const int v0 = c * (32 * DC_U) + lane;
        uint4 v[DC_U];
#pragma unroll
        for (int q = 0; q < DC_U; ++q)
            if (v0 + 32 * q < C)
                v[q] = ld_stream_v4(x + t * C + v0 + 32 * q);
        const int32_t mine = lane < k ? ld_nc_s32(slot_of + t * k + lane) : -1;
        for (int j = 0; j < k; ++j) {
            const int32_t s = __shfl_sync(FULL_MASK, mine, j);
            if ((unsigned)s >= (unsigned)N) {
                if (lane == 0 && c == 0)
                    report(err_word, MOE_ERRBIT_BAD_INDEX);
                continue;
            }
#pragma unroll
            for (int q = 0; q < DC_U; ++q)
                if (v0 + 32 * q < C)
                    st_v4(recv + (int64_t)s * C + v0 + 32 * q, v[q]);
        }
        __threadfence();
        __syncwarp();
        if (lane < k && (unsigned)mine < (unsigned)N && t * k + lane != skip_pair)
            st_relaxed_u32(seq + (int64_t)mine * nchunks + c, epoch);
    }

    // ---- consume: wait for the k row chunks, fold them in slot order
    for (int64_t u = u0; u < u1; ++u) {
        const int64_t t = u / nchunks;
        const int c = (int)(u - t * nchunks);
        const int v0 = c * (32 * DC_U) + lane;
        const int32_t ms = lane < k ? ld_nc_s32(slot_of + t * k + lane) : 0;
        const float mw = lane < k ? ld_nc_f32(topk_w + t * k + lane) : 0.0f;
        float acc[DC_U][8];
#pragma unroll
        for (int q = 0; q < DC_U; ++q)
#pragma unroll
            for (int i = 0; i < 8; ++i)
                acc[q][i] = 0.0f;
        bool ready = true;
        for (int j = 0; j < k; ++j) {
            const int32_t s = __shfl_sync(FULL_MASK, ms, j);
            const float w = __shfl_sync(FULL_MASK, mw, j);
            if ((unsigned)s >= (unsigned)N)
                continue;
            // every lane acquires the word itself, so its own loads below are
            // ordered after the producer's fence; the exit is warp-uniform
            const uint32_t *word = seq + (int64_t)s * nchunks + c;
            bool arrived = __all_sync(FULL_MASK, ld_acquire_word(word) == epoch);
            if (!arrived) {
                const uint64_t t0 = global_ns();
                for (;;) {
                    if (__all_sync(FULL_MASK, ld_acquire_word(word) == epoch)) {
                        arrived = true;
                        break;
                    }
                    if (__shfl_sync(FULL_MASK, (int)(global_ns() - t0 > spin_limit_ns), 0))
                        break;
                }
            }
            if (!arrived) {
                if (lane == 0)
                    report(err_word, MOE_ERRBIT_TIMEOUT);
                ready = false;
                break;
            }
#pragma unroll
            for (int q = 0; q < DC_U; ++q) {
                if (v0 + 32 * q < C) {
                    const uint4 r = ld_cg_v4(recv + (int64_t)s * C + v0 + 32 * q);
                    const uint32_t p[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        acc[q][2 * h] = __fmaf_rn(w, bf16lo(p[h]), acc[q][2 * h]);
                        acc[q][2 * h + 1] = __fmaf_rn(w, bf16hi(p[h]), acc[q][2 * h + 1]);
                    }
                }
            }
        }
        if (!ready)
            continue;  // this unit's output stays unwritten; the error word says why
#pragma unroll
        for (int q = 0; q < DC_U; ++q) {
            const int cv = v0 + 32 * q;
            if (cv >= C)
                continue;
            if (out_f32) {
                float4 *o = static_cast<float4 *>(out) + (t * C + cv) * 2;
                st_v4(o, make_uint4(__float_as_uint(acc[q][0]), __float_as_uint(acc[q][1]),
                                    __float_as_uint(acc[q][2]), __float_as_uint(acc[q][3])));
                st_v4(o + 1, make_uint4(__float_as_uint(acc[q][4]), __float_as_uint(acc[q][5]),
                                        __float_as_uint(acc[q][6]), __float_as_uint(acc[q][7])));
            } else {
                uint32_t rr[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[q][2 * h], acc[q][2 * h + 1]);
                    rr[h] = *reinterpret_cast<const uint32_t *>(&b);
                }
                st_v4(static_cast<uint4 *>(out) + t * C + cv, make_uint4(rr[0], rr[1], rr[2], rr[3]));
            }
        }
    }
}

int flagged_chunks(int H) { return (2 * H + DC_CHUNK - 1) / DC_CHUNK; }

cudaError_t launch_dispatch_combine_flagged(int T, int H, int k, const void *x,
                                            const int32_t *slot_of, const float *topk_w,
                                            void *recv, void *out, bool out_f32, uint32_t *seq,
                                            uint32_t epoch, uint64_t spin_limit_ns,
                                            int64_t skip_pair, uint32_t *err_word,
                                            cudaStream_t stream)
{
    if (T == 0)
        return cudaSuccess;
    const int C = H / 8;
    const int nchunks = flagged_chunks(H);
    const int64_t units = (int64_t)T * nchunks;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, dispatch_combine_flagged_kernel, DC_THREADS, 0);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    const int64_t warps_needed = units;
    int64_t grid = (int64_t)sm_count() * per_sm;  // every CTA co-resident
    const int64_t need = (warps_needed + DC_THREADS / 32 - 1) / (DC_THREADS / 32);
    if (need < grid)
        grid = need;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(DC_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dispatch_combine_flagged_kernel,
                              static_cast<const uint4 *>(x), slot_of, topk_w,
                              static_cast<uint4 *>(recv), out, out_f32 ? 1 : 0, T, k, C, nchunks,
                              units, seq, epoch, spin_limit_ns, skip_pair, err_word);
}

}  // namespace moe

// Combine: gather the k expert-output rows of each token and reduce them as a
// router-weighted fp32 sum (sm_103a).
//
// HyperParallel-MoE, section 2.2 (expert outputs weighted by routing scores and
// combined) and section 4.1 (top-k contributions accumulated according to the
// routing scores); RailWave, section 3 (combine uses the saved dispatch
// metadata to return rows to their token positions).
//
// GPU design: a pull.  The work item is one warp on one (token, row chunk).
// Each lane holds 8 channels x U vectors; the k source rows are loaded KC at a
// time (KC x U independent 16-byte loads in flight per lane, 512 contiguous
// bytes per warp instruction), then folded into fp32 accumulators with one
// fused multiply-add per slot in slot order j = 0..k-1, starting from +0.  The
// result is rounded once (nearest-even) and stored with 16-byte stores.  No
// atomics: every output element is written by exactly one lane, so the result
// is deterministic.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"

namespace moe {

constexpr int COMBINE_THREADS = 256;

template <int KC, int U>
__global__ void __launch_bounds__(COMBINE_THREADS, 2)
    combine_kernel(const uint4 *__restrict__ y, const int32_t *__restrict__ slot_of,
                   const float *__restrict__ topk_w, void *__restrict__ out, int out_f32, int k,
                   int C, int groups, int64_t items, int N, uint32_t *err_word)
{
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (COMBINE_THREADS / 32);
    for (int64_t it = (int64_t)blockIdx.x * (COMBINE_THREADS / 32) + (threadIdx.x >> 5);
         it < items; it += nwarps) {
        const int64_t t = it / groups;
        const int c0 = (int)(it - t * groups) * (32 * U) + lane;
        float acc[U][8];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int i = 0; i < 8; ++i)
                acc[u][i] = 0.0f;

        const int32_t *so = slot_of + t * k;
        const float *wt = topk_w + t * k;
        int32_t my_slot = 0;
        float my_w = 0.0f;
        for (int jb = 0; jb < k; jb += KC) {
            if ((jb & 31) == 0) {
                my_slot = jb + lane < k ? ld_nc_s32(so + jb + lane) : 0;
                my_w = jb + lane < k ? ld_nc_f32(wt + jb + lane) : 0.0f;
            }
            uint4 v[KC][U];
            bool ok[KC];
#pragma unroll
            for (int q = 0; q < KC; ++q) {
                const int32_t s = __shfl_sync(FULL_MASK, my_slot, (jb + q) & 31);
                ok[q] = jb + q < k && (unsigned)s < (unsigned)N;
                const uint4 *row = y + (int64_t)s * C;
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (ok[q] && c0 + u * 32 < C)
                        v[q][u] = ld_stream_v4(row + c0 + u * 32);
                    else
                        v[q][u] = make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < KC; ++q) {
                const float w = __shfl_sync(FULL_MASK, my_w, (jb + q) & 31);
                if (jb + q < k && !ok[q]) {
                    if (lane == 0)
                        report(err_word, MOE_ERRBIT_BAD_INDEX);
                }
                if (!ok[q])
                    continue;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint32_t p[4] = {v[q][u].x, v[q][u].y, v[q][u].z, v[q][u].w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        acc[u][2 * h] = __fmaf_rn(w, bf16lo(p[h]), acc[u][2 * h]);
                        acc[u][2 * h + 1] = __fmaf_rn(w, bf16hi(p[h]), acc[u][2 * h + 1]);
                    }
                }
            }
        }

#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + u * 32;
            if (c >= C)
                continue;
            if (out_f32) {
                float4 *o = static_cast<float4 *>(out) + (t * C + c) * 2;
                st_v4(o, make_uint4(__float_as_uint(acc[u][0]), __float_as_uint(acc[u][1]),
                                    __float_as_uint(acc[u][2]), __float_as_uint(acc[u][3])));
                st_v4(o + 1, make_uint4(__float_as_uint(acc[u][4]), __float_as_uint(acc[u][5]),
                                        __float_as_uint(acc[u][6]), __float_as_uint(acc[u][7])));
            } else {
                uint32_t r[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[u][2 * h], acc[u][2 * h + 1]);
                    r[h] = *reinterpret_cast<const uint32_t *>(&b);
                }
                st_v4(static_cast<uint4 *>(out) + t * C + c, make_uint4(r[0], r[1], r[2], r[3]));
            }
        }
    }
}

template <int KC, int U>
static cudaError_t launch_combine_t(int T, int H, int k, const void *y, const int32_t *slot_of,
                                    const float *topk_w, void *out, bool out_f32,
                                    uint32_t *err_word, cudaStream_t stream)
{
    const int C = H / 8;
    const int groups = (C + 32 * U - 1) / (32 * U);
    const int64_t items = (int64_t)T * groups;
    const int grid = warp_item_grid((const void *)combine_kernel<KC, U>, COMBINE_THREADS, 0, items);
    combine_kernel<KC, U><<<grid, COMBINE_THREADS, 0, stream>>>(
        static_cast<const uint4 *>(y), slot_of, topk_w, out, out_f32 ? 1 : 0, k, C, groups, items,
        T * k, err_word);
    return cudaGetLastError();
}

cudaError_t launch_combine(int T, int H, int k, const void *y, const int32_t *slot_of,
                           const float *topk_w, void *out, bool out_f32, uint32_t *err_word,
                           cudaStream_t stream)
{
    if (T == 0)
        return cudaSuccess;
    // KC x U ~ 16 independent 16-byte loads in flight per lane.
    if (k <= 2)
        return launch_combine_t<2, 4>(T, H, k, y, slot_of, topk_w, out, out_f32, err_word, stream);
    if (k <= 4)
        return launch_combine_t<4, 4>(T, H, k, y, slot_of, topk_w, out, out_f32, err_word, stream);
    return launch_combine_t<8, 2>(T, H, k, y, slot_of, topk_w, out, out_f32, err_word, stream);
}

}  // namespace moe

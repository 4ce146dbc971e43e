// Expert parallelism across real ranks: the receiver's reorder (sm_103a).
//
// UBEP, section 2.3 / Figure 2: each rank's receive region is partitioned by
// source rank and expert, and in Phase 5 the receiver computes offsets from
// the per-expert counts of every source and reorders the tokens contiguously
// per expert; section 4: the receive address space is partitioned in advance.
// StrataCL, Appendix D: the same counts and offsets return the rows on the
// combine path.
//
// After the all-to-all exchange a receiver holds, source by source, each
// source's segment of its own rank-ordered buffer: for source s, its rows for
// local expert 0, then 1, ... (source-major).  The reorder places them
// expert-major: for local expert el, the rows of source 0, then 1, ..., each
// in the source's (token, slot) order.  The combine's return path applies the
// inverse before the reverse exchange.
//
// GPU design.  Every CTA scans the W x El count matrix twice in shared memory
// (source-major and expert-major exclusive prefix sums; at most
// MOE_MAX_EXPERTS segments), then its warps copy (row, chunk) items with
// 16-byte loads and stores (4-byte ones for rows of another size, such as
// the FP8 scale rows), EP_U vectors in flight per lane.  A row's segment
// is found by a binary search over the source-major prefix sums; its
// destination is the segment's expert-major start plus its index inside the
// segment.  One pass over the rows: 2 x rows x row bytes.
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace moe {

constexpr int EP_THREADS = 256;
constexpr int EP_U = 4;  // vectors per lane per item

// VEC is the copy width in bytes: 16 for rows whose size and addresses are
// multiples of 16 (bf16 rows, FP8 codes), 4 otherwise (the FP8 scale rows of
// H / 128 fp32 values).  C is the row size in VEC-byte vectors.
template <int VEC>
__global__ void __launch_bounds__(EP_THREADS)
    ep_reorder_kernel(const int32_t *__restrict__ counts, int W, int El, int64_t rows, int C,
                      int groups, int64_t items, const uint8_t *__restrict__ src,
                      uint8_t *__restrict__ dst, int to_source,
                      int32_t *__restrict__ local_expert_offsets, uint32_t *err_word)
{
    using vec_t = typename std::conditional<VEC == 16, uint4, uint32_t>::type;
    __shared__ int32_t s_off[MOE_MAX_EXPERTS + 1];  // source-major starts, [s*El + el]
    __shared__ int32_t d_off[MOE_MAX_EXPERTS];      // expert-major starts, same index
    __shared__ int ok;
    wait_prior_grid();
    allow_next_grid();
    const int G = W * El;
    if (threadIdx.x < 32) {
        // two exclusive scans over the G segments by one warp: each lane sums
        // a run of ceil(G/32) segments, one warp scan, each lane fills its run
        const int lane = threadIdx.x;
        const int per = (G + 31) / 32;
        const int g0 = lane * per;
        bool bad = false;
        for (int pass = 0; pass < 2; ++pass) {
            // pass 0: segment order g = s*El + el; pass 1: order el*W + s
            auto seg = [&](int o) { return pass == 0 ? o : (o % W) * El + o / W; };
            int32_t sum = 0;
            for (int q = 0; q < per && g0 + q < G; ++q) {
                const int32_t c = ld_nc_s32(counts + seg(g0 + q));
                bad |= c < 0;
                sum += c < 0 ? 0 : c;
            }
            int32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t n = __shfl_up_sync(FULL_MASK, incl, o);
                if (lane >= o)
                    incl += n;
            }
            int32_t run = incl - sum;
            for (int q = 0; q < per && g0 + q < G; ++q) {
                const int g = seg(g0 + q);
                const int32_t c = ld_nc_s32(counts + g);
                (pass == 0 ? s_off : d_off)[g] = run;
                run += c < 0 ? 0 : c;
            }
            if (pass == 0 && lane == 31)
                s_off[G] = incl;
        }
        bad = __any_sync(FULL_MASK, bad);
        if (lane == 0)
            ok = !bad && (int64_t)s_off[G] == rows;
    }
    __syncthreads();
    if (!ok) {
        // counts that are negative or do not add up to `rows`: copy nothing
        if (blockIdx.x == 0 && threadIdx.x == 0)
            report(err_word, MOE_ERRBIT_BAD_INDEX);
        return;
    }
    if (blockIdx.x == 0 && local_expert_offsets != nullptr)
        for (int el = threadIdx.x; el <= El; el += EP_THREADS)
            local_expert_offsets[el] = el < El ? d_off[el] : s_off[G];  // d_off[0*El + el]

    const vec_t *vs = reinterpret_cast<const vec_t *>(src);
    vec_t *vd = reinterpret_cast<vec_t *>(dst);
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (EP_THREADS / 32);
    for (int64_t it = (int64_t)blockIdx.x * (EP_THREADS / 32) + (threadIdx.x >> 5); it < items;
         it += nwarps) {
        const int64_t q = it / groups;  // source-major row
        const int c0 = (int)(it - q * groups) * (32 * EP_U) + lane;
        // the segment holding row q: the last g with s_off[g] <= q (empty
        // segments share their start with the next one, so the last is the
        // one that holds q; s_off[0] = 0 <= q < s_off[G] = rows)
        int lo = 0, hi = G - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_off[mid] <= q)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int64_t f = d_off[lo] + (q - s_off[lo]);  // expert-major row
        const vec_t *from = vs + (to_source ? f : q) * C;
        vec_t *to = vd + (to_source ? q : f) * C;
        vec_t v[EP_U];
#pragma unroll
        for (int u = 0; u < EP_U; ++u)
            if (c0 + u * 32 < C) {
                if constexpr (VEC == 16)
                    v[u] = ld_stream_v4(from + c0 + u * 32);
                else
                    v[u] = (vec_t)ld_nc_s32(reinterpret_cast<const int32_t *>(from + c0 + u * 32));
            }
#pragma unroll
        for (int u = 0; u < EP_U; ++u)
            if (c0 + u * 32 < C) {
                if constexpr (VEC == 16)
                    st_v4(to + c0 + u * 32, v[u]);
                else
                    to[c0 + u * 32] = v[u];
            }
    }
}

template <int VEC>
static cudaError_t launch_ep_reorder_t(int W, int El, int64_t row_bytes, const int32_t *counts,
                                       int64_t rows, const void *src, void *dst, bool to_source,
                                       int32_t *local_expert_offsets, uint32_t *err_word,
                                       cudaStream_t stream)
{
    const int C = (int)(row_bytes / VEC);
    const int groups = (C + 32 * EP_U - 1) / (32 * EP_U);
    const int64_t items = rows * groups;
    const int grid = warp_item_grid((const void *)ep_reorder_kernel<VEC>, EP_THREADS, 0,
                                    items > 0 ? items : 1);
    return launch_pdl(ep_reorder_kernel<VEC>, dim3(grid), dim3(EP_THREADS), 0, stream, counts, W,
                      El, rows, C, groups, items, static_cast<const uint8_t *>(src),
                      static_cast<uint8_t *>(dst), to_source ? 1 : 0, local_expert_offsets,
                      err_word);
}

cudaError_t launch_ep_reorder(int W, int El, int64_t row_bytes, const int32_t *recv_counts,
                              int64_t rows, const void *src, void *dst, bool to_source,
                              int32_t *local_expert_offsets, uint32_t *err_word,
                              cudaStream_t stream)
{
    const bool v16 = row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(dst) & 15) == 0;
    if (v16)
        return launch_ep_reorder_t<16>(W, El, row_bytes, recv_counts, rows, src, dst, to_source,
                                       local_expert_offsets, err_word, stream);
    return launch_ep_reorder_t<4>(W, El, row_bytes, recv_counts, rows, src, dst, to_source,
                                  local_expert_offsets, err_word, stream);
}

}  // namespace moe

// Layout: count -> exclusive scan -> stable slot map (sm_103a).
//
// UBEP, section 2.3 / Figure 2: the dispatch ends with per-expert token counts,
// offsets computed from them, and a contiguous per-expert reorder; StrataCL,
// Appendix D: the placement metadata is destination expert, per-expert counts,
// prefix-sum offsets and token-local offsets.
//
// GPU design.  The (token, slot) pairs i = t*k + j are cut into equal
// contiguous tiles, one per CTA, and each tile into equal warp spans (UBEP
// section 3.3's token-level load partition: loads differ by at most one warp
// step).  Two launches, no cross-CTA waiting:
//   count   each warp builds a private histogram of its span in shared memory
//           (peers found with match.any, one shared-memory add per group of
//           equal experts); the CTA writes its per-expert tile counts.
//   assign  each CTA re-counts its tile, reads the tile-count table to get the
//           global totals (exclusive scan -> expert offsets) and the counts of
//           earlier tiles, turns the per-warp histograms into per-warp cursors,
//           and walks its span again: slot = cursor[e] + rank of the lane among
//           earlier lanes of the same step with the same expert.
// Slots are handed out in pair order inside each warp span, spans in order
// inside a tile, tiles in order: the result is the stable order (expert, t, j)
// independent of scheduling.
#include "common.cuh"
#include "launch.h"

namespace moe {

constexpr int LAYOUT_THREADS = 512;
constexpr int LAYOUT_WARPS = LAYOUT_THREADS / 32;
constexpr int LAYOUT_TARGET_TILE = 4096;  // pairs per CTA while the tile count is small
constexpr int LAYOUT_MAX_TILES = 128;     // bounds the tile-count table each CTA reads
constexpr int LAYOUT_BATCH = 8;           // expert ids loaded ahead per lane

// Out-of-span lanes carry NO_PAIR; pairs with an expert id outside [0, E) carry
// BAD_PAIR (they get slot -1 and take no slot).
constexpr int NO_PAIR = -1;
constexpr int BAD_PAIR = -2;

// Loads the expert ids of up to LAYOUT_BATCH warp steps starting at pair
// `first` (lane-strided), marking pairs past `end` as NO_PAIR.
__device__ __forceinline__ void load_batch(const int32_t *__restrict__ idx, int64_t first,
                                           int64_t end, int E, int lane,
                                           int (&ev)[LAYOUT_BATCH])
{
#pragma unroll
    for (int b = 0; b < LAYOUT_BATCH; ++b) {
        const int64_t i = first + b * 32 + lane;
        int e = NO_PAIR;
        if (i < end) {
            e = ld_nc_s32(idx + i);
            if ((unsigned)e >= (unsigned)E)
                e = BAD_PAIR;
        }
        ev[b] = e;
    }
}

// Per-warp histogram of the pairs [begin, end): wcnt[e] += #pairs with expert e.
// Returns true (on every lane) when an out-of-range expert id was seen.
__device__ __forceinline__ bool warp_histogram(const int32_t *__restrict__ idx, int64_t begin,
                                               int64_t end, int E, int32_t *wcnt)
{
    const int lane = threadIdx.x & 31;
    bool bad = false;
    for (int64_t first = begin; first < end; first += 32 * LAYOUT_BATCH) {
        int ev[LAYOUT_BATCH];
        load_batch(idx, first, end, E, lane, ev);
#pragma unroll
        for (int b = 0; b < LAYOUT_BATCH; ++b) {
            const int e = ev[b];
            bad |= (e == BAD_PAIR);
            const unsigned peers = __match_any_sync(FULL_MASK, e);
            if (e >= 0 && lane == __ffs(peers) - 1)
                wcnt[e] += __popc(peers);
            __syncwarp();
        }
    }
    return __any_sync(FULL_MASK, bad);
}

__global__ void __launch_bounds__(LAYOUT_THREADS)
    layout_count_kernel(const int32_t *__restrict__ idx, int64_t N, int E, int span,
                        int32_t *__restrict__ tile_counts, uint32_t *err_word)
{
    extern __shared__ int32_t smem[];
    int32_t *wcnt = smem;  // [LAYOUT_WARPS][E]
    for (int i = threadIdx.x; i < LAYOUT_WARPS * E; i += LAYOUT_THREADS)
        wcnt[i] = 0;
    __syncthreads();

    const int warp = threadIdx.x >> 5;
    const int64_t begin = ((int64_t)blockIdx.x * LAYOUT_WARPS + warp) * span;
    const int64_t end = min(begin + span, N);
    const bool bad = warp_histogram(idx, begin, end, E, wcnt + warp * E);
    if (bad && (threadIdx.x & 31) == 0)
        report(err_word, MOE_ERRBIT_BAD_INDEX);
    __syncthreads();

    for (int e = threadIdx.x; e < E; e += LAYOUT_THREADS) {
        int32_t s = 0;
#pragma unroll 4
        for (int w = 0; w < LAYOUT_WARPS; ++w)
            s += wcnt[w * E + e];
        tile_counts[(int64_t)blockIdx.x * E + e] = s;
    }
}

__global__ void __launch_bounds__(LAYOUT_THREADS)
    layout_assign_kernel(const int32_t *__restrict__ idx, int64_t N, int E, int R, int span,
                         int tiles, const int32_t *__restrict__ tile_counts,
                         int32_t *__restrict__ expert_counts,
                         int32_t *__restrict__ expert_offsets,
                         int32_t *__restrict__ rank_offsets, int32_t *__restrict__ slot_of,
                         int32_t *__restrict__ src_of)
{
    extern __shared__ int32_t smem[];
    int32_t *wcnt = smem;                     // [LAYOUT_WARPS][E]: counts, then cursors
    int32_t *offs = wcnt + LAYOUT_WARPS * E;  // [E]: totals, then exclusive offsets
    int32_t *pre = offs + E;                  // [E]: pairs of e in earlier tiles
    int32_t *carry = pre + E;                 // [LAYOUT_WARPS]: scan of warp sums

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < LAYOUT_WARPS * E; i += LAYOUT_THREADS)
        wcnt[i] = 0;
    __syncthreads();

    const int64_t begin = ((int64_t)blockIdx.x * LAYOUT_WARPS + warp) * span;
    const int64_t end = min(begin + span, N);
    (void)warp_histogram(idx, begin, end, E, wcnt + warp * E);

    // Column sums of the tile-count table: all tiles, and tiles before this one.
    for (int e = tid; e < E; e += LAYOUT_THREADS) {
        int32_t before = 0, after = 0;
        int b = 0;
#pragma unroll 8
        for (; b < (int)blockIdx.x; ++b)
            before += tile_counts[(int64_t)b * E + e];
#pragma unroll 8
        for (; b < tiles; ++b)
            after += tile_counts[(int64_t)b * E + e];
        offs[e] = before + after;
        pre[e] = before;
    }
    __syncthreads();

    // Exclusive scan of the totals over experts (E <= 2 * LAYOUT_THREADS).
    const int per = (E + LAYOUT_THREADS - 1) / LAYOUT_THREADS;
    int32_t mine[2] = {0, 0};
    int32_t sum = 0;
    for (int q = 0; q < per; ++q) {
        const int e = tid * per + q;
        mine[q] = e < E ? offs[e] : 0;
        sum += mine[q];
    }
    int32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(FULL_MASK, incl, o);
        if (lane >= o)
            incl += n;
    }
    if (lane == 31)
        carry[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int32_t v = lane < LAYOUT_WARPS ? carry[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t n = __shfl_up_sync(FULL_MASK, v, o);
            if (lane >= o)
                v += n;
        }
        if (lane < LAYOUT_WARPS)
            carry[lane] = v;
    }
    __syncthreads();
    const int32_t total = carry[LAYOUT_WARPS - 1];
    int32_t run = incl - sum + (warp > 0 ? carry[warp - 1] : 0);
    for (int q = 0; q < per; ++q) {
        const int e = tid * per + q;
        if (e < E) {
            offs[e] = run;
            if (blockIdx.x == 0) {
                expert_counts[e] = mine[q];
                expert_offsets[e] = run;
            }
        }
        run += mine[q];
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        const int El = E / R;
        for (int r = tid; r <= R; r += LAYOUT_THREADS)
            rank_offsets[r] = r == R ? total : offs[r * El];
        if (tid == 0)
            expert_offsets[E] = total;
    }

    // Per-warp cursors: offset of e + earlier tiles + earlier warps of this tile.
    for (int e = tid; e < E; e += LAYOUT_THREADS) {
        int32_t c = offs[e] + pre[e];
#pragma unroll 4
        for (int w = 0; w < LAYOUT_WARPS; ++w) {
            const int32_t n = wcnt[w * E + e];
            wcnt[w * E + e] = c;
            c += n;
        }
    }
    __syncthreads();

    // Walk the span again and hand out slots in pair order.
    int32_t *cur = wcnt + warp * E;
    const unsigned lt = lanemask_lt();
    for (int64_t first = begin; first < end; first += 32 * LAYOUT_BATCH) {
        int ev[LAYOUT_BATCH];
        load_batch(idx, first, end, E, lane, ev);
#pragma unroll
        for (int b = 0; b < LAYOUT_BATCH; ++b) {
            const int64_t i = first + b * 32 + lane;
            const int e = ev[b];
            const unsigned peers = __match_any_sync(FULL_MASK, e);
            if (e >= 0) {
                const int32_t s = cur[e] + __popc(peers & lt);
                slot_of[i] = s;
                src_of[s] = (int32_t)i;
            } else if (e == BAD_PAIR) {
                slot_of[i] = -1;
            }
            __syncwarp();
            if (e >= 0 && lane == __ffs(peers) - 1)
                cur[e] += __popc(peers);
            __syncwarp();
        }
    }
}

// ---------------------------------------------------------------- host side

struct LayoutPlan {
    int tiles;
    int span;  // pairs per warp, a multiple of 32
};

static LayoutPlan layout_plan(int64_t N)
{
    LayoutPlan p{0, 32};
    if (N <= 0)
        return p;
    int64_t tiles = (N + LAYOUT_TARGET_TILE - 1) / LAYOUT_TARGET_TILE;
    if (tiles > LAYOUT_MAX_TILES)
        tiles = LAYOUT_MAX_TILES;
    const int64_t per_tile = (N + tiles - 1) / tiles;
    int64_t span = (per_tile + LAYOUT_WARPS - 1) / LAYOUT_WARPS;
    span = (span + 31) / 32 * 32;
    const int64_t tile = span * LAYOUT_WARPS;
    p.tiles = (int)((N + tile - 1) / tile);
    p.span = (int)span;
    return p;
}

static size_t count_smem(int E) { return sizeof(int32_t) * (size_t)LAYOUT_WARPS * E; }
static size_t assign_smem(int E)
{
    return sizeof(int32_t) * ((size_t)LAYOUT_WARPS * E + 2 * (size_t)E + LAYOUT_WARPS);
}

size_t layout_workspace_bytes(int64_t N, int E)
{
    const LayoutPlan p = layout_plan(N);
    size_t bytes = sizeof(int32_t) * (size_t)p.tiles * (size_t)E;
    bytes = (bytes + 255) / 256 * 256;
    return bytes < 256 ? 256 : bytes;
}

cudaError_t launch_layout(int T, int k, int E, int R, const int32_t *topk_idx,
                          int32_t *expert_counts, int32_t *expert_offsets,
                          int32_t *rank_offsets, int32_t *slot_of, int32_t *src_of,
                          void *workspace, uint32_t *err_word, cudaStream_t stream)
{
    const int64_t N = (int64_t)T * k;
    if (N == 0) {
        cudaError_t e = cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * E, stream);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (E + 1), stream);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(rank_offsets, 0, sizeof(int32_t) * (R + 1), stream);
        return e;
    }
    const LayoutPlan p = layout_plan(N);
    const size_t sc = count_smem(E), sa = assign_smem(E);
    cudaError_t e = cudaSuccess;
    if (sc > 48 * 1024)
        e = cudaFuncSetAttribute(layout_count_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sc);
    if (e == cudaSuccess && sa > 48 * 1024)
        e = cudaFuncSetAttribute(layout_assign_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sa);
    if (e != cudaSuccess)
        return e;
    int32_t *tile_counts = static_cast<int32_t *>(workspace);
    layout_count_kernel<<<p.tiles, LAYOUT_THREADS, sc, stream>>>(topk_idx, N, E, p.span,
                                                                  tile_counts, err_word);
    layout_assign_kernel<<<p.tiles, LAYOUT_THREADS, sa, stream>>>(
        topk_idx, N, E, R, p.span, p.tiles, tile_counts, expert_counts, expert_offsets,
        rank_offsets, slot_of, src_of);
    return cudaGetLastError();
}

}  // namespace moe

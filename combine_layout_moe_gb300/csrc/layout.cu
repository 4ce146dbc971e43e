// Layout: count -> exclusive scan -> stable slot map (sm_103a).
//
// UBEP, section 2.3 / Figure 2: the dispatch ends with per-expert token counts,
// offsets computed from them, and a contiguous per-expert reorder; StrataCL,
// Appendix D: the placement metadata is destination expert, per-expert counts,
// prefix-sum offsets and token-local offsets.
//
// GPU design.  The (token, slot) pairs i = t*k + j are cut into equal
// contiguous tiles of ~2048 pairs, one per CTA, and each tile into equal warp
// spans (UBEP section 3.3's token-level load partition).  Two launches, no
// CTA ever waits on another:
//   count   each CTA histograms its tile with shared-memory atomics and writes
//           one row of the tile-count table.
//   assign  each CTA histograms its tile again per warp, column-sums the
//           tile-count table (all tiles -> totals -> exclusive scan over
//           experts; earlier tiles -> this tile's base), turns the per-warp
//           histograms into per-warp cursors, and walks its span in order:
//           slot = cursor[e] + number of lower lanes of the same 32-pair step
//           with the same expert.  That peer mask comes from a warp multisplit:
//           one ballot per bit of the expert id (ceil(log2 E) ballots).
// Slots are handed out in pair order within a warp span, spans in order within
// a tile, tiles in order: the stable order (expert, t, j), independent of
// scheduling, with no order-dependent atomics.  Both kernels use programmatic
// dependent launch: assign becomes resident while count runs and does its own
// histogram pass (which needs only topk_idx) before waiting for count's table.
#include "common.cuh"
#include "launch.h"

namespace moe {

constexpr int LAYOUT_THREADS = 512;
constexpr int LAYOUT_WARPS = LAYOUT_THREADS / 32;
constexpr int LAYOUT_TARGET_TILE = 2048;  // pairs per CTA while the tile count is small
constexpr int LAYOUT_MAX_TILES = 128;     // bounds the tile-count table each CTA reads
constexpr int LAYOUT_BATCH = 8;           // expert ids loaded ahead per lane
constexpr int TABLE_UNROLL = 8;           // independent table loads in flight per thread

// Out-of-span lanes carry NO_PAIR; pairs with an expert id outside [0, E) carry
// BAD_PAIR (they get slot -1 and take no slot).
constexpr int NO_PAIR = -1;
constexpr int BAD_PAIR = -2;

// Loads the expert ids of up to LAYOUT_BATCH warp steps starting at pair
// `first` (lane-strided), marking pairs at or past `end` as NO_PAIR.
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

// Lanes of the warp holding the same valid expert id as this lane (this lane
// included when e >= 0): one ballot per bit of the id.
__device__ __forceinline__ unsigned warp_peers(int e, int nbits)
{
    unsigned peers = __ballot_sync(FULL_MASK, e >= 0);
    for (int b = 0; b < nbits; ++b) {
        const bool bit = (e >> b) & 1;
        const unsigned m = __ballot_sync(FULL_MASK, bit);
        peers &= bit ? m : ~m;
    }
    return peers;
}

// hist[e] += number of pairs in [begin, end) routed to e (shared-memory
// atomics; hist may be shared by several warps).  Returns true on every lane
// when an out-of-range expert id was seen.
__device__ __forceinline__ bool histogram(const int32_t *__restrict__ idx, int64_t begin,
                                          int64_t end, int E, int32_t *hist)
{
    const int lane = threadIdx.x & 31;
    bool bad = false;
    for (int64_t first = begin; first < end; first += 32 * LAYOUT_BATCH) {
        int ev[LAYOUT_BATCH];
        load_batch(idx, first, end, E, lane, ev);
#pragma unroll
        for (int b = 0; b < LAYOUT_BATCH; ++b) {
            bad |= ev[b] == BAD_PAIR;
            if (ev[b] >= 0)
                atomicAdd(hist + ev[b], 1);
        }
    }
    return __any_sync(FULL_MASK, bad);
}

__global__ void __launch_bounds__(LAYOUT_THREADS)
    layout_count_kernel(const int32_t *__restrict__ idx, int64_t N, int E, int span,
                        int32_t *__restrict__ tile_counts, uint32_t *err_word)
{
    extern __shared__ int32_t smem[];
    int32_t *hist = smem;  // [E]
    for (int e = threadIdx.x; e < E; e += LAYOUT_THREADS)
        hist[e] = 0;
    wait_prior_grid();
    allow_next_grid();
    __syncthreads();

    const int warp = threadIdx.x >> 5;
    const int64_t begin = ((int64_t)blockIdx.x * LAYOUT_WARPS + warp) * span;
    const int64_t end = min(begin + span, N);
    const bool bad = histogram(idx, begin, end, E, hist);
    if (bad && (threadIdx.x & 31) == 0)
        report(err_word, MOE_ERRBIT_BAD_INDEX);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += LAYOUT_THREADS)
        tile_counts[(int64_t)blockIdx.x * E + e] = hist[e];
}

__global__ void __launch_bounds__(LAYOUT_THREADS)
    layout_assign_kernel(const int32_t *__restrict__ idx, int64_t N, int E, int R, int nbits,
                         int span, int tiles, const int32_t *__restrict__ tile_counts,
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
    for (int i = tid; i < LAYOUT_WARPS * E + 2 * E; i += LAYOUT_THREADS)
        wcnt[i] = 0;
    __syncthreads();

    // The per-warp histogram reads only topk_idx, which was complete before the
    // count kernel let this grid launch (count waits for the producer of
    // topk_idx first), so it runs before the wait for the count kernel and
    // overlaps it.  A span of at most one batch keeps its expert ids in
    // registers for the walk below.
    const int64_t begin = ((int64_t)blockIdx.x * LAYOUT_WARPS + warp) * span;
    const int64_t end = min(begin + span, N);
    const bool cached = end - begin <= 32 * LAYOUT_BATCH;
    int ev0[LAYOUT_BATCH];
    if (cached) {
        load_batch(idx, begin, end, E, lane, ev0);
#pragma unroll
        for (int b = 0; b < LAYOUT_BATCH; ++b)
            if (ev0[b] >= 0)
                atomicAdd(wcnt + warp * E + ev0[b], 1);
    } else {
        (void)histogram(idx, begin, end, E, wcnt + warp * E);
    }
    wait_prior_grid();
    allow_next_grid();

    // Column sums of the tile-count table.  Thread (part, e) sums rows
    // part, part + P, ... so all threads have loads in flight.
    {
        const int P = E >= LAYOUT_THREADS ? 1 : LAYOUT_THREADS / E;
        const int part = tid / E;
        for (int e = tid % E; part < P && e < E; e += LAYOUT_THREADS) {
            int32_t before = 0, total = 0;
            for (int b0 = part; b0 < tiles; b0 += P * TABLE_UNROLL) {
                int32_t v[TABLE_UNROLL];
#pragma unroll
                for (int u = 0; u < TABLE_UNROLL; ++u) {
                    const int b = b0 + u * P;
                    v[u] = b < tiles ? tile_counts[(int64_t)b * E + e] : 0;
                }
#pragma unroll
                for (int u = 0; u < TABLE_UNROLL; ++u) {
                    const int b = b0 + u * P;
                    total += v[u];
                    before += b < (int)blockIdx.x ? v[u] : 0;
                }
            }
            atomicAdd(offs + e, total);
            atomicAdd(pre + e, before);
        }
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
        if (cached) {
#pragma unroll
            for (int b = 0; b < LAYOUT_BATCH; ++b)
                ev[b] = ev0[b];
        } else {
            load_batch(idx, first, end, E, lane, ev);
        }
#pragma unroll
        for (int b = 0; b < LAYOUT_BATCH; ++b) {
            if (first + b * 32 >= end)
                break;  // warp-uniform: the rest of the batch is past the span
            const int64_t i = first + b * 32 + lane;
            const int e = ev[b];
            const unsigned peers = warp_peers(e, nbits);
            if (e >= 0) {
                const int32_t s = cur[e] + __popc(peers & lt);
                slot_of[i] = s;
                src_of[s] = (int32_t)i;
            } else if (e == BAD_PAIR) {
                slot_of[i] = -1;
            }
            __syncwarp();
            if (e >= 0 && (peers & lt) == 0)
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

static size_t count_smem(int E) { return sizeof(int32_t) * (size_t)E; }
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
    int nbits = 0;
    while ((1 << nbits) < E)
        ++nbits;
    cudaError_t e = cudaSuccess;
    if (sa > 48 * 1024)
        e = cudaFuncSetAttribute(layout_assign_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sa);
    if (e != cudaSuccess)
        return e;
    int32_t *tile_counts = static_cast<int32_t *>(workspace);
    e = launch_pdl(layout_count_kernel, dim3(p.tiles), dim3(LAYOUT_THREADS), sc, stream,
                   topk_idx, N, E, p.span, tile_counts, err_word);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(layout_assign_kernel, dim3(p.tiles), dim3(LAYOUT_THREADS), sa, stream,
                      topk_idx, N, E, R, nbits, p.span, p.tiles, tile_counts, expert_counts,
                      expert_offsets, rank_offsets, slot_of, src_of);
}

}  // namespace moe

// Layout: count -> exclusive scan -> stable slot map (sm_103a).
//
// UBEP, section 2.3 / Figure 2: the dispatch ends with per-expert token counts,
// offsets computed from them, and a contiguous per-expert reorder; StrataCL,
// Appendix D: the placement metadata is destination expert, per-expert counts,
// prefix-sum offsets and token-local offsets.
//
// GPU design: one launch, one 512-thread CTA per tile.  The (token, slot)
// pairs i = t*k + j are cut into equal contiguous tiles of about 1024 pairs
// (at most LAYOUT_MAX_TILES tiles), and each tile into equal warp spans (UBEP
// section 3.3's token-level load partition).
//   1. Each warp histograms its span into a private shared-memory row (the
//      expert ids stay in registers); the CTA sums the rows into its tile's
//      counts.
//   2. The tiles' counts are exchanged.  One tile needs no exchange.  Up to
//      CLUSTER_MAX_TILES (16) tiles the grid is one thread-block cluster
//      (sizes above 8 only where the GPU can place one): each CTA keeps its
//      counts in shared memory, a hardware cluster barrier publishes them, and
//      step 3 reads the other CTAs' counts through distributed shared memory
//      (no table in global memory, no atomics, no polling).  Beyond that the
//      launch is cooperative: the counts go to a tile-count table in the
//      workspace and a grid barrier (arrival count and generation in the
//      workspace head, time-bounded) follows.
//   3. Each CTA column-sums the counts (all tiles -> totals -> exclusive scan
//      over experts; earlier tiles -> this tile's base), turns the per-warp
//      histograms into per-warp cursors, and walks its span in order:
//      slot = cursor[e] + number of lower lanes of the same 32-pair step with
//      the same expert.  That peer mask comes from a warp multisplit: one
//      ballot per bit of the expert id (ceil(log2 E) ballots).
// Slots are handed out in pair order within a warp span, spans in order within
// a tile, tiles in order: the stable order (expert, t, j), independent of
// scheduling, with no order-dependent atomics.
#include "common.cuh"
#include "launch.h"
#include "grid_sync.cuh"
#include "tma.cuh"

namespace moe {

constexpr int LAYOUT_THREADS = 512;
constexpr int LAYOUT_WARPS = LAYOUT_THREADS / 32;
// Tunable (compile-time; the default is the shipped configuration).
#ifndef MOE_LAYOUT_TARGET_TILE
#define MOE_LAYOUT_TARGET_TILE 1024
#endif
constexpr int LAYOUT_TARGET_TILE = MOE_LAYOUT_TARGET_TILE;  // pairs per CTA while tiles are few
constexpr int LAYOUT_MAX_TILES = 128;     // bounds the tile-count table each CTA reads
constexpr int LAYOUT_BATCH = 8;           // expert ids loaded ahead per lane
#ifndef MOE_LAYOUT_TABLE_UNROLL
#define MOE_LAYOUT_TABLE_UNROLL 8
#endif
constexpr int TABLE_UNROLL = MOE_LAYOUT_TABLE_UNROLL;  // independent table loads in flight per thread
constexpr size_t LAYOUT_BARRIER_BYTES = 256;  // workspace head: grid-barrier count and generation
constexpr int CLUSTER_MAX_TILES = 16;         // largest cluster (non-portable beyond 8)
constexpr int CLUSTER_PORTABLE = 8;           // cluster sizes every sm_90+ GPU accepts

// Thread-block cluster barrier, split into its arrive (release) and wait
// (acquire) halves; every thread of every CTA of the cluster takes part.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// 32-bit load from the shared memory of CTA `rank` of this cluster, at the
// offset that `local` (a shared-memory address of this CTA) has here.
__device__ __forceinline__ int32_t ld_dsmem_s32(uint32_t local, uint32_t rank)
{
    uint32_t remote;
    int32_t v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
    return v;
}

// Out-of-span lanes carry NO_PAIR; pairs with an expert id outside [0, E) carry
// BAD_PAIR (they get slot -1 and take no slot).  With COAL, a pair whose rank
// an earlier slot j' of its token already chose carries SHARED_PAIR - j': it
// takes no row of its own and shares slot j''s.
constexpr int NO_PAIR = -1;
constexpr int BAD_PAIR = -2;
constexpr int SHARED_PAIR = -3;

// Key of pair i: its expert id, or (COAL) its destination rank when it is the
// first slot of its token that chose that rank (else SHARED_PAIR - that
// slot).  Ids outside [0, E) give BAD_PAIR.
template <bool COAL>
__device__ __forceinline__ int pair_key(const int32_t *__restrict__ idx, int64_t i, int E, int El,
                                        int k)
{
    const int e = ld_nc_s32(idx + i);
    if ((unsigned)e >= (unsigned)E)
        return BAD_PAIR;
    if (!COAL)
        return e;
    const int r = e / El;
    const int j = (int)(i % k);
    for (int jj = 0; jj < j; ++jj) {
        const int e2 = ld_nc_s32(idx + i - j + jj);
        if ((unsigned)e2 < (unsigned)E && e2 / El == r)
            return SHARED_PAIR - jj;
    }
    return r;
}

// Loads the keys of up to LAYOUT_BATCH warp steps starting at pair `first`
// (lane-strided), marking pairs at or past `end` as NO_PAIR.
template <bool COAL>
__device__ __forceinline__ void load_batch(const int32_t *__restrict__ idx, int64_t first,
                                           int64_t end, int E, int El, int k, int lane,
                                           int (&ev)[LAYOUT_BATCH])
{
#pragma unroll
    for (int b = 0; b < LAYOUT_BATCH; ++b) {
        const int64_t i = first + b * 32 + lane;
        ev[b] = i < end ? pair_key<COAL>(idx, i, E, El, k) : NO_PAIR;
    }
}

// Lanes of the warp holding the same valid expert id as this lane (this lane
// included when e >= 0): one ballot per bit of the id (NBITS = ceil(log2 E)).
template <int NBITS>
__device__ __forceinline__ unsigned warp_peers(int e)
{
    unsigned peers = __ballot_sync(FULL_MASK, e >= 0);
#pragma unroll
    for (int b = 0; b < NBITS; ++b) {
        const bool bit = (e >> b) & 1;
        const unsigned m = __ballot_sync(FULL_MASK, bit);
        peers &= bit ? m : ~m;
    }
    return peers;
}

// Phase timestamps for tuning builds (-DMOE_TRACE): CTA 0 stores %globaltimer
// at each phase boundary into the 64-bit words that follow the error word.
#ifdef MOE_TRACE
#define LAYOUT_TRACE(n)                                                                \
    do {                                                                               \
        __syncthreads();                                                               \
        if (blockIdx.x == 0 && threadIdx.x == 0 && err_word)                            \
            reinterpret_cast<unsigned long long *>(err_word)[8 + (n)] = global_ns();   \
    } while (0)
#else
#define LAYOUT_TRACE(n) \
    do {                \
    } while (0)
#endif

// Keys: expert ids (K = E), or with COAL destination ranks of owner pairs
// (K = R); e_real and El are the expert count and experts per rank.
template <int NBITS, bool COAL>
__global__ void __launch_bounds__(LAYOUT_THREADS)
    layout_kernel(const int32_t *__restrict__ idx, int64_t N, int E, int R, int e_real, int El,
                  int k, int span,
                  int tiles, int cluster, unsigned *barrier, int32_t *tile_counts,
                  int32_t *__restrict__ expert_counts, int32_t *__restrict__ expert_offsets,
                  int32_t *__restrict__ rank_offsets, int32_t *__restrict__ slot_of,
                  int32_t *__restrict__ src_of, const int32_t *__restrict__ plain_slot,
                  int32_t *__restrict__ expand, uint32_t *err_word)
{
    extern __shared__ int32_t smem[];
    int32_t *wcnt = smem;                     // [LAYOUT_WARPS][E]: counts, then cursors
    int32_t *offs = wcnt + LAYOUT_WARPS * E;  // [E]: totals, then exclusive offsets
    int32_t *pre = offs + E;                  // [E]: pairs of e in earlier tiles
    int32_t *carry = pre + E;                 // [LAYOUT_WARPS]: scan of warp sums
    int32_t *tsum = carry + LAYOUT_WARPS;     // [E]: this tile's counts (cluster path)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < LAYOUT_WARPS * E + 2 * E; i += LAYOUT_THREADS)
        wcnt[i] = 0;
    wait_prior_grid();
    allow_next_grid();
    __syncthreads();
    LAYOUT_TRACE(0);

    // 1. per-warp histograms of this tile; the ids of a span of at most one
    //    batch stay in registers for the walk
    const int64_t begin = ((int64_t)blockIdx.x * LAYOUT_WARPS + warp) * span;
    const int64_t end = min(begin + span, N);
    const bool cached = end - begin <= 32 * LAYOUT_BATCH;
    int ev0[LAYOUT_BATCH];
#pragma unroll
    for (int b = 0; b < LAYOUT_BATCH; ++b)
        ev0[b] = NO_PAIR;
    bool bad = false;
    for (int64_t first = begin; first < end; first += 32 * LAYOUT_BATCH) {
        int ev[LAYOUT_BATCH];
        load_batch<COAL>(idx, first, end, e_real, El, k, lane, ev);
#pragma unroll
        for (int b = 0; b < LAYOUT_BATCH; ++b) {
            bad |= ev[b] == BAD_PAIR;
            if (ev[b] >= 0)
                atomicAdd(wcnt + warp * E + ev[b], 1);
            ev0[b] = ev[b];
        }
    }
    if (__any_sync(FULL_MASK, bad) && lane == 0)
        report(err_word, MOE_ERRBIT_BAD_INDEX);
    __syncthreads();
    LAYOUT_TRACE(1);
    if (tiles == 1) {
        // one tile: the totals are this CTA's own counts, and no tile comes
        // before it (pre stays 0); no table, no grid barrier
        for (int e = tid; e < E; e += LAYOUT_THREADS) {
            int32_t s = 0;
#pragma unroll 4
            for (int w = 0; w < LAYOUT_WARPS; ++w)
                s += wcnt[w * E + e];
            offs[e] = s;
        }
        LAYOUT_TRACE(2);
        LAYOUT_TRACE(3);
    } else {
        for (int e = tid; e < E; e += LAYOUT_THREADS) {
            int32_t s = 0;
#pragma unroll 4
            for (int w = 0; w < LAYOUT_WARPS; ++w)
                s += wcnt[w * E + e];
            if (cluster)
                tsum[e] = s;
            else
                tile_counts[(int64_t)blockIdx.x * E + e] = s;
        }

        LAYOUT_TRACE(2);
        // 2. every tile row is written
        if (cluster) {
            cluster_arrive();
            cluster_wait();
        } else if (!grid_barrier(barrier, err_word)) {
            return;
        }
        LAYOUT_TRACE(3);
    }

    // 3a. column sums of the table; thread (part, e) sums rows part, part+P, ...
    if (tiles > 1 && cluster) {
        // the rows are the cluster's tsum arrays (CTA rank = tile); only ranks
        // that exist are read, and a cluster of another size is reported
        uint32_t ncta;
        asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncta));
        const int nread = min(tiles, (int)ncta);
        if (tid == 0 && (int)ncta != tiles)
            report(err_word, MOE_ERRBIT_LAUNCH);
        for (int e = tid; e < E; e += LAYOUT_THREADS) {
            const uint32_t la = smem_addr(tsum + e);
            int32_t before = 0, total = 0;
            for (int b0 = 0; b0 < nread; b0 += CLUSTER_PORTABLE) {
                int32_t v[CLUSTER_PORTABLE];
#pragma unroll
                for (int q = 0; q < CLUSTER_PORTABLE; ++q)  // eight remote loads in flight at once
                    v[q] = b0 + q < nread ? ld_dsmem_s32(la, (uint32_t)(b0 + q)) : 0;
#pragma unroll
                for (int q = 0; q < CLUSTER_PORTABLE; ++q) {
                    total += v[q];
                    before += b0 + q < (int)blockIdx.x ? v[q] : 0;
                }
            }
            offs[e] = total;
            pre[e] = before;
        }
        cluster_arrive();  // done reading the other CTAs' shared memory
        if ((int)ncta != tiles) {
            // a cluster of another size: the sums are partial, so write no
            // offsets or slots; still wait, so that no CTA leaves while
            // another may read its tsum
            cluster_wait();
            return;
        }
    } else if (tiles > 1) {
        const int P = E >= LAYOUT_THREADS ? 1 : LAYOUT_THREADS / E;
        const int part = tid / E;
        for (int e = tid % E; part < P && e < E; e += LAYOUT_THREADS) {
            int32_t before = 0, total = 0;
            for (int b0 = part; b0 < tiles; b0 += P * TABLE_UNROLL) {
                int32_t v[TABLE_UNROLL];
#pragma unroll
                for (int u = 0; u < TABLE_UNROLL; ++u) {
                    const int b = b0 + u * P;
                    v[u] = b < tiles ? __ldcg(tile_counts + (int64_t)b * E + e) : 0;
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
    LAYOUT_TRACE(4);

    // 3b. exclusive scan of the totals over experts, by warp 0 alone: each lane
    //     sums a run of ceil(E/32) experts, one warp scan, each lane writes
    //     its run's offsets (E <= MOE_MAX_EXPERTS = 1024)
    if (warp == 0) {
        const int per = (E + 31) / 32;
        const int e0 = lane * per;
        int32_t sum = 0;
        for (int q = 0; q < per; ++q)
            sum += e0 + q < E ? offs[e0 + q] : 0;
        int32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t n = __shfl_up_sync(FULL_MASK, incl, o);
            if (lane >= o)
                incl += n;
        }
        int32_t run = incl - sum;
        for (int q = 0; q < per && e0 + q < E; ++q) {
            const int e = e0 + q;
            const int32_t cnt = offs[e];
            offs[e] = run;
            if (blockIdx.x == 0) {
                expert_counts[e] = cnt;
                expert_offsets[e] = run;
            }
            run += cnt;
        }
        if (lane == 31)
            carry[0] = incl;
    }
    __syncthreads();
    const int32_t total = carry[0];
    if (blockIdx.x == 0) {
        if (rank_offsets) {
            const int Kl = E / R;
            for (int r = tid; r <= R; r += LAYOUT_THREADS)
                rank_offsets[r] = r == R ? total : offs[r * Kl];
        }
        if (tid == 0)
            expert_offsets[E] = total;
    }

    LAYOUT_TRACE(5);
    // 3c. per-warp cursors: offset of e + earlier tiles + earlier warps here
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

    LAYOUT_TRACE(6);
    // 3d. walk the span again and hand out slots in pair order
    int32_t *cur = wcnt + warp * E;
    const unsigned lt = lanemask_lt();
    for (int64_t first = begin; first < end; first += 32 * LAYOUT_BATCH) {
        int ev[LAYOUT_BATCH];
        if (cached) {
#pragma unroll
            for (int b = 0; b < LAYOUT_BATCH; ++b)
                ev[b] = ev0[b];
        } else {
            load_batch<COAL>(idx, first, end, e_real, El, k, lane, ev);
        }
#pragma unroll
        for (int b = 0; b < LAYOUT_BATCH; ++b) {
            if (first + b * 32 >= end)
                break;  // warp-uniform: the rest of the batch is past the span
            const int64_t i = first + b * 32 + lane;
            const int e = ev[b];
            const unsigned peers = warp_peers<NBITS>(e);
            int32_t s = -1;
            if (e >= 0) {
                s = cur[e] + __popc(peers & lt);
                slot_of[i] = s;
                src_of[s] = (int32_t)i;
                if (COAL && plain_slot != nullptr) {
                    // an owner maps its plain slot to its own row here; the
                    // shared pairs do it below, after the shuffle
                    const int32_t ps = ld_nc_s32(plain_slot + i);
                    if ((unsigned)ps < (unsigned)N)
                        expand[ps] = s;
                }
            } else if (e == BAD_PAIR) {
                slot_of[i] = -1;
            }
            if (COAL && plain_slot != nullptr) {
                // k divides 32, so this step starts a token and holds whole
                // tokens: a shared pair takes its row from the lane of the
                // slot that owns it and maps its plain slot to that row
                const int j = lane % k;
                const int oj = e <= SHARED_PAIR ? SHARED_PAIR - e : j;
                const int32_t c = __shfl_sync(FULL_MASK, s, lane - j + oj);
                if (e <= SHARED_PAIR) {
                    slot_of[i] = c;
                    const int32_t ps = ld_nc_s32(plain_slot + i);
                    if ((unsigned)ps < (unsigned)N)
                        expand[ps] = c;
                }
            }
            __syncwarp();
            if (e >= 0 && (peers & lt) == 0)
                cur[e] += __popc(peers);
            __syncwarp();
        }
    }
    LAYOUT_TRACE(7);
    if (tiles > 1 && cluster)
        cluster_wait();  // no CTA leaves while another may still read its tsum
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

static size_t layout_smem(int E)
{
    return sizeof(int32_t) * ((size_t)LAYOUT_WARPS * E + 3 * (size_t)E + LAYOUT_WARPS);
}

size_t layout_workspace_bytes(int64_t N, int E)
{
    const LayoutPlan p = layout_plan(N);
    size_t bytes = sizeof(int32_t) * (size_t)p.tiles * (size_t)E;
    bytes = (bytes + 255) / 256 * 256;
    return LAYOUT_BARRIER_BYTES + bytes;
}

// The form of the layout kernel that this host thread launched last
// (MOE_LAYOUT_FORM_*), for moe_layout_last_form().
static thread_local int g_last_form = MOE_LAYOUT_FORM_NONE;

void note_layout_form(int form) { g_last_form = form; }

template <int NBITS, bool COAL>
static cudaError_t launch_layout_t(int64_t N, int E, int R, int e_real, int El, int k,
                                   const LayoutPlan &p,
                                   const int32_t *topk_idx, unsigned *barrier,
                                   int32_t *tile_counts, int32_t *expert_counts,
                                   int32_t *expert_offsets, int32_t *rank_offsets,
                                   int32_t *slot_of, int32_t *src_of, const int32_t *plain_slot,
                                   int32_t *expand, uint32_t *err_word, bool clear_barrier,
                                   cudaStream_t stream)
{
    const size_t smem = layout_smem(E);
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024)
        e = cudaFuncSetAttribute(layout_kernel<NBITS, COAL>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    // One cluster (at most CLUSTER_MAX_TILES CTAs): the cluster barrier and
    // distributed shared memory replace the table and the grid barrier.
    // Otherwise cooperative: all CTAs are co-resident, as the grid barrier
    // requires.  Either way with programmatic serialisation: the grid may
    // become resident while the previous kernel in the stream finishes.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.tiles);
    cfg.blockDim = dim3(LAYOUT_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    auto launch = [&](int cluster, int nattr) {
        cfg.numAttrs = nattr;
        return cudaLaunchKernelEx(&cfg, layout_kernel<NBITS, COAL>, topk_idx, N, E, R, e_real,
                                  El, k, p.span, p.tiles, cluster, barrier, tile_counts,
                                  expert_counts, expert_offsets, rank_offsets, slot_of, src_of,
                                  plain_slot, expand, err_word);
    };
    if (p.tiles > 1 && p.tiles <= CLUSTER_MAX_TILES) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)p.tiles;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        bool fits = true;
        if (p.tiles > CLUSTER_PORTABLE) {
            // a non-portable size: allowed explicitly, and used only if the
            // GPU can place one such cluster of these CTAs
            int nclusters = 0;
            cfg.numAttrs = 1;
            fits = cudaFuncSetAttribute(layout_kernel<NBITS, COAL>,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed,
                                        1) == cudaSuccess &&
                   cudaOccupancyMaxActiveClusters(&nclusters, layout_kernel<NBITS, COAL>,
                                                  &cfg) == cudaSuccess &&
                   nclusters >= 1;
            if (!fits)
                (void)cudaGetLastError();
        }
        if (fits) {
            e = launch(1, 2);
            if (e != cudaSuccess) {
                (void)cudaGetLastError();
                e = launch(1, 1);  // without the programmatic attribute
            }
            if (e == cudaSuccess) {
                note_layout_form(MOE_LAYOUT_FORM_CLUSTER);
                return e;
            }
            (void)cudaGetLastError();  // no cluster of this size: the cooperative form below
        }
    }
    if (clear_barrier && p.tiles > 1) {
        // only the grid-barrier form reads the barrier head: a caller that
        // cannot vouch for it being zero has it cleared here, on the stream
        e = cudaMemsetAsync(barrier, 0, 8, stream);
        if (e != cudaSuccess)
            return e;
    }
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    e = launch(0, 2);
    if (e == cudaErrorInvalidValue || e == cudaErrorNotSupported) {
        // the driver refused the attribute pair: launch cooperatively only
        (void)cudaGetLastError();
        e = launch(0, 1);
    }
    if (e == cudaSuccess)
        note_layout_form(p.tiles == 1 ? MOE_LAYOUT_FORM_SINGLE : MOE_LAYOUT_FORM_COOPERATIVE);
    return e;
}

// Count / scan / slot map over keys in [0, K): expert ids (COAL false) or the
// destination ranks of owner pairs (COAL true; with plain_slot, the shared
// pairs and the expand map are resolved in the same launch).
template <bool COAL>
static cudaError_t launch_keys(int T, int k, int K, int R, int e_real, int El,
                               const int32_t *topk_idx, int32_t *counts, int32_t *offsets,
                               int32_t *rank_offsets, int32_t *slot_of, int32_t *src_of,
                               const int32_t *plain_slot, int32_t *expand, void *workspace,
                               uint32_t *err_word, bool clear_barrier, cudaStream_t stream)
{
    const int64_t N = (int64_t)T * k;
    if (N == 0) {
        note_layout_form(MOE_LAYOUT_FORM_NONE);
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * K, stream);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (K + 1), stream);
        if (e == cudaSuccess && rank_offsets)
            e = cudaMemsetAsync(rank_offsets, 0, sizeof(int32_t) * (R + 1), stream);
        return e;
    }
    const LayoutPlan p = layout_plan(N);
    int nbits = 0;
    while ((1 << nbits) < K)
        ++nbits;
    unsigned *barrier = static_cast<unsigned *>(workspace);
    int32_t *tile_counts = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(workspace) +
                                                       LAYOUT_BARRIER_BYTES);
    switch (nbits) {
#define MOE_LAYOUT_CASE(B)                                                                     \
    case B:                                                                                    \
        return launch_layout_t<B, COAL>(N, K, R, e_real, El, k, p, topk_idx, barrier,          \
                                        tile_counts, counts, offsets, rank_offsets, slot_of,   \
                                        src_of, plain_slot, expand, err_word,          \
                                        clear_barrier, stream);
        MOE_LAYOUT_CASE(0)
        MOE_LAYOUT_CASE(1)
        MOE_LAYOUT_CASE(2)
        MOE_LAYOUT_CASE(3)
        MOE_LAYOUT_CASE(4)
        MOE_LAYOUT_CASE(5)
        MOE_LAYOUT_CASE(6)
        MOE_LAYOUT_CASE(7)
        MOE_LAYOUT_CASE(8)
        MOE_LAYOUT_CASE(9)
        MOE_LAYOUT_CASE(10)
#undef MOE_LAYOUT_CASE
    default:
        return cudaErrorInvalidValue;
    }
}

cudaError_t launch_layout(int T, int k, int E, int R, const int32_t *topk_idx,
                          int32_t *expert_counts, int32_t *expert_offsets,
                          int32_t *rank_offsets, int32_t *slot_of, int32_t *src_of,
                          void *workspace, uint32_t *err_word, cudaStream_t stream,
                          bool clear_barrier)
{
    return launch_keys<false>(T, k, E, R, E, E / R, topk_idx, expert_counts, expert_offsets,
                              rank_offsets, slot_of, src_of, nullptr, nullptr, workspace,
                              err_word, clear_barrier, stream);
}

// Non-owner slots take their owner's coalesced row; expand[slot_of[i]] = crow[i].
__global__ void coalesce_finish_kernel(const int32_t *__restrict__ idx,
                                       const int32_t *__restrict__ slot_of, int32_t *crow,
                                       int32_t *__restrict__ expand, int64_t N, int E, int El,
                                       int k)
{
    wait_prior_grid();
    allow_next_grid();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < N;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int e = ld_nc_s32(idx + i);
        if ((unsigned)e >= (unsigned)E)
            continue;
        const int r = e / El;
        const int j = (int)(i % k);
        int owner = j;
        for (int jj = 0; jj < j; ++jj) {
            const int e2 = ld_nc_s32(idx + i - j + jj);
            if ((unsigned)e2 < (unsigned)E && e2 / El == r) {
                owner = jj;
                break;
            }
        }
        const int32_t c = owner == j ? crow[i] : crow[i - j + owner];
        if (owner != j)
            crow[i] = c;
        const int32_t s = ld_nc_s32(slot_of + i);
        if ((unsigned)s < (unsigned)N)
            expand[s] = c;
    }
}

cudaError_t launch_layout_coalesced(int T, int k, int E, int R, const int32_t *topk_idx,
                                    const int32_t *slot_of, int32_t *rank_counts_c,
                                    int32_t *rank_offsets_c, int32_t *crow, int32_t *src_pair_c,
                                    int32_t *expand, void *workspace, uint32_t *err_word,
                                    cudaStream_t stream)
{
    // When k divides 32 every 32-pair warp step holds whole tokens, and the
    // layout kernel resolves shared pairs and the expand map itself;
    // otherwise a second pass does.
    const bool fused = 32 % k == 0;
    cudaError_t e = launch_keys<true>(T, k, R, R, E, E / R, topk_idx, rank_counts_c,
                                      rank_offsets_c, nullptr, crow, src_pair_c,
                                      fused ? slot_of : nullptr, fused ? expand : nullptr,
                                      workspace, err_word, false, stream);
    const int64_t N = (int64_t)T * k;
    if (e != cudaSuccess || N == 0 || fused)
        return e;
    const int threads = 256;
    int64_t blocks = (N + threads - 1) / threads;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap)
        blocks = cap;
    return launch_pdl(coalesce_finish_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
                      topk_idx, slot_of, crow, expand, N, E, E / R, k);
}

}  // namespace moe

extern "C" MOE_API int moe_layout_last_form(void) { return moe::g_last_form; }

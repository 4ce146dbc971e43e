// Dispatch: scatter token rows into the packed, rank-segmented, expert-contiguous
// receive buffer (sm_103a).
//
// UBEP, section 2.3 (Phase 2: each token goes to every expert it chose) and
// section 4 (senders write straight into the pre-partitioned receive region);
// RailWave, section 3.2 (payload packed without padding).  The FP8 variant is
// in dispatch_quant.cu.
//
// GPU design.  The work item is one warp on one (token, row chunk): the warp
// reads 32 x U 16-byte vectors of the token's row (U loads in flight per lane,
// 512 contiguous bytes per warp instruction), then stores them to the k
// destination rows, each store again 512 contiguous bytes.  The row is read
// from HBM once and written k times; slot indices are read once per item by
// lanes 0..k-1 and broadcast with shuffles.  The grid is capped at the number
// of co-resident CTAs and strides over items.
#include "common.cuh"
#include "launch.h"
#include "tma.cuh"
#include "sched.cuh"

namespace moe {

#ifndef MOE_DB_STAGES
#define MOE_DB_STAGES 4
#endif
#ifndef MOE_DB_CHUNK
#define MOE_DB_CHUNK 8192
#endif
constexpr int DB_STAGES = MOE_DB_STAGES;  // row chunks in flight per pipe
constexpr int DB_CHUNK = MOE_DB_CHUNK;    // bytes per bulk copy (last chunk of a row may be shorter)
#ifndef MOE_DB_STATIC_PCT
#define MOE_DB_STATIC_PCT 50
#endif
#ifndef MOE_DB_GRAB
#define MOE_DB_GRAB 1
#endif
#ifndef MOE_DB_DYN_MIN
#define MOE_DB_DYN_MIN 8
#endif
constexpr int DB_STATIC_PCT = MOE_DB_STATIC_PCT;  // share of the units split statically
constexpr int DB_GRAB = MOE_DB_GRAB;              // units per draw from the pool
constexpr int DB_DYN_MIN = MOE_DB_DYN_MIN;        // below this many units per CTA: no pool
static_assert(DB_STAGES >= 2 && DB_STAGES <= 16, "stage ring size");

// bf16 dispatch through bulk copies.  Each CTA is one warp driving one
// pipeline over units (unit = token t, chunk c of its row): lane 0 loads the
// chunk into a ring of shared-memory stages with one cp.async.bulk
// (completion on the stage's mbarrier); once it has landed, lanes 0..k-1 each
// store it to their destination row with one shared -> global cp.async.bulk.
// A stage is refilled only after every lane's stores from it have finished
// reading shared memory (bulk async-group accounting: every lane commits one
// group per unit, possibly empty).  The row is read from HBM once and written
// k times with no per-element instructions.
//
// Units: each CTA first takes `per_cta` consecutive units of its own, then
// draws `grab` consecutive units at a time from the pool of the rest (the
// scheduling slot `sched_slot` of the launch; see sched.cuh).  With
// sched_slot < 0 there is no pool: CTA b takes units [units*b/G,
// units*(b+1)/G) of G CTAs.  The stage ring records the unit each stage
// holds.
//
// COAL: rows go to the rank-coalesced buffer (one row per token and distinct
// destination rank).  slot_of is then the coalesced row map, where every slot
// of a token on one rank names the same row; only the lowest such slot
// stores it, so each row is written once.  `rows` bounds the row indices.
//
// prefetch_x: the first stages' loads of x are issued before waiting on the
// previous grid.  Only for a launch whose previous grid is this library's
// layout kernel: that kernel lets dependents launch only after its own wait,
// so x (written before the layout) is final, and only slot_of is not.
__device__ SchedSlot g_dispatch_sched[SCHED_SLOTS];
static std::atomic<unsigned> g_dispatch_seq{0};

template <bool COAL>
__global__ void __launch_bounds__(32)
    dispatch_bulk_kernel(const uint8_t *__restrict__ x, const int32_t *__restrict__ slot_of,
                         uint8_t *__restrict__ recv, int T, int k, int64_t rowbytes, int CH,
                         int nchunks, int64_t units, int64_t per_cta, int grab, int sched_slot,
                         int rows, int prefetch_x, uint32_t *err_word)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int64_t stage_unit[DB_STAGES];
    const uint32_t bars = smem_addr(smem);
    const uint32_t stages = bars + 128;
    auto full = [&](int s) { return bars + 8u * s; };
    const int lane = threadIdx.x;

    if (lane == 0) {
        for (int s = 0; s < DB_STAGES; ++s)
            mbar_init(full(s), 1);
        mbar_fence_init();
    }
    __syncwarp();

    // the unit source (warp-uniform): this CTA's range, then draws from the
    // pool [per_cta * gridDim.x, units); a draw is requested as soon as the
    // current range is used up, so it travels while the last unit loads
    const bool pooled = sched_slot >= 0;
    SchedSlot *sched = g_dispatch_sched + (pooled ? sched_slot : 0);
    const int64_t pool0 = pooled ? per_cta * gridDim.x : units;
    int64_t r_cur = pooled ? per_cta * blockIdx.x : units * blockIdx.x / gridDim.x;
    int64_t r_end = pooled ? r_cur + per_cta : units * (blockIdx.x + 1) / gridDim.x;
    unsigned long long drawn = 0;  // lane 0: the pending draw's pool offset
    bool pending = false, dry = pool0 >= units;
    auto request = [&]() {
        if (lane == 0)
            drawn = atomicAdd(&sched->taken, (unsigned long long)grab);
        pending = true;
    };
    auto next_unit = [&]() -> int64_t {
        if (r_cur == r_end) {
            if (dry)
                return -1;
            if (!pending)
                request();
            const int64_t v = pool0 + (int64_t)__shfl_sync(FULL_MASK, drawn, 0);
            pending = false;
            if (v >= units) {
                dry = true;
                return -1;
            }
            r_cur = v;
            r_end = min(v + (int64_t)grab, units);
        }
        const int64_t u = r_cur++;
        if (r_cur == r_end && !dry)
            request();
        return u;
    };

    // load side (the whole warp runs it; lane 0 issues the copy)
    int64_t loaded = 0;
    bool more = true;
    auto issue_load = [&]() {
        const int64_t u = next_unit();
        if (u < 0) {
            more = false;
            return;
        }
        const int s = (int)(loaded % DB_STAGES);
        const int64_t lt = u / nchunks;
        const int lc = (int)(u - lt * nchunks);
        const uint32_t cb = (uint32_t)min((int64_t)CH, rowbytes - (int64_t)lc * CH);
        if (lane == 0) {
            stage_unit[s] = u;
            mbar_arrive_expect_tx(full(s), cb);
            bulk_g2s(stages + (uint32_t)s * CH, x + lt * rowbytes + (int64_t)lc * CH, cb, full(s));
        }
        ++loaded;
        __syncwarp();  // stage_unit[s] is visible to every lane
    };
    if (prefetch_x) {
        while (more && loaded < DB_STAGES)
            issue_load();
    }
    wait_prior_grid();
    allow_next_grid();
    while (more && loaded < DB_STAGES)
        issue_load();

    // store side: a lane stores its slot's row unless (COAL) a lower slot of
    // the token names the same row; the slots of the next unit's token are
    // requested one unit ahead
    const bool kl = lane < k;
    const unsigned kmask = k >= 32 ? FULL_MASK : (1u << k) - 1u;
    auto first_of_row = [&](int32_t v) {
        if (!COAL)
            return kl;
        const unsigned same = __match_any_sync(FULL_MASK, v) & kmask;
        return kl && (same & lanemask_lt()) == 0;
    };
    int64_t cur_t = -1, nxt_t = -1;
    int32_t cur = 0, nxt = 0;
    bool st = false;
    int64_t n = 0;
    bool timed_out = false;
    for (; n < loaded; ++n) {
        const int s = (int)(n % DB_STAGES);
        const int64_t u = stage_unit[s];
        const int64_t t = u / nchunks;
        const int c = (int)(u - t * nchunks);
        if (t != cur_t) {
            cur = t == nxt_t ? nxt : kl ? ld_nc_s32(slot_of + t * k + lane) : 0;
            cur_t = t;
            st = first_of_row(cur);
        }
        if (n + 1 < loaded) {
            const int64_t tn = stage_unit[(n + 1) % DB_STAGES] / nchunks;
            if (tn != cur_t && tn != nxt_t) {
                nxt = kl ? ld_nc_s32(slot_of + tn * k + lane) : 0;
                nxt_t = tn;
            }
        }
        if (!mbar_wait(full(s), (uint32_t)(n / DB_STAGES) & 1)) {
            timed_out = true;
            break;
        }
        const uint32_t cb = (uint32_t)min((int64_t)CH, rowbytes - (int64_t)c * CH);
        fence_proxy_async_smem();
        if (st) {
            if ((unsigned)cur < (unsigned)rows)
                bulk_s2g(recv + (int64_t)cur * rowbytes + (int64_t)c * CH, stages + (uint32_t)s * CH, cb);
            else if (c == 0)
                report(err_word, MOE_ERRBIT_BAD_INDEX);
        }
        bulk_commit();
        // refill the stage unit n-1 used with the next unit to load
        if (n >= 1 && more) {
            bulk_wait_read<1>();
            __syncwarp();
            issue_load();
        }
    }
    if (timed_out) {
        if (lane == 0)
            report(err_word, MOE_ERRBIT_TIMEOUT);
        for (int64_t m = n + lane; m < loaded; m += 32)  // let issued loads land
            (void)mbar_wait(full((int)(m % DB_STAGES)), (uint32_t)(m / DB_STAGES) & 1);
    }
    bulk_wait_all();
    if (pooled && lane == 0)
        sched_finish(sched);
}

constexpr int DISPATCH_THREADS = 256;
constexpr int DISPATCH_U = 4;  // 16-byte vectors per lane per item

template <int U>
__global__ void __launch_bounds__(DISPATCH_THREADS)
    dispatch_bf16_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ slot_of,
                         uint4 *__restrict__ recv, int k, int C, int groups, int64_t items,
                         int N, uint32_t *err_word)
{
    wait_prior_grid();
    allow_next_grid();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (DISPATCH_THREADS / 32);
    for (int64_t it = (int64_t)blockIdx.x * (DISPATCH_THREADS / 32) + (threadIdx.x >> 5);
         it < items; it += nwarps) {
        const int64_t t = it / groups;
        const int c0 = (int)(it - t * groups) * (32 * U) + lane;
        const uint4 *src = x + t * C;
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (c0 + u * 32 < C)
                v[u] = ld_stream_v4(src + c0 + u * 32);
        const int32_t *so = slot_of + t * k;
        for (int jb = 0; jb < k; jb += 32) {
            const int32_t mine = jb + lane < k ? ld_nc_s32(so + jb + lane) : 0;
            const int jn = min(32, k - jb);
            for (int q = 0; q < jn; ++q) {
                const int32_t s = __shfl_sync(FULL_MASK, mine, q);
                if ((unsigned)s >= (unsigned)N) {
                    if (lane == 0)
                        report(err_word, MOE_ERRBIT_BAD_INDEX);
                    continue;
                }
                uint4 *dst = recv + (int64_t)s * C;
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (c0 + u * 32 < C)
                        st_v4(dst + c0 + u * 32, v[u]);
            }
        }
    }
}

template <bool COAL>
static cudaError_t launch_dispatch_bulk(int T, int H, int k, const void *x,
                                       const int32_t *slot_of, void *recv, int rows,
                                       bool prefetch_x, uint32_t *err_word, cudaStream_t stream)
{
    const int64_t rowbytes = 2 * (int64_t)H;
    const int CH = rowbytes < DB_CHUNK ? (int)rowbytes : DB_CHUNK;
    const int nchunks = (int)((rowbytes + CH - 1) / CH);
    const int64_t units = (int64_t)T * nchunks;
    const size_t smem = 128 + (size_t)DB_STAGES * CH;
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024)
        e = cudaFuncSetAttribute(dispatch_bulk_kernel<COAL>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    int per_sm = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_bulk_kernel<COAL>, 32,
                                                      smem) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    const int64_t g = units < cap ? units : cap;
    const int64_t even = units / g;
    const bool pooled = even >= DB_DYN_MIN;
    const int64_t per_cta = pooled ? units * DB_STATIC_PCT / 100 / g : 0;
    return launch_pdl(dispatch_bulk_kernel<COAL>, dim3((unsigned)g), dim3(32), smem, stream,
                      static_cast<const uint8_t *>(x), slot_of, static_cast<uint8_t *>(recv), T, k,
                      rowbytes, CH, nchunks, units, per_cta, DB_GRAB,
                      pooled ? next_sched_slot(g_dispatch_seq) : -1, rows, prefetch_x ? 1 : 0,
                      err_word);
}

cudaError_t launch_dispatch_coalesced(int T, int H, int k, const void *x, const int32_t *crow,
                                      void *recv_c, int rows, uint32_t *err_word,
                                      cudaStream_t stream)
{
    if (T == 0)
        return cudaSuccess;
    return launch_dispatch_bulk<true>(T, H, k, x, crow, recv_c, rows, false, err_word, stream);
}

cudaError_t launch_dispatch_bf16(int T, int H, int k, const void *x, const int32_t *slot_of,
                                 void *recv, uint32_t *err_word, cudaStream_t stream)
{
    if (T == 0)
        return cudaSuccess;
    if (k <= 32)
        return launch_dispatch_bulk<false>(T, H, k, x, slot_of, recv, T * k, false, err_word,
                                           stream);
    const int C = H / 8;
    const int groups = (C + 32 * DISPATCH_U - 1) / (32 * DISPATCH_U);
    const int64_t items = (int64_t)T * groups;
    const int grid = warp_item_grid((const void *)dispatch_bf16_kernel<DISPATCH_U>,
                                    DISPATCH_THREADS, 0, items);
    return launch_pdl(dispatch_bf16_kernel<DISPATCH_U>, dim3(grid), dim3(DISPATCH_THREADS), 0,
                      stream, static_cast<const uint4 *>(x), slot_of, static_cast<uint4 *>(recv),
                      k, C, groups, items, T * k, err_word);
}

cudaError_t launch_layout_dispatch(int T, int H, int k, int E, int R, const int32_t *topk_idx,
                                   const void *x, int32_t *expert_counts,
                                   int32_t *expert_offsets, int32_t *rank_offsets,
                                   int32_t *slot_of, int32_t *src_of, void *recv,
                                   void *workspace, uint32_t *err_word, cudaStream_t stream)
{
    // small batches: one kernel in which every CTA computes the layout itself
    if (layout_dispatch_fused_fits(T, H, k, E))
        return launch_layout_dispatch_fused(T, H, k, E, R, topk_idx, x, expert_counts,
                                            expert_offsets, rank_offsets, slot_of, src_of, recv,
                                            err_word, stream);
    cudaError_t e = launch_layout(T, k, E, R, topk_idx, expert_counts, expert_offsets,
                                  rank_offsets, slot_of, src_of, workspace, err_word, stream);
    if (e != cudaSuccess || T == 0)
        return e;
    if (k <= 32)  // the layout kernel is the previous grid: x may be read early
        return launch_dispatch_bulk<false>(T, H, k, x, slot_of, recv, T * k, true, err_word,
                                           stream);
    return launch_dispatch_bf16(T, H, k, x, slot_of, recv, err_word, stream);
}

}  // namespace moe

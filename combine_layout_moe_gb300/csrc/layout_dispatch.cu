// moe_layout_dispatch for small batches: the whole layout (count, scan, slot
// map) and the bf16 dispatch in one kernel, with no exchange between CTAs
// (sm_103a).
//
// UBEP, section 3.2: token sending overlaps the count and its prefix sum
// (CalCumSum) instead of waiting behind them; UBEP section 2.3 / Figure 2 and
// StrataCL Appendix D: per-expert counts -> prefix-sum offsets -> token-local
// offsets.
//
// GPU design.  The (token, row chunk) units are split evenly over at most one
// CTA per SM.  Each CTA
//   1. issues one bulk copy per unit of its share of x into shared memory, all
//      at once (x is complete when the call is made); the whole share stays
//      resident, so no stage is ever recycled;
//   2. while those land, counts every (t, j) pair of the batch itself (the ids
//      are read once per CTA, from L2 after the first, with 16-byte loads)
//      into two shared-memory histograms: pairs before its first token, and
//      the rest;
//   3. scans the totals over experts and gives each pair of its own tokens the
//      slot offset[e] + (pairs of e before its first token) + (pairs of e
//      among its own before it) -- the stable order (expert, t, j), the same
//      in every CTA because every CTA counts the same ids;
//   4. stores each landed unit to its k slots with bulk shared -> global
//      copies, issued by as many threads as there are (unit, slot) pairs.
// No grid barrier, tile table or global atomic: each CTA re-counts the batch,
// a 4*T*k-byte read per CTA.  That pays while the batch is small; the host
// uses this form only up to FUSED_MAX_PAIRS pairs and when each CTA's share
// of x fits in shared memory, and otherwise launches the layout kernel and
// then the dispatch kernel.
#include "common.cuh"
#include "launch.h"
#include "tma.cuh"

namespace moe {

constexpr int FUSED_THREADS = 512;
constexpr int FUSED_MAX_UNITS = 32;                // units per CTA (one mbarrier each)
constexpr int FUSED_MAX_OWN = 512;                 // pairs of the tokens a CTA touches
constexpr int64_t FUSED_MAX_PAIRS = 16384;         // T*k of the batches this form takes
constexpr int FUSED_CHUNK = 16384;                 // bytes per unit (a row, or part of one)
constexpr size_t FUSED_PAYLOAD_MAX = 200 * 1024;   // x bytes resident per CTA

__device__ __forceinline__ int4 ld_nc_v4_s32(const int4 *p)
{
    int4 v;
    asm volatile("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Shared-memory header: mbarriers, histograms, the CTA's own pairs, flags.
__host__ __device__ constexpr size_t fused_payload_offset(int E)
{
    return (256 + sizeof(int32_t) * (2 * (size_t)E + 2 * FUSED_MAX_OWN + 4) + 127) / 128 * 128;
}

// Phase timestamps for tuning builds (-DMOE_TRACE): CTA 0 stores %globaltimer
// at phase boundaries into the 64-bit words that follow the error word; word
// 14 gets the latest CTA start and word 15 the latest CTA end.
#ifdef MOE_TRACE
#define FUSED_TRACE(n)                                                                 \
    do {                                                                               \
        if (blockIdx.x == 0 && threadIdx.x == 0 && err_word)                            \
            reinterpret_cast<unsigned long long *>(err_word)[8 + (n)] = global_ns();   \
    } while (0)
#define FUSED_TRACE_MAX(n)                                                                      \
    do {                                                                                        \
        if (threadIdx.x == 0 && err_word)                                                       \
            atomicMax(reinterpret_cast<unsigned long long *>(err_word) + 8 + (n), global_ns()); \
    } while (0)
#else
#define FUSED_TRACE(n) \
    do {               \
    } while (0)
#define FUSED_TRACE_MAX(n) \
    do {                   \
    } while (0)
#endif

__global__ void __launch_bounds__(FUSED_THREADS, 1)
    layout_dispatch_fused_kernel(const int32_t *__restrict__ idx, const uint8_t *__restrict__ x,
                                 int T, int k, int E, int R, int64_t rowbytes, int CH, int nch,
                                 int64_t units, int32_t *__restrict__ expert_counts,
                                 int32_t *__restrict__ expert_offsets,
                                 int32_t *__restrict__ rank_offsets,
                                 int32_t *__restrict__ slot_of, int32_t *__restrict__ src_of,
                                 uint8_t *__restrict__ recv, uint32_t *err_word)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t bars = smem_addr(smem);                   // [FUSED_MAX_UNITS] mbarriers
    int32_t *pre = reinterpret_cast<int32_t *>(smem + 256);  // [E] pairs of e before P0, then cursors
    int32_t *post = pre + E;                                 // [E] the rest, then offsets
    int32_t *own = post + E;                                 // [FUSED_MAX_OWN] ids of pairs P0..P1
    int32_t *sl = own + FUSED_MAX_OWN;                       // [FUSED_MAX_OWN] their slots
    int32_t *flags = sl + FUSED_MAX_OWN;                     // bad id, total, timeout
    const uint32_t payload = bars + (uint32_t)fused_payload_offset(E);

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int64_t N = (int64_t)T * k;
    const int64_t u_lo = units * blockIdx.x / gridDim.x;
    const int64_t u_hi = units * (blockIdx.x + 1) / gridDim.x;
    const int Uc = (int)(u_hi - u_lo);             // >= 1: the grid is at most `units`
    const int64_t t_lo = u_lo / nch, t_hi = (u_hi - 1) / nch;
    const int64_t P0 = t_lo * k, P1 = (t_hi + 1) * k;
    const int p = (int)(P1 - P0);                  // <= FUSED_MAX_OWN (checked on the host)
    FUSED_TRACE(0);
    FUSED_TRACE_MAX(6);

    wait_prior_grid();
    allow_next_grid();
    // the first batch of ids is requested before anything else: their
    // latency is the head of the critical path
    const bool vec = (reinterpret_cast<uintptr_t>(idx) & 15) == 0;
    const int64_t nv = vec ? N / 4 : 0;
    const int4 *iv = reinterpret_cast<const int4 *>(idx);
    int4 v0[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int64_t q = tid + (int64_t)u * nthr;
        v0[u] = q < nv ? ld_nc_v4_s32(iv + q) : make_int4(0, 0, 0, 0);
    }
    for (int i = tid; i < 2 * E; i += nthr)
        pre[i] = 0;
    if (tid < 4)
        flags[tid] = 0;
    if (tid == 0) {
        for (int q = 0; q < Uc; ++q)
            mbar_init(bars + 8u * q, 1);
        mbar_fence_init();
    }
    __syncthreads();

    // 1. the CTA's share of x, one bulk copy per unit
    auto load_x = [&]() {
        if (tid < Uc) {
            const int64_t u = u_lo + tid, t = u / nch;
            const int c = (int)(u - t * nch);
            const uint32_t cb = (uint32_t)min((int64_t)CH, rowbytes - (int64_t)c * CH);
            mbar_arrive_expect_tx(bars + 8u * tid, cb);
            bulk_g2s(payload + (uint32_t)tid * CH, x + t * rowbytes + (int64_t)c * CH, cb,
                     bars + 8u * tid);
        }
    };
#ifdef MOE_FUSED_X_FIRST
    load_x();
#endif

    // 2. the whole batch's histogram, split at this CTA's first pair P0
    bool bad = false;
    auto count = [&](int64_t i, int e) {
        const bool mine = i >= P0 && i < P1;
        if ((unsigned)e >= (unsigned)E) {
            bad = true;
            if (mine)
                own[i - P0] = -1;
            return;
        }
        atomicAdd(i < P0 ? pre + e : post + e, 1);
        if (mine)
            own[i - P0] = e;
    };
    if (vec) {
        for (int64_t q0 = tid; q0 < nv; q0 += (int64_t)nthr * 4) {
            int4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t q = q0 + (int64_t)u * nthr;
                v[u] = q0 == tid ? v0[u] : q < nv ? ld_nc_v4_s32(iv + q) : make_int4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t q = q0 + (int64_t)u * nthr;
                if (q < nv) {
                    count(4 * q, v[u].x);
                    count(4 * q + 1, v[u].y);
                    count(4 * q + 2, v[u].z);
                    count(4 * q + 3, v[u].w);
                }
            }
        }
        for (int64_t i = nv * 4 + tid; i < N; i += nthr)
            count(i, ld_nc_s32(idx + i));
    } else {
        for (int64_t i0 = tid; i0 < N; i0 += (int64_t)nthr * 4) {
            int e[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t i = i0 + (int64_t)u * nthr;
                e[u] = i < N ? ld_nc_s32(idx + i) : 0;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t i = i0 + (int64_t)u * nthr;
                if (i < N)
                    count(i, e[u]);
            }
        }
    }
    if (bad)
        flags[0] = 1;
#ifndef MOE_FUSED_X_FIRST
    // issued once the ids are in: the ids then meet an idle memory system,
    // and x (at most ~200 KB per SM) still lands before the slots are known
    load_x();
#endif
    __syncthreads();
    FUSED_TRACE(1);

    // 3. warp 0: exclusive scan of the totals over experts.  Each lane sums
    //    a run of ceil(E/32) experts, one warp scan, each lane writes its
    //    run's offsets (post) and cursors (pre: offset + pairs before P0).
    //    Meanwhile the other warps rank each pair of this CTA's tokens among
    //    the earlier such pairs of its expert (sl: the rank, or -1).
    if (tid < 32) {
        const int lane = tid;
        const int per = (E + 31) / 32;
        const int e0 = lane * per;
        int32_t sum = 0;
        for (int q = 0; q < per && e0 + q < E; ++q)
            sum += pre[e0 + q] + post[e0 + q];
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
            const int32_t tot = pre[e] + post[e];
            if (blockIdx.x == 0) {
                expert_counts[e] = tot;
                expert_offsets[e] = run;
            }
            post[e] = run;
            pre[e] += run;
            run += tot;
        }
        if (lane == 31)
            flags[1] = incl;
    } else {
        for (int q = tid - 32; q < p; q += nthr - 32) {
            const int e = own[q];
            int32_t c = -1;
            if (e >= 0) {
                c = 0;
#pragma unroll 8
                for (int q2 = 0; q2 < q; ++q2)  // independent loads, eight in flight
                    c += own[q2] == e;
            }
            sl[q] = c;
        }
    }
    __syncthreads();
    FUSED_TRACE(2);
    if (blockIdx.x == 0) {
        const int32_t total = flags[1];
        if (tid == 0)
            expert_offsets[E] = total;
        const int El = E / R;
        for (int r = tid; r <= R; r += nthr)
            rank_offsets[r] = r == R ? total : post[r * El];
    }
    FUSED_TRACE(3);

    // 4. every landed unit to its k slots: slot = cursor of the expert + the
    //    pair's rank among this CTA's pairs of that expert.  The task of a
    //    token's first chunk also writes the pair's slot_of and src_of entries
    //    (each token's first chunk lies in exactly one CTA).
    bool timed_out = false;
    for (int task = tid; task < Uc * k; task += nthr) {
        const int q = task / k, j = task - q * k;
        const int64_t u = u_lo + q, t = u / nch;
        const int c = (int)(u - t * nch);
        const int qo = (int)(t - t_lo) * k + j;
        const int e = own[qo];
        const int32_t s = e >= 0 ? pre[e] + sl[qo] : -1;
        if (c == 0) {
            const int64_t i = t * k + j;
            slot_of[i] = s;
            if (s >= 0)
                src_of[s] = (int32_t)i;
        }
        if ((unsigned)s >= (unsigned)N)
            continue;  // an id out of range: reported below
        if (!mbar_wait(bars + 8u * q, 0)) {
            timed_out = true;
            break;
        }
        const uint32_t cb = (uint32_t)min((int64_t)CH, rowbytes - (int64_t)c * CH);
        fence_proxy_async_smem();
        bulk_s2g(recv + (int64_t)s * rowbytes + (int64_t)c * CH, payload + (uint32_t)q * CH, cb);
        bulk_commit();
    }
    if (timed_out)
        flags[2] = 1;
    FUSED_TRACE(4);
    bulk_wait_all();
    __syncthreads();
    FUSED_TRACE(5);
    FUSED_TRACE_MAX(7);
    if (flags[2]) {
        // a load that did not land in time: report it, and let every issued
        // load land (again bounded) before the CTA's shared memory goes away
        if (tid == 0)
            report(err_word, MOE_ERRBIT_TIMEOUT);
        if (tid < Uc)
            (void)mbar_wait(bars + 8u * tid, 0);
    }
    if (tid == 0 && blockIdx.x == 0 && flags[0])
        report(err_word, MOE_ERRBIT_BAD_INDEX);
}

// How a batch is cut into units: rows split into nch chunks of CH bytes (a
// multiple of 16), the units spread over G CTAs, at most umax per CTA.  Rows
// are split further while that keeps at most FUSED_TARGET_UNITS units per CTA
// and chunks of at least FUSED_MIN_CHUNK bytes: finer units even out the
// CTAs' shares (1024 rows of 14 KB over 152 SMs is 6 or 7 rows each, 16 %
// apart; halves of rows are 13 or 14, 7 % apart).
struct FusedPlan {
    bool ok;
    int CH, nch, G, umax;
    int64_t units;
};

constexpr int FUSED_TARGET_UNITS = 24;
constexpr int FUSED_MIN_CHUNK = 2048;

static FusedPlan fused_plan(int T, int H, int k, int E)
{
    FusedPlan p{false, 0, 0, 0, 0, 0};
    const int64_t N = (int64_t)T * k;
    if (T < 1 || N > FUSED_MAX_PAIRS || k > 32 || E > MOE_MAX_EXPERTS)
        return p;
    const int64_t rowbytes = 2 * (int64_t)H;
    const int sms = sm_count();
    auto cut = [&](int64_t want, FusedPlan &q) {
        const int64_t ch = ((rowbytes + want - 1) / want + 15) / 16 * 16;
        q.CH = (int)(ch < FUSED_CHUNK ? ch : FUSED_CHUNK);
        q.nch = (int)((rowbytes + q.CH - 1) / q.CH);
        q.units = (int64_t)T * q.nch;
        q.G = (int)(q.units < sms ? q.units : sms);
        q.umax = (int)((q.units + q.G - 1) / q.G);
    };
    cut((rowbytes + FUSED_CHUNK - 1) / FUSED_CHUNK, p);
    for (;;) {
        FusedPlan q = p;
        cut(2 * (int64_t)p.nch, q);
        if (q.nch <= p.nch || q.CH < FUSED_MIN_CHUNK || q.umax > FUSED_TARGET_UNITS)
            break;
        p = q;
    }
    if (p.umax > FUSED_MAX_UNITS || (size_t)p.umax * p.CH > FUSED_PAYLOAD_MAX)
        return p;
    // a CTA's units span at most ceil(umax / nch) + 1 tokens
    p.ok = ((p.umax + p.nch - 1) / p.nch + 1) * (int64_t)k <= FUSED_MAX_OWN;
    return p;
}

bool layout_dispatch_fused_fits(int T, int H, int k, int E) { return fused_plan(T, H, k, E).ok; }

cudaError_t launch_layout_dispatch_fused(int T, int H, int k, int E, int R,
                                         const int32_t *topk_idx, const void *x,
                                         int32_t *expert_counts, int32_t *expert_offsets,
                                         int32_t *rank_offsets, int32_t *slot_of,
                                         int32_t *src_of, void *recv, uint32_t *err_word,
                                         cudaStream_t stream)
{
    const FusedPlan p = fused_plan(T, H, k, E);
    if (!p.ok)
        return cudaErrorInvalidValue;
    const size_t smem = fused_payload_offset(E) + (size_t)p.umax * p.CH;
    cudaError_t e = cudaFuncSetAttribute(layout_dispatch_fused_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    e = launch_pdl(layout_dispatch_fused_kernel, dim3((unsigned)p.G), dim3(FUSED_THREADS), smem,
                   stream, topk_idx, static_cast<const uint8_t *>(x), T, k, E, R,
                   2 * (int64_t)H, p.CH, p.nch, p.units, expert_counts, expert_offsets,
                   rank_offsets, slot_of, src_of, static_cast<uint8_t *>(recv), err_word);
    if (e == cudaSuccess)
        note_layout_form(MOE_LAYOUT_FORM_FUSED);
    return e;
}

}  // namespace moe

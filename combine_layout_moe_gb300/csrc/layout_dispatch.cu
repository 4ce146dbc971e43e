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
    const int64_t t_own = (u_lo + nch - 1) / nch;  // first token whose chunk 0 is here

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
    wait_prior_grid();
    allow_next_grid();

    // 1. the CTA's share of x, one bulk copy per unit
    if (tid < Uc) {
        const int64_t u = u_lo + tid, t = u / nch;
        const int c = (int)(u - t * nch);
        const uint32_t cb = (uint32_t)min((int64_t)CH, rowbytes - (int64_t)c * CH);
        mbar_arrive_expect_tx(bars + 8u * tid, cb);
        bulk_g2s(payload + (uint32_t)tid * CH, x + t * rowbytes + (int64_t)c * CH, cb,
                 bars + 8u * tid);
    }

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
    if ((reinterpret_cast<uintptr_t>(idx) & 15) == 0) {
        const int64_t nv = N / 4;
        const int4 *iv = reinterpret_cast<const int4 *>(idx);
        for (int64_t q0 = tid; q0 < nv; q0 += (int64_t)nthr * 4) {
            int4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t q = q0 + (int64_t)u * nthr;
                v[u] = q < nv ? ld_nc_v4_s32(iv + q) : make_int4(0, 0, 0, 0);
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
    __syncthreads();

    // 3a. exclusive scan of the totals over experts by warp 0: each lane sums
    //     a run of ceil(E/32) experts, one warp scan, each lane writes its
    //     run's offsets (post) and cursors (pre: offset + pairs before P0)
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
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        const int32_t total = flags[1];
        if (tid == 0)
            expert_offsets[E] = total;
        const int El = E / R;
        for (int r = tid; r <= R; r += nthr)
            rank_offsets[r] = r == R ? total : post[r * El];
    }

    // 3b. slots of the pairs of this CTA's tokens; the CTA holding a token's
    //     first chunk writes its slot_of and src_of entries
    for (int q = tid; q < p; q += nthr) {
        const int e = own[q];
        int32_t s = -1;
        if (e >= 0) {
            int c = 0;
            for (int q2 = 0; q2 < q; ++q2)
                c += own[q2] == e;
            s = pre[e] + c;
        }
        sl[q] = s;
        const int64_t i = P0 + q;
        if (i / k >= t_own) {
            slot_of[i] = s;
            if (s >= 0)
                src_of[s] = (int32_t)i;
        }
    }
    __syncthreads();

    // 4. every landed unit to its k slots
    bool timed_out = false;
    for (int task = tid; task < Uc * k; task += nthr) {
        const int q = task / k, j = task - q * k;
        const int64_t u = u_lo + q, t = u / nch;
        const int c = (int)(u - t * nch);
        const int32_t s = sl[(t - t_lo) * k + j];
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
    bulk_wait_all();
    __syncthreads();
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

bool layout_dispatch_fused_fits(int T, int H, int k, int E)
{
    const int64_t N = (int64_t)T * k;
    if (T < 1 || N > FUSED_MAX_PAIRS || k > 32 || E > MOE_MAX_EXPERTS)
        return false;
    const int64_t rowbytes = 2 * (int64_t)H;
    const int CH = rowbytes < FUSED_CHUNK ? (int)rowbytes : FUSED_CHUNK;
    const int64_t nch = (rowbytes + CH - 1) / CH;
    const int64_t units = (int64_t)T * nch;
    const int64_t G = units < sm_count() ? units : sm_count();
    const int64_t umax = (units + G - 1) / G;
    if (umax > FUSED_MAX_UNITS || (size_t)umax * CH > FUSED_PAYLOAD_MAX)
        return false;
    // a CTA's units span at most ceil(umax / nch) + 1 tokens
    return ((umax + nch - 1) / nch + 1) * k <= FUSED_MAX_OWN;
}

cudaError_t launch_layout_dispatch_fused(int T, int H, int k, int E, int R,
                                         const int32_t *topk_idx, const void *x,
                                         int32_t *expert_counts, int32_t *expert_offsets,
                                         int32_t *rank_offsets, int32_t *slot_of,
                                         int32_t *src_of, void *recv, uint32_t *err_word,
                                         cudaStream_t stream)
{
    const int64_t rowbytes = 2 * (int64_t)H;
    const int CH = rowbytes < FUSED_CHUNK ? (int)rowbytes : FUSED_CHUNK;
    const int nch = (int)((rowbytes + CH - 1) / CH);
    const int64_t units = (int64_t)T * nch;
    const int64_t G = units < sm_count() ? units : sm_count();
    const int64_t umax = (units + G - 1) / G;
    const size_t smem = fused_payload_offset(E) + (size_t)umax * CH;
    cudaError_t e = cudaFuncSetAttribute(layout_dispatch_fused_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    e = launch_pdl(layout_dispatch_fused_kernel, dim3((unsigned)G), dim3(FUSED_THREADS), smem,
                   stream, topk_idx, static_cast<const uint8_t *>(x), T, k, E, R, rowbytes, CH,
                   nch, units, expert_counts, expert_offsets, rank_offsets, slot_of, src_of,
                   static_cast<uint8_t *>(recv), err_word);
    if (e == cudaSuccess)
        note_layout_form(MOE_LAYOUT_FORM_FUSED);
    return e;
}

}  // namespace moe

// Dispatch -> identity expert -> combine in one persistent kernel, each hop
// synchronised by the reader observing the data's readiness (sm_103a).
//
// UBEP, section 3.4 (Data-as-Flag: readiness travels with the data instead of
// a global barrier; Figure 6 compares Token-Flag Fusion, Data-for-Checksum
// and Sentinel Polling), section 3.2 (kernel decomposition: a consumer starts
// on a piece of work as soon as its inputs are signalled) and section 6
// (without atomic 512-byte writes, fall back to explicit fences).
//
// Structure: one cooperative launch, every warp resident.  Each warp runs
// three phases over its own contiguous range of units; a unit is W bytes of
// one row -- W = max(G, 2048), or one batch (BATCH) -- where G is the
// synchronisation granularity.  A lane issues the loads of four 512-byte warp
// steps before it stores any of them, and combine loads up to eight slots'
// rows before folding them:
//   produce  (token t, unit): x[t] -> the k rows slot_of[t, :] of recv
//   expert   (receive row s, unit), in receive (expert-major) order:
//            recv[s] -> y[s] (the identity expert)
//   combine  (token t, unit): out[t] = sum_j w[t, j] * y[slot_of[t, j]]
//            (fp32 fused multiply-adds in slot order from +0, one rounding)
// The expert phase reads rows other warps produced and the combine phase rows
// other warps copied, so every hop crosses SMs.  Producing never waits and the
// expert phase waits only on producers, so with every warp resident every wait
// ends; each is still bounded, and a warp whose wait ran out gives up at once
// on any later wait whose data is not already there.
//
// How a reader learns that a block of G bytes has arrived (MOE_SYNC_*):
//   WORD      one 32-bit word per (row, block): the writer stores the block,
//             fences, then stores the call's epoch; the reader acquires the
//             word.  A GPU has no 512-byte atomic store, so the flag cannot
//             share a store with the data as in Token-Flag Fusion: this is the
//             explicit-fence form.
//   SENTINEL  no words: recv and y start out holding the sentinel in every
//             32-bit word; the reader polls the data itself until none of its
//             words is the sentinel (32-bit accesses are single-copy atomic;
//             wider ones are not, so every word is checked, not a 32-byte
//             marker), uses it, and writes the sentinel back for the next
//             call (Sentinel Polling's buffer reset).  The sentinel is the
//             pair of bf16 NaNs 0xFFFF 0xFFFF; a payload word equal to it is
//             reported (MOE_ERRBIT_SENTINEL) and its reader's wait runs out.
//   BATCH     one 64-bit word per (row, batch of G bytes, G a multiple of
//             512): the writer stores the batch, fences, then stores (epoch,
//             sum of the first 32-bit word of each 512-byte block); the reader
//             acquires the word and checks the sum against the words it read
//             (Data-for-Checksum; a mismatch sets MOE_ERRBIT_CHECKSUM).
//   BARRIER   no readiness at all: a grid barrier between the phases (the
//             stop-and-wait baseline).
#include <cuda_bf16.h>

#include "common.cuh"
#include "grid_sync.cuh"
#include "launch.h"
#include "tma.cuh"

namespace moe {

constexpr int DF_THREADS = 256;
constexpr int DF_WARPS = DF_THREADS / 32;
constexpr int DF_STEP = 512;  // bytes a warp moves per step: 32 lanes x 16 B
// Tunables (compile-time; the defaults are the shipped configuration).
#ifndef MOE_DF_ILP
#define MOE_DF_ILP 4
#endif
#ifndef MOE_DF_MINB
#define MOE_DF_MINB 4
#endif
constexpr int DF_ILP = MOE_DF_ILP;  // steps whose loads a lane issues before storing
constexpr int DF_JG = 8;      // slots whose rows combine loads before folding
constexpr int DF_UNIT = DF_STEP * DF_ILP;  // smallest unit (WORD, SENTINEL, BARRIER)
constexpr uint32_t DF_SENTINEL = 0xFFFFFFFFu;

__device__ __forceinline__ void st_relaxed_u32(uint32_t *p, uint32_t v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
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

// Accesses to data that is itself polled (SENTINEL): volatile, so every load
// goes to memory and each 32-bit element is read and written whole.
__device__ __forceinline__ uint4 ld_volatile_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.volatile.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_volatile_v4(void *p, uint4 v)
{
    asm volatile("st.volatile.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ bool has_sentinel(uint4 d)
{
    return d.x == DF_SENTINEL || d.y == DF_SENTINEL || d.z == DF_SENTINEL || d.w == DF_SENTINEL;
}

__device__ __forceinline__ uint4 sentinel4()
{
    return make_uint4(DF_SENTINEL, DF_SENTINEL, DF_SENTINEL, DF_SENTINEL);
}

// Spins (this lane alone) until ready() holds.  False once limit_ns has
// passed, or at once when give_up is set and the data is not there yet.
template <class F>
__device__ __forceinline__ bool spin_until(F ready, uint64_t limit_ns, bool give_up)
{
    if (ready())
        return true;
    if (give_up)
        return false;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (ready())
            return true;
        if (global_ns() - t0 > limit_ns)
            return false;
    }
}

struct DfArgs {
    const uint4 *x;
    const int32_t *slot_of;
    const float *topk_w;
    uint4 *recv;
    uint4 *y;
    void *out;
    int out_f32;
    int T, k, C;  // tokens, slots per token, 16-byte vectors per row
    int G;        // synchronisation granularity in bytes
    int W;        // unit bytes: G (BATCH) or max(G, DF_UNIT)
    int upr;      // units per row
    int nblk;     // G-byte blocks per row
    uint32_t *words;
    uint32_t epoch;
    uint64_t spin_ns;
    int64_t skip_pair;
    uint32_t *err;
};

template <int MODE>
__global__ void __launch_bounds__(DF_THREADS, MOE_DF_MINB) dispatch_combine_flagged_kernel(const DfArgs a)
{
    wait_prior_grid();
    allow_next_grid();
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * DF_WARPS;
    const int64_t gw = (int64_t)blockIdx.x * DF_WARPS + (threadIdx.x >> 5);
    const int k = a.k, C = a.C, N = a.T * a.k;
    const int nsteps = a.W / DF_STEP;
    const int vpu = a.W / 16;  // vectors per unit
    const int64_t tok_units = (int64_t)a.T * a.upr, row_units = (int64_t)N * a.upr;
    uint32_t *const dwords = a.words;                       // WORD: dispatch hop
    uint32_t *const ewords = a.words + (size_t)N * a.nblk;  // WORD: expert hop
    unsigned long long *const dbatch = reinterpret_cast<unsigned long long *>(a.words);
    unsigned long long *const ebatch = dbatch + (size_t)N * a.nblk;
    bool give_up = false;  // warp-uniform: a wait of this warp already ran out
    auto timed_out = [&]() {
        if (lane == 0)
            report(a.err, MOE_ERRBIT_TIMEOUT);
        give_up = true;
    };
    // vector of this lane in step q of unit cu
    auto vec = [&](int cu, int q) { return cu * vpu + q * 32 + lane; };
    // WORD: wait (this lane alone) for the word of every block its vectors of
    // unit cu of row s fall in; false if a wait ran out
    auto wait_blocks = [&](const uint32_t *words, int64_t s, int cu, uint64_t limit) {
        bool ok = true;
        int last = -1;
        for (int q = 0; q < nsteps; ++q) {
            const int v = vec(cu, q);
            if (v >= C)
                break;
            const int b = v * 16 / a.G;
            if (b == last)
                continue;
            last = b;
            const uint32_t *w = words + (size_t)s * a.nblk + b;
            ok = ok && spin_until([&] { return ld_acquire_u32(w) == a.epoch; }, limit,
                                  give_up || !ok);
        }
        return ok;
    };
    // WORD: publish the words of the blocks of unit cu of row s (after a fence)
    auto publish_blocks = [&](uint32_t *words, int64_t s, int cu) {
        const int b0 = cu * a.W / a.G, nb = a.W / a.G;
        for (int b = lane; b < nb && b0 + b < a.nblk; b += 32)
            st_relaxed_u32(words + (size_t)s * a.nblk + b0 + b, a.epoch);
    };

    // ------------------------------------------------------------ produce
    {
        const int64_t u0 = tok_units * gw / nw, u1 = tok_units * (gw + 1) / nw;
        for (int64_t u = u0; u < u1; ++u) {
            const int64_t t = u / a.upr;
            const int cu = (int)(u - t * a.upr);
            const int32_t mine = lane < k ? ld_nc_s32(a.slot_of + t * k + lane) : -1;
            uint32_t csum = 0;  // lane 0: the first word of each 512-byte block
            bool hit = false;
            for (int q0 = 0; q0 < nsteps; q0 += DF_ILP) {
                uint4 d[DF_ILP];
                bool in[DF_ILP];
#pragma unroll
                for (int r = 0; r < DF_ILP; ++r) {
                    const int v = vec(cu, q0 + r);
                    in[r] = q0 + r < nsteps && v < C;
                    d[r] = in[r] ? ld_stream_v4(a.x + t * C + v) : make_uint4(0, 0, 0, 0);
                    csum += d[r].x;
                    hit |= in[r] && has_sentinel(d[r]);
                }
                for (int j = 0; j < k; ++j) {
                    const int32_t s = __shfl_sync(FULL_MASK, mine, j);
                    if ((unsigned)s >= (unsigned)N) {
                        if (lane == 0 && cu == 0 && q0 == 0)
                            report(a.err, MOE_ERRBIT_BAD_INDEX);
                        continue;
                    }
                    if (MODE == MOE_SYNC_SENTINEL && t * k + j == a.skip_pair)
                        continue;
#pragma unroll
                    for (int r = 0; r < DF_ILP; ++r) {
                        if (!in[r])
                            continue;
                        uint4 *dst = a.recv + (int64_t)s * C + vec(cu, q0 + r);
                        if (MODE == MOE_SYNC_SENTINEL)
                            st_volatile_v4(dst, d[r]);
                        else
                            st_v4(dst, d[r]);
                    }
                }
            }
            if (MODE == MOE_SYNC_SENTINEL && __any_sync(FULL_MASK, hit) && lane == 0)
                report(a.err, MOE_ERRBIT_SENTINEL);
            if (MODE != MOE_SYNC_WORD && MODE != MOE_SYNC_BATCH)
                continue;
            __threadfence();  // this lane's row stores, before any word below
            __syncwarp();
            for (int j = 0; j < k; ++j) {
                const int32_t s = __shfl_sync(FULL_MASK, mine, j);
                if ((unsigned)s >= (unsigned)N || t * k + j == a.skip_pair)
                    continue;
                if (MODE == MOE_SYNC_WORD) {
                    publish_blocks(dwords, s, cu);
                } else {
                    const uint32_t sum = __shfl_sync(FULL_MASK, csum, 0);
                    if (lane == 0)
                        st_relaxed_u64(dbatch + (size_t)s * a.nblk + cu,
                                       ((unsigned long long)a.epoch << 32) | sum);
                }
            }
        }
    }

    if (MODE == MOE_SYNC_BARRIER && !grid_barrier(a.words, a.err))
        return;

    // ------------------------------------------------------------ expert
    {
        const int64_t u0 = row_units * gw / nw, u1 = row_units * (gw + 1) / nw;
        for (int64_t u = u0; u < u1; ++u) {
            const int64_t s = u / a.upr;
            const int cu = (int)(u - s * a.upr);
            if (MODE == MOE_SYNC_WORD) {
                if (!__all_sync(FULL_MASK, wait_blocks(dwords, s, cu, a.spin_ns))) {
                    timed_out();
                    continue;
                }
            } else if (MODE == MOE_SYNC_BATCH) {
                const unsigned long long *w = dbatch + (size_t)s * a.nblk + cu;
                const bool r = spin_until(
                    [&] { return (uint32_t)(ld_acquire_u64(w) >> 32) == a.epoch; }, a.spin_ns,
                    give_up);
                if (!__all_sync(FULL_MASK, r)) {
                    timed_out();
                    continue;
                }
            }
            uint32_t csum = 0;
            bool ok = true;
            for (int q0 = 0; q0 < nsteps; q0 += DF_ILP) {
                uint4 d[DF_ILP];
                bool in[DF_ILP];
#pragma unroll
                for (int r = 0; r < DF_ILP; ++r) {
                    const int v = vec(cu, q0 + r);
                    in[r] = q0 + r < nsteps && v < C;
                    d[r] = make_uint4(0, 0, 0, 0);
                    if (in[r])
                        d[r] = MODE == MOE_SYNC_SENTINEL ? ld_volatile_v4(a.recv + s * C + v)
                                                         : ld_cg_v4(a.recv + s * C + v);
                }
#pragma unroll
                for (int r = 0; r < DF_ILP; ++r) {
                    if (!in[r])
                        continue;
                    uint4 *src = a.recv + s * C + vec(cu, q0 + r);
                    if (MODE == MOE_SYNC_SENTINEL) {
                        if (has_sentinel(d[r]) &&
                            !spin_until(
                                [&] {
                                    d[r] = ld_volatile_v4(src);
                                    return !has_sentinel(d[r]);
                                },
                                a.spin_ns, give_up || !ok)) {
                            ok = false;
                            continue;
                        }
                        st_volatile_v4(a.y + s * C + vec(cu, q0 + r), d[r]);
                        st_volatile_v4(src, sentinel4());
                    } else {
                        st_v4(a.y + s * C + vec(cu, q0 + r), d[r]);
                    }
                    csum += d[r].x;
                }
            }
            if (MODE == MOE_SYNC_SENTINEL) {
                if (!__all_sync(FULL_MASK, ok))
                    timed_out();
                continue;
            }
            if (MODE == MOE_SYNC_BARRIER)
                continue;
            if (MODE == MOE_SYNC_BATCH && lane == 0 &&
                csum != (uint32_t)ld_acquire_u64(dbatch + (size_t)s * a.nblk + cu))
                report(a.err, MOE_ERRBIT_CHECKSUM);
            __threadfence();
            __syncwarp();
            if (MODE == MOE_SYNC_WORD) {
                publish_blocks(ewords, s, cu);
            } else if (lane == 0) {
                st_relaxed_u64(ebatch + (size_t)s * a.nblk + cu,
                               ((unsigned long long)a.epoch << 32) | csum);
            }
        }
    }

    if (MODE == MOE_SYNC_BARRIER && !grid_barrier(a.words, a.err))
        return;

    // ------------------------------------------------------------ combine
    // A combine wait can sit behind one expert wait that ran out, so its
    // bound is three times the expert's.
    const uint64_t climit = 3 * a.spin_ns;
    {
        const int64_t u0 = tok_units * gw / nw, u1 = tok_units * (gw + 1) / nw;
        for (int64_t u = u0; u < u1; ++u) {
            const int64_t t = u / a.upr;
            const int cu = (int)(u - t * a.upr);
            const int32_t ms = lane < k ? ld_nc_s32(a.slot_of + t * k + lane) : 0;
            const float mw = lane < k ? ld_nc_f32(a.topk_w + t * k + lane) : 0.0f;
            bool ok = true;
            if (MODE == MOE_SYNC_WORD || MODE == MOE_SYNC_BATCH) {
                for (int j = 0; j < k && ok; ++j) {
                    const int32_t s = __shfl_sync(FULL_MASK, ms, j);
                    if ((unsigned)s >= (unsigned)N)
                        continue;
                    bool r;
                    if (MODE == MOE_SYNC_WORD) {
                        r = wait_blocks(ewords, s, cu, climit);
                    } else {
                        const unsigned long long *w = ebatch + (size_t)s * a.nblk + cu;
                        r = spin_until(
                            [&] { return (uint32_t)(ld_acquire_u64(w) >> 32) == a.epoch; },
                            climit, give_up);
                    }
                    ok = __all_sync(FULL_MASK, r);
                }
                if (!ok) {
                    timed_out();
                    continue;
                }
            }
            uint32_t csum = 0;  // lane j: the block markers of row j (BATCH)
            for (int q = 0; q < nsteps; ++q) {
                const int v = vec(cu, q);
                const bool in = v < C;
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    acc[i] = 0.0f;
                for (int jb = 0; jb < k; jb += DF_JG) {
                    // the rows of up to DF_JG slots are loaded before any is used
                    uint4 d[DF_JG];
#pragma unroll
                    for (int r = 0; r < DF_JG; ++r) {
                        const int32_t s = __shfl_sync(FULL_MASK, ms, (jb + r) & 31);
                        d[r] = make_uint4(0, 0, 0, 0);
                        if (in && jb + r < k && (unsigned)s < (unsigned)N)
                            d[r] = MODE == MOE_SYNC_SENTINEL ? ld_volatile_v4(a.y + (int64_t)s * C + v)
                                                             : ld_cg_v4(a.y + (int64_t)s * C + v);
                    }
#pragma unroll
                    for (int r = 0; r < DF_JG; ++r) {
                        const int j = jb + r;
                        const int32_t s = __shfl_sync(FULL_MASK, ms, j & 31);
                        const float w = __shfl_sync(FULL_MASK, mw, j & 31);
                        if (j >= k || (unsigned)s >= (unsigned)N)
                            continue;
                        if (MODE == MOE_SYNC_SENTINEL && in) {
                            uint4 *src = a.y + (int64_t)s * C + v;
                            if (has_sentinel(d[r]) &&
                                !spin_until(
                                    [&] {
                                        d[r] = ld_volatile_v4(src);
                                        return !has_sentinel(d[r]);
                                    },
                                    climit, give_up || !ok))
                                ok = false;
                            else
                                st_volatile_v4(src, sentinel4());
                        }
                        if (MODE == MOE_SYNC_BATCH) {
                            const uint32_t marker = __shfl_sync(FULL_MASK, d[r].x, 0);
                            if (lane == j)
                                csum += marker;
                        }
                        const uint32_t p[4] = {d[r].x, d[r].y, d[r].z, d[r].w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            acc[2 * h] = __fmaf_rn(w, bf16lo(p[h]), acc[2 * h]);
                            acc[2 * h + 1] = __fmaf_rn(w, bf16hi(p[h]), acc[2 * h + 1]);
                        }
                    }
                }
                if (!in || !ok)
                    continue;
                if (a.out_f32) {
                    float4 *o = static_cast<float4 *>(a.out) + (t * C + v) * 2;
                    st_v4(o, make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]),
                                        __float_as_uint(acc[2]), __float_as_uint(acc[3])));
                    st_v4(o + 1, make_uint4(__float_as_uint(acc[4]), __float_as_uint(acc[5]),
                                            __float_as_uint(acc[6]), __float_as_uint(acc[7])));
                } else {
                    uint32_t rr[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * h], acc[2 * h + 1]);
                        rr[h] = *reinterpret_cast<const uint32_t *>(&b);
                    }
                    st_v4(static_cast<uint4 *>(a.out) + t * C + v,
                          make_uint4(rr[0], rr[1], rr[2], rr[3]));
                }
            }
            if (MODE == MOE_SYNC_SENTINEL && !__all_sync(FULL_MASK, ok))
                timed_out();
            if (MODE == MOE_SYNC_BATCH && lane < k && (unsigned)ms < (unsigned)N &&
                csum != (uint32_t)ld_acquire_u64(ebatch + (size_t)ms * a.nblk + cu))
                report(a.err, MOE_ERRBIT_CHECKSUM);
        }
    }
}

// Geometry of granularity G: unit bytes, units per row, blocks per row; false
// when G is not a valid granularity for the mode.  A unit is one batch
// (BATCH) or max(G, DF_UNIT) bytes, and holds whole blocks.
static bool df_geometry(int mode, int H, int G, int &W, int &upr, int &nblk)
{
    const int rowbytes = 2 * H;
    if (G < 16 || G % 16 != 0)
        return false;
    if (mode == MOE_SYNC_BATCH) {
        if (G % DF_STEP != 0)
            return false;
        W = G;
    } else {
        if (G < DF_UNIT ? DF_UNIT % G != 0 : G % DF_STEP != 0)
            return false;
        W = G < DF_UNIT ? DF_UNIT : G;
    }
    upr = (rowbytes + W - 1) / W;
    nblk = (rowbytes + G - 1) / G;
    return true;
}

bool sync_granularity_ok(int mode, int H, int G)
{
    int W, upr, nblk;
    return df_geometry(mode, H, G, W, upr, nblk);
}

size_t sync_words(int T, int H, int k, int mode, int G)
{
    int W, upr, nblk;
    if (!df_geometry(mode, H, G, W, upr, nblk))
        return 0;
    const size_t N = (size_t)T * k;
    switch (mode) {
    case MOE_SYNC_WORD:
        return 2 * N * nblk;
    case MOE_SYNC_BATCH:
        return 4 * N * nblk;  // 64-bit words
    case MOE_SYNC_BARRIER:
        return 2;
    default:
        return 0;
    }
}

template <int MODE>
static cudaError_t launch_df(const DfArgs &a, cudaStream_t stream)
{
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, dispatch_combine_flagged_kernel<MODE>, DF_THREADS, 0);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    const int64_t units = (int64_t)a.T * a.k * a.upr;  // the largest phase
    int64_t grid = (int64_t)sm_count() * per_sm;       // every CTA co-resident
    const int64_t need = (units + DF_WARPS - 1) / DF_WARPS;
    if (need < grid)
        grid = need;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(DF_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dispatch_combine_flagged_kernel<MODE>, a);
}

cudaError_t launch_dispatch_combine_flagged(int T, int H, int k, const void *x,
                                            const int32_t *slot_of, const float *topk_w,
                                            void *recv, void *y, void *out, bool out_f32,
                                            int mode, int G, uint32_t *words, uint32_t epoch,
                                            uint64_t spin_limit_ns, int64_t skip_pair,
                                            uint32_t *err_word, cudaStream_t stream)
{
    if (T == 0)
        return cudaSuccess;
    DfArgs a;
    a.x = static_cast<const uint4 *>(x);
    a.slot_of = slot_of;
    a.topk_w = topk_w;
    a.recv = static_cast<uint4 *>(recv);
    a.y = static_cast<uint4 *>(y);
    a.out = out;
    a.out_f32 = out_f32 ? 1 : 0;
    a.T = T;
    a.k = k;
    a.C = H / 8;
    a.G = G;
    if (!df_geometry(mode, H, G, a.W, a.upr, a.nblk))
        return cudaErrorInvalidValue;
    a.words = words;
    a.epoch = epoch;
    a.spin_ns = spin_limit_ns;
    a.skip_pair = skip_pair;
    a.err = err_word;
    switch (mode) {
    case MOE_SYNC_WORD:
        return launch_df<MOE_SYNC_WORD>(a, stream);
    case MOE_SYNC_SENTINEL:
        return launch_df<MOE_SYNC_SENTINEL>(a, stream);
    case MOE_SYNC_BATCH:
        return launch_df<MOE_SYNC_BATCH>(a, stream);
    case MOE_SYNC_BARRIER:
        return launch_df<MOE_SYNC_BARRIER>(a, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace moe

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
// one row, W = max(G, 512), where G is the synchronisation granularity:
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
    int W;        // unit bytes, max(G, DF_STEP)
    int upr;      // units per row
    int nblk;     // G-byte blocks per row
    uint32_t *words;
    uint32_t epoch;
    uint64_t spin_ns;
    int64_t skip_pair;
    uint32_t *err;
};

template <int MODE>
__global__ void __launch_bounds__(DF_THREADS) dispatch_combine_flagged_kernel(const DfArgs a)
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
    // the G-block of this lane's vector in unit cu (G < 512: one step per
    // unit; G >= 512: the unit is one block)
    auto lane_block = [&](int cu) { return (cu * a.W + (a.G < DF_STEP ? lane * 16 : 0)) / a.G; };

    // ------------------------------------------------------------ produce
    {
        const int64_t u0 = tok_units * gw / nw, u1 = tok_units * (gw + 1) / nw;
        for (int64_t u = u0; u < u1; ++u) {
            const int64_t t = u / a.upr;
            const int cu = (int)(u - t * a.upr);
            const int32_t mine = lane < k ? ld_nc_s32(a.slot_of + t * k + lane) : -1;
            uint32_t csum = 0;
            bool hit = false;
            for (int q = 0; q < nsteps; ++q) {
                const int v = cu * vpu + q * 32 + lane;
                const bool in = v < C;
                const uint4 d = in ? ld_stream_v4(a.x + t * C + v) : make_uint4(0, 0, 0, 0);
                csum += d.x;  // lane 0: the first word of each 512-byte block
                hit |= in && has_sentinel(d);
                for (int j = 0; j < k; ++j) {
                    const int32_t s = __shfl_sync(FULL_MASK, mine, j);
                    if ((unsigned)s >= (unsigned)N) {
                        if (lane == 0 && cu == 0 && q == 0)
                            report(a.err, MOE_ERRBIT_BAD_INDEX);
                        continue;
                    }
                    if (!in)
                        continue;
                    if (MODE == MOE_SYNC_SENTINEL) {
                        if (t * k + j != a.skip_pair)
                            st_volatile_v4(a.recv + (int64_t)s * C + v, d);
                    } else {
                        st_v4(a.recv + (int64_t)s * C + v, d);
                    }
                }
            }
            if (MODE == MOE_SYNC_SENTINEL && __any_sync(FULL_MASK, hit) && lane == 0)
                report(a.err, MOE_ERRBIT_SENTINEL);
            if (MODE != MOE_SYNC_WORD && MODE != MOE_SYNC_BATCH)
                continue;
            __threadfence();  // this lane's row stores, before any word below
            __syncwarp();
            if (MODE == MOE_SYNC_WORD) {
                // one word per (slot row, block of this unit)
                const int b0 = cu * a.W / a.G;
                const int nb = a.G < DF_STEP ? DF_STEP / a.G : 1;
                for (int base = 0; base < k * nb; base += 32) {
                    const int f = base + lane;
                    const int j = f < k * nb ? f / nb : 0;
                    const int32_t s = __shfl_sync(FULL_MASK, mine, j);
                    const int b = b0 + f % nb;
                    if (f < k * nb && b < a.nblk && (unsigned)s < (unsigned)N &&
                        t * k + j != a.skip_pair)
                        st_relaxed_u32(dwords + (size_t)s * a.nblk + b, a.epoch);
                }
            } else {
                const uint32_t sum = __shfl_sync(FULL_MASK, csum, 0);
                if (lane < k && (unsigned)mine < (unsigned)N && t * k + lane != a.skip_pair)
                    st_relaxed_u64(dbatch + (size_t)mine * a.nblk + cu,
                                   ((unsigned long long)a.epoch << 32) | sum);
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
            const bool lane_has = cu * vpu + lane < C;  // this lane has a vector in the unit
            if (MODE == MOE_SYNC_WORD) {
                const uint32_t *w = dwords + (size_t)s * a.nblk + lane_block(cu);
                const bool r =
                    !lane_has ||
                    spin_until([&] { return ld_acquire_u32(w) == a.epoch; }, a.spin_ns, give_up);
                if (!__all_sync(FULL_MASK, r)) {
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
            for (int q = 0; q < nsteps; ++q) {
                const int v = cu * vpu + q * 32 + lane;
                if (v >= C)
                    continue;
                uint4 *src = a.recv + s * C + v;
                uint4 d;
                if (MODE == MOE_SYNC_SENTINEL) {
                    const bool r = spin_until(
                        [&] {
                            d = ld_volatile_v4(src);
                            return !has_sentinel(d);
                        },
                        a.spin_ns, give_up || !ok);
                    if (!r) {
                        ok = false;
                        continue;
                    }
                    st_volatile_v4(a.y + s * C + v, d);
                    st_volatile_v4(src, sentinel4());
                } else {
                    d = ld_cg_v4(src);
                    st_v4(a.y + s * C + v, d);
                }
                csum += d.x;
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
                const int b0 = cu * a.W / a.G;
                const int nb = a.G < DF_STEP ? DF_STEP / a.G : 1;
                if (lane < nb && b0 + lane < a.nblk)
                    st_relaxed_u32(ewords + (size_t)s * a.nblk + b0 + lane, a.epoch);
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
            const bool lane_has = cu * vpu + lane < C;
            bool ok = true;
            if (MODE == MOE_SYNC_WORD || MODE == MOE_SYNC_BATCH) {
                for (int j = 0; j < k && ok; ++j) {
                    const int32_t s = __shfl_sync(FULL_MASK, ms, j);
                    if ((unsigned)s >= (unsigned)N)
                        continue;
                    bool r;
                    if (MODE == MOE_SYNC_WORD) {
                        const uint32_t *w = ewords + (size_t)s * a.nblk + lane_block(cu);
                        r = !lane_has || spin_until([&] { return ld_acquire_u32(w) == a.epoch; },
                                                    climit, give_up);
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
                const int v = cu * vpu + q * 32 + lane;
                const bool in = v < C;
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    acc[i] = 0.0f;
                for (int j = 0; j < k; ++j) {
                    const int32_t s = __shfl_sync(FULL_MASK, ms, j);
                    const float w = __shfl_sync(FULL_MASK, mw, j);
                    if ((unsigned)s >= (unsigned)N)
                        continue;
                    uint4 d = make_uint4(0, 0, 0, 0);
                    if (in) {
                        uint4 *src = a.y + (int64_t)s * C + v;
                        if (MODE == MOE_SYNC_SENTINEL) {
                            const bool r = spin_until(
                                [&] {
                                    d = ld_volatile_v4(src);
                                    return !has_sentinel(d);
                                },
                                climit, give_up || !ok);
                            if (r)
                                st_volatile_v4(src, sentinel4());
                            else
                                ok = false;
                        } else {
                            d = ld_cg_v4(src);
                        }
                    }
                    if (MODE == MOE_SYNC_BATCH) {
                        const uint32_t marker = __shfl_sync(FULL_MASK, d.x, 0);
                        if (lane == j)
                            csum += marker;
                    }
                    const uint32_t p[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        acc[2 * h] = __fmaf_rn(w, bf16lo(p[h]), acc[2 * h]);
                        acc[2 * h + 1] = __fmaf_rn(w, bf16hi(p[h]), acc[2 * h + 1]);
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
// when G is not a valid granularity for the mode.
static bool df_geometry(int mode, int H, int G, int &W, int &upr, int &nblk)
{
    const int rowbytes = 2 * H;
    if (G < 16 || G % 16 != 0)
        return false;
    if (G < DF_STEP ? DF_STEP % G != 0 : G % DF_STEP != 0)
        return false;
    if (mode == MOE_SYNC_BATCH && G % DF_STEP != 0)
        return false;
    W = G < DF_STEP ? DF_STEP : G;
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

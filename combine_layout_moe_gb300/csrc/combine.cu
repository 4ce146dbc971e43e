// Combine: gather the k expert-output rows of each token and reduce them as a
// router-weighted fp32 sum (sm_103a).
//
// HyperParallel-MoE, section 2.2 (expert outputs weighted by routing scores and
// combined) and section 4.1 (top-k contributions accumulated according to the
// routing scores); RailWave, section 3 (combine uses the saved dispatch
// metadata to return rows to their token positions).
//
// GPU design: a pull through a bulk-copy pipeline.  One persistent CTA per SM
// owns a contiguous range of work units; a unit is one token and one chunk of
// CH bytes of each of its k source rows (k * CH ~ 32 KB, equal chunks).  A
// producer warp issues one cp.async.bulk per source row chunk into a ring of 6
// shared-memory stages, completing on the stage's "full" mbarrier, and writes
// the token's weights and valid-slot mask into the stage header; the stage's
// consumer warps (one group of up to three per stage, splitting its 16-byte
// vectors) wait on it, fold the k chunks into fp32 accumulators with one fused
// multiply-add per slot in slot order j = 0..k-1 (starting from +0), round
// once (nearest-even), store 16-byte vectors, and release the stage through
// its "empty" mbarrier.  The SM keeps up to ~190 KB of reads in flight without
// holding them in registers.  Every output element is written by exactly one
// lane: no atomics, deterministic.  Every mbarrier wait is bounded and reports
// MOE_ERRBIT_TIMEOUT if it gives up.
//
// For k > 32 a register-only variant (one warp per token and row chunk, KC
// source rows loaded at a time) does the same arithmetic in the same order.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"
#include "tma.cuh"

namespace moe {

constexpr int COMBINE_THREADS = 256;
// Rows in flight and 16-byte vectors per lane of the k > 32 combine
// (compile-time tunable; the defaults are the shipped configuration).  Four
// rows of four vectors (2 KB contiguous per row and warp) against eight rows
// of two (1 KB): 215 against 485 us on 2048 tokens, H = 7168, k = 40, each
// launch after a flush (0.83 against 0.37 of the copy peak); the smaller
// contiguous pieces read far slower from HBM.
#ifndef MOE_CF_KC
#define MOE_CF_KC 4
#endif
#ifndef MOE_CF_U
#define MOE_CF_U 4
#endif
#ifndef MOE_CF_MINB
#define MOE_CF_MINB 2
#endif

template <int KC, int U>
__global__ void __launch_bounds__(COMBINE_THREADS, MOE_CF_MINB)
    combine_kernel(const uint4 *__restrict__ y, const int32_t *__restrict__ slot_of,
                   const float *__restrict__ topk_w, void *__restrict__ out, int out_f32, int k,
                   int C, int groups, int64_t items, int N, uint32_t *err_word)
{
    // the slot indices and weights are reloaded when jb crosses a multiple
    // of 32, which jb (a multiple of KC) only lands on when KC divides 32
    static_assert(32 % KC == 0, "rows in flight must divide 32");
    wait_prior_grid();
    allow_next_grid();
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
        const float *wt = topk_w ? topk_w + t * k : nullptr;
        int32_t my_slot = 0;
        float my_w = 0.0f;
        for (int jb = 0; jb < k; jb += KC) {
            if ((jb & 31) == 0) {
                my_slot = jb + lane < k ? ld_nc_s32(so + jb + lane) : 0;
                my_w = jb + lane < k ? (topk_w ? ld_nc_f32(wt + jb + lane) : 1.0f) : 0.0f;
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

// Tunables (compile-time; the defaults are the shipped configuration).
#ifndef MOE_CT_CONSUMERS
#define MOE_CT_CONSUMERS 6
#endif
#ifndef MOE_CT_STAGES
#define MOE_CT_STAGES 6
#endif
#ifndef MOE_CT_STAGE_TARGET
#define MOE_CT_STAGE_TARGET 32768
#endif
#ifndef MOE_CT_MAX_WPS
#define MOE_CT_MAX_WPS 3
#endif
// CT_CONSUMERS consumer groups own the stages (stage s belongs to group
// s % CT_CONSUMERS); each group has `wps` warps (a launch argument, at most
// CT_MAX_WPS) that split a stage's 16-byte vectors between them, so a landed
// stage is folded and released sooner.
constexpr int CT_CONSUMERS = MOE_CT_CONSUMERS;
constexpr int CT_MAX_WPS = MOE_CT_MAX_WPS;
constexpr int CT_MAX_THREADS = 32 * (CT_CONSUMERS * CT_MAX_WPS + 1);
constexpr int CT_STAGES = MOE_CT_STAGES;
constexpr int CT_STAGE_TARGET = MOE_CT_STAGE_TARGET;  // bytes of k row chunks per stage
// Stage header words: [0, 32) slot weights, 32 valid-slot mask, 33 group-leader
// mask, [36, 68) member mask of each leader's group, [68, 100) its output row.
constexpr int CT_HDR_WORDS = 100;
constexpr int CT_HDR_OK = 32, CT_HDR_LEAD = 33, CT_HDR_MEMB = 36, CT_HDR_ROW = 68;
constexpr int CT_BAR_BYTES = 16 * CT_STAGES;
constexpr int CT_HDR_BYTES = 4 * CT_HDR_WORDS * CT_STAGES;
constexpr int CT_PREFIX = (CT_BAR_BYTES + CT_HDR_BYTES + 127) / 128 * 128;
static_assert(CT_STAGES % CT_CONSUMERS == 0, "each consumer group owns whole stages");

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// Advances a (token, chunk) cursor by `step` units.
__device__ __forceinline__ void advance(int64_t &t, int &c, int step, int nchunks)
{
    c += step;
    while (c >= nchunks) {
        c -= nchunks;
        ++t;
    }
}

// Per-CTA timestamps for tuning builds (-DMOE_TRACE): slot 8 + 4*cta + i of
// the 64-bit words after the error word (0 start, 1 first stage landed,
// 2 consumers done).
#ifdef MOE_TRACE
#define CT_TRACE(i)                                                                   \
    do {                                                                              \
        if (err_word)                                                                 \
            reinterpret_cast<unsigned long long *>(err_word)[8 + 4 * blockIdx.x + (i)] = \
                global_ns();                                                          \
    } while (0)
#else
#define CT_TRACE(i) \
    do {            \
    } while (0)
#endif

// Stores eight fp32 accumulators at element e0 of out: fp32, or rounded once
// to bf16 (nearest-even).
__device__ __forceinline__ void store_row8(void *out, int out_f32, int64_t e0, const float (&a)[8])
{
    if (out_f32) {
        float *o = static_cast<float *>(out) + e0;
        st_v4(o, make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                            __float_as_uint(a[3])));
        st_v4(o + 4, make_uint4(__float_as_uint(a[4]), __float_as_uint(a[5]),
                                __float_as_uint(a[6]), __float_as_uint(a[7])));
    } else {
        uint32_t rr[4];
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(a[2 * hh], a[2 * hh + 1]);
            rr[hh] = *reinterpret_cast<const uint32_t *>(&b);
        }
        st_v4(static_cast<__nv_bfloat16 *>(out) + e0, make_uint4(rr[0], rr[1], rr[2], rr[3]));
    }
}

// What a unit (token t, chunk c) of the bulk combine reduces.
//   CB_PLAIN  out[t] from slots slot_of[t, :], weights topk_w[t, :] (null: 1)
//   CB_COAL   the coalesced combine in one pass: the token's slots are grouped
//             by coalesced row crow[t, :]; each group's weighted sum (members
//             folded in increasing j) is rounded to bf16 and stored to
//             part[crow] -- the rank-side pre-reduction -- and out[t] is the
//             fp32 sum of those rounded rows in order of their first slot --
//             the token-side sum
enum { CB_PLAIN = 0, CB_COAL = 1 };

template <int KMAX, int MODE>
__global__ void __launch_bounds__(CT_MAX_THREADS, 1)
    combine_bulk_kernel(const uint8_t *__restrict__ y, const int32_t *__restrict__ slot_of,
                        const float *__restrict__ topk_w, const int32_t *__restrict__ crow,
                        void *__restrict__ part, void *__restrict__ out, int out_f32, int T,
                        int H, int k, int bound, int gbound, int CH, int nchunks, int64_t units,
                        int wps, uint32_t *err_word)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t bars = smem_addr(smem);
    float *hdr = reinterpret_cast<float *>(smem + CT_BAR_BYTES);  // [CT_STAGES][CT_HDR_WORDS]
    const uint32_t stages = bars + CT_PREFIX;
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (CT_STAGES + s); };
    const uint32_t stage_bytes = (uint32_t)k * CH;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t rowbytes = 2 * (int64_t)H;

    if (threadIdx.x == 0) {
        for (int s = 0; s < CT_STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), (uint32_t)wps);
        }
        mbar_fence_init();
    }
    __syncthreads();
    wait_prior_grid();
    allow_next_grid();
    if (threadIdx.x == 0)
        CT_TRACE(0);

    // this CTA's contiguous range of units (unit = token t, chunk c)
    const int64_t u0 = units * blockIdx.x / gridDim.x;
    const int64_t u1 = units * (blockIdx.x + 1) / gridDim.x;
    const int64_t nloc = u1 - u0;
    if (nloc <= 0)
        return;

    if (warp == 0) {
        // ---------------- producer: header + one bulk copy per source row chunk
        int64_t t = u0 / nchunks;
        int c = (int)(u0 - t * nchunks);
        const bool kl = lane < k;
        // this lane's slot of token `row`: source row, weight, whether it takes
        // part, and (CB_COAL) its coalesced row
        auto row_info = [&](int64_t row, int32_t &slot, float &w, bool &want, int32_t &grp) {
            slot = kl ? ld_nc_s32(slot_of + row * k + lane) : 0;
            // a null weight array means unit weights (the gradient of dispatch)
            w = kl ? (topk_w ? ld_nc_f32(topk_w + row * k + lane) : 1.0f) : 0.0f;
            want = kl;
            grp = MODE == CB_COAL && kl ? ld_nc_s32(crow + row * k + lane) : 0;
        };
        int32_t cur_slot, nxt_slot = 0, cur_grp, nxt_grp = 0;
        float cur_w, nxt_w = 0.0f;
        bool cur_want, nxt_want = false;
        row_info(t, cur_slot, cur_w, cur_want, cur_grp);
        if (t + 1 < T)
            row_info(t + 1, nxt_slot, nxt_w, nxt_want, nxt_grp);
        int64_t n = 0;
        bool timed_out = false;
        for (; n < nloc; ++n) {
            if (n > 0) {
                const int64_t t_prev = t;
                advance(t, c, 1, nchunks);
                if (t != t_prev) {
                    cur_slot = nxt_slot;
                    cur_w = nxt_w;
                    cur_want = nxt_want;
                    cur_grp = nxt_grp;
                    if (t + 1 < T)
                        row_info(t + 1, nxt_slot, nxt_w, nxt_want, nxt_grp);
                }
            }
            const int s = (int)(n % CT_STAGES);
            const uint32_t r = (uint32_t)(n / CT_STAGES);
            if (r > 0 && !mbar_wait(empty(s), (r - 1) & 1)) {
                timed_out = true;
                break;
            }
            const uint32_t cb = (uint32_t)min((int64_t)CH, rowbytes - (int64_t)c * CH);
            const bool ok = cur_want && (unsigned)cur_slot < (unsigned)bound &&
                            (MODE != CB_COAL || (unsigned)cur_grp < (unsigned)gbound);
            const unsigned okmask = __ballot_sync(FULL_MASK, ok);
            const unsigned wantmask = __ballot_sync(FULL_MASK, cur_want);
            float *h = hdr + s * CT_HDR_WORDS;
            if (MODE == CB_COAL) {
                // groups of valid slots sharing a coalesced row, led by their first slot
                const unsigned same = __match_any_sync(FULL_MASK, ok ? cur_grp : -1) & okmask;
                const bool lead = ok && (same & lanemask_lt()) == 0;
                uint32_t *hu = reinterpret_cast<uint32_t *>(h);
                hu[CT_HDR_MEMB + lane] = lead ? same : 0u;
                hu[CT_HDR_ROW + lane] = (uint32_t)cur_grp;
                const unsigned leaders = __ballot_sync(FULL_MASK, lead);
                if (lane == 0)
                    hu[CT_HDR_LEAD] = leaders;
                __syncwarp();
            }
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                const float wj = __shfl_sync(FULL_MASK, cur_w, j);
                if (lane == 0 && j < k)
                    h[j] = wj;
            }
            if (lane == 0) {
                reinterpret_cast<uint32_t *>(h)[CT_HDR_OK] = okmask;
                if (c == 0 && okmask != wantmask)
                    report(err_word, MOE_ERRBIT_BAD_INDEX);
                mbar_arrive_expect_tx(full(s), (uint32_t)__popc(okmask) * cb);
            }
            __syncwarp();
            if (ok)
                bulk_g2s(stages + (uint32_t)s * stage_bytes + (uint32_t)lane * CH,
                         y + (int64_t)cur_slot * rowbytes + (int64_t)c * CH, cb, full(s));
        }
        if (timed_out && lane == 0)
            report(err_word, MOE_ERRBIT_TIMEOUT);
        // drain: every copy this CTA issued has landed before it exits
        const int64_t first = n > CT_STAGES ? n - CT_STAGES : 0;
        for (int64_t m = first + lane; m < n; m += 32) {
            if (!mbar_wait(full((int)(m % CT_STAGES)), (uint32_t)(m / CT_STAGES) & 1))
                report(err_word, MOE_ERRBIT_TIMEOUT);
        }
        return;
    }

    // ---------------- consumers: unit n goes to group n % CT_CONSUMERS, whose
    // wps warps take every wps-th vector of it
    const int cw = (warp - 1) % CT_CONSUMERS;
    const int sub = (warp - 1) / CT_CONSUMERS;
    int64_t t = (u0 + cw) / nchunks;
    int c = (int)(u0 + cw - t * nchunks);
    for (int64_t n = cw; n < nloc; n += CT_CONSUMERS) {
        if (n > cw)
            advance(t, c, CT_CONSUMERS, nchunks);
        const int s = (int)(n % CT_STAGES);
        const uint32_t r = (uint32_t)(n / CT_STAGES);
        if (!mbar_wait(full(s), r & 1)) {
            if (lane == 0)
                report(err_word, MOE_ERRBIT_TIMEOUT);
            return;
        }
        if (n == 0 && sub == 0 && lane == 0)
            CT_TRACE(1);
        const float *h = hdr + s * CT_HDR_WORDS;
        const unsigned okmask = reinterpret_cast<const uint32_t *>(h)[CT_HDR_OK];
        float w[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
            w[j] = j < k ? h[j] : 0.0f;
        const int cb = (int)min((int64_t)CH, rowbytes - (int64_t)c * CH);
        const uint32_t base = stages + (uint32_t)s * stage_bytes;
        const int64_t out_elem0 = t * H + (int64_t)c * (CH / 2);
        if (MODE == CB_COAL) {
            // one partial row per group (members in increasing slot order),
            // and the token's sum of the rounded rows in group order
            const uint32_t *hu = reinterpret_cast<const uint32_t *>(h);
            const unsigned leaders = hu[CT_HDR_LEAD];
            const int64_t col0 = (int64_t)c * (CH / 2);
            for (int v = lane + 32 * sub; v < cb / 16; v += 32 * wps) {
                float tot[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    tot[i] = 0.0f;
                for (unsigned ls = leaders; ls; ls &= ls - 1) {
                    const int o = __ffs(ls) - 1;
                    float acc[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        acc[i] = 0.0f;
                    for (unsigned mm = hu[CT_HDR_MEMB + o]; mm; mm &= mm - 1) {
                        const int j = __ffs(mm) - 1;
                        const float wj = h[j];
                        const uint4 q = lds128(base + (uint32_t)j * CH + (uint32_t)v * 16);
                        const uint32_t p[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int hh = 0; hh < 4; ++hh) {
                            acc[2 * hh] = __fmaf_rn(wj, bf16lo(p[hh]), acc[2 * hh]);
                            acc[2 * hh + 1] = __fmaf_rn(wj, bf16hi(p[hh]), acc[2 * hh + 1]);
                        }
                    }
                    uint32_t rr[4];
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) {
                        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * hh], acc[2 * hh + 1]);
                        rr[hh] = *reinterpret_cast<const uint32_t *>(&b);
                    }
                    const int64_t e0 = (int64_t)(int32_t)hu[CT_HDR_ROW + o] * H + col0 + (int64_t)v * 8;
                    st_v4(static_cast<__nv_bfloat16 *>(part) + e0, make_uint4(rr[0], rr[1], rr[2], rr[3]));
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) {
                        tot[2 * hh] = __fadd_rn(tot[2 * hh], bf16lo(rr[hh]));
                        tot[2 * hh + 1] = __fadd_rn(tot[2 * hh + 1], bf16hi(rr[hh]));
                    }
                }
                store_row8(out, out_f32, out_elem0 + (int64_t)v * 8, tot);
            }
        } else {
            for (int v = lane + 32 * sub; v < cb / 16; v += 32 * wps) {
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    acc[i] = 0.0f;
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    if (j < k && ((okmask >> j) & 1u)) {
                        const uint4 q = lds128(base + (uint32_t)j * CH + (uint32_t)v * 16);
                        const uint32_t p[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int hh = 0; hh < 4; ++hh) {
                            acc[2 * hh] = __fmaf_rn(w[j], bf16lo(p[hh]), acc[2 * hh]);
                            acc[2 * hh + 1] = __fmaf_rn(w[j], bf16hi(p[hh]), acc[2 * hh + 1]);
                        }
                    }
                }
                store_row8(out, out_f32, out_elem0 + (int64_t)v * 8, acc);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(empty(s));
    }
#ifdef MOE_TRACE
    if (lane == 0)
        atomicMax(reinterpret_cast<unsigned long long *>(err_word) + 8 + 4 * blockIdx.x + 2,
                  (unsigned long long)global_ns());
#endif
}

// T tokens; slot indices must lie in [0, bound) and (CB_COAL) partial rows in
// [0, gbound).
template <int KMAX, int MODE>
static cudaError_t launch_combine_bulk(int T, int H, int k, const void *y,
                                       const int32_t *slot_of, const float *topk_w,
                                       const int32_t *crow, void *part, void *out, bool out_f32,
                                       int bound, int gbound, uint32_t *err_word,
                                       cudaStream_t stream)
{
    // Equal chunks (multiples of 16 bytes) of about CT_STAGE_TARGET / k bytes:
    // the fewest chunks per row whose k-row stage fits the target.
    const int rowbytes = 2 * H;
    const int vec = rowbytes / 16;
    int nchunks = (int)(((int64_t)rowbytes * k + CT_STAGE_TARGET - 1) / CT_STAGE_TARGET);
    if (nchunks < 1)
        nchunks = 1;
    if (nchunks > vec)
        nchunks = vec;
    const int CH = (vec + nchunks - 1) / nchunks * 16;
    nchunks = (rowbytes + CH - 1) / CH;
    const int64_t units = (int64_t)T * nchunks;
    const size_t smem = CT_PREFIX + (size_t)CT_STAGES * k * CH;
    // Consumer warps per stage.  Splitting a stage over three warps folds and
    // releases it sooner (measured, one GB300, each combine after a flush:
    // 1024 tokens, H = 7168, k = 8: 29.9 -> 27.2 us; 8192 tokens: 178 -> 166 us;
    // coalesced 1024 tokens: 60.0 -> 41.5 us).  The plain combine of k <= 2
    // keeps one warp per stage: its producer issues a unit every 2 rows and
    // loses issue slots to the extra warps (65536 tokens, H = 4096, k = 2:
    // 240 us with one warp, 280 us with three).
    const int wps = (MODE == CB_PLAIN && k <= 2) ? 1 : CT_MAX_WPS;
    const int threads = 32 * (CT_CONSUMERS * wps + 1);
    auto kern = combine_bulk_kernel<KMAX, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    int per_sm = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) !=
            cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    const int64_t g = units < cap ? units : cap;
    return launch_pdl(kern, dim3((unsigned)g), dim3(threads), smem, stream,
                      static_cast<const uint8_t *>(y), slot_of, topk_w, crow, part, out,
                      out_f32 ? 1 : 0, T, H, k, bound, gbound, CH, nchunks, units, wps,
                      err_word);
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
    return launch_pdl(combine_kernel<KC, U>, dim3(grid), dim3(COMBINE_THREADS), 0, stream,
                      static_cast<const uint4 *>(y), slot_of, topk_w, out, out_f32 ? 1 : 0, k, C,
                      groups, items, T * k, err_word);
}

// ---------------------------------------------------------------- backward
//
// HyperParallel-MoE, section 2.2 / Figure 2(b): the backward Dispatch is the
// gradient of the forward Combine.  Three forms: a warp per token for k <= 4,
// the bulk-copy pipeline below for 5 <= k <= 8, and for larger k (or when the
// pipeline does not fit in shared memory) one CTA per token: its 8 warps take
// equal slices of the row; per 16-byte vector a lane loads dout and the k rows of y
// (KMAX / 8 groups of 8 loads in flight), stores the k scaled copies
// dy[slot_of[t,j]] = bf16(w[t,j] * dout[t]) (one fp32 multiply, one rounding)
// and accumulates the k dot products <y[slot_of[t,j]], dout[t]> in fp32.  The
// partial dot products are reduced in a fixed order (xor-shuffle tree, then
// the warps in index order through shared memory): deterministic.
constexpr int CB_WARPS = 8;

// Minimum resident blocks of the CTA-per-token kernel for k <= 8
// (compile-time tunable; the default is the shipped configuration).  Three
// blocks cap it at 80 registers: a few bytes spill, but the extra resident
// warps keep more loads in flight (measured: 67 -> 55 us on a 1024-token,
// H = 7168, k = 8 batch).  The k <= 32 instance keeps one block: at 80
// registers its accumulators would spill heavily.
#ifndef MOE_CB_MINB
#define MOE_CB_MINB 3
#endif
// For 9 <= k <= 16 an instance sized to 16 slots at three resident blocks
// (80 registers and 220 bytes of spills; the k <= 32 instance needs 151
// registers and runs one block): measured
// on one GB300, each launch after a flush, 4096 tokens, H = 4096: k = 16 379
// -> 226 us, k = 12 346 -> 184 us; 2048 tokens, H = 7168, k = 10: 291 ->
// 158 us (one block of the 16-slot instance: 234, 203, 166 us).
#ifndef MOE_CB16_MINB
#define MOE_CB16_MINB 3
#endif
#ifndef MOE_CB_K16
#define MOE_CB_K16 1
#endif

template <int KMAX>
__global__ void __launch_bounds__(32 * CB_WARPS,
                                  KMAX <= 8 ? MOE_CB_MINB : KMAX <= 16 ? MOE_CB16_MINB : 1)
    combine_backward_kernel(const uint4 *__restrict__ dout, const uint4 *__restrict__ y,
                            const int32_t *__restrict__ slot_of, const float *__restrict__ topk_w,
                            uint4 *__restrict__ dy, float *__restrict__ dw, int T, int k, int C,
                            uint32_t *err_word)
{
    __shared__ float red[CB_WARPS][KMAX];
    wait_prior_grid();
    allow_next_grid();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int N = T * k;
    const int per = (C + CB_WARPS - 1) / CB_WARPS;
    const int c0 = warp * per, c1 = min(C, c0 + per);
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        const int32_t ms = lane < k ? ld_nc_s32(slot_of + t * k + lane) : -1;
        const float mw = lane < k ? ld_nc_f32(topk_w + t * k + lane) : 0.0f;
        const unsigned okmask = __ballot_sync(FULL_MASK, lane < k && (unsigned)ms < (unsigned)N);
        if (warp == 0 && lane == 0 && okmask != (k >= 32 ? FULL_MASK : ((1u << k) - 1u)))
            report(err_word, MOE_ERRBIT_BAD_INDEX);
        float part[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
            part[j] = 0.0f;
        // warp-uniform loop (the shuffles below need every lane); a lane past
        // the slice only skips its loads, arithmetic and stores
        for (int cb = c0; cb < c1; cb += 32) {
            const int c = cb + lane;
            const bool act = c < c1;
            const uint4 d = act ? ld_stream_v4(dout + t * C + c) : make_uint4(0, 0, 0, 0);
            const uint32_t dw4[4] = {d.x, d.y, d.z, d.w};
            float df[8];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                df[2 * h] = bf16lo(dw4[h]);
                df[2 * h + 1] = bf16hi(dw4[h]);
            }
#pragma unroll
            for (int jb = 0; jb < KMAX; jb += 8) {
                if (jb >= k)
                    break;
                uint4 yv[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int j = jb + q;
                    const int32_t s = __shfl_sync(FULL_MASK, ms, j & 31);
                    yv[q] = (act && y && j < k && ((okmask >> j) & 1u))
                                ? ld_stream_v4(y + (int64_t)s * C + c)
                                : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int j = jb + q;
                    const int32_t s = __shfl_sync(FULL_MASK, ms, j & 31);
                    const float w = __shfl_sync(FULL_MASK, mw, j & 31);
                    if (!act || j >= k || !((okmask >> j) & 1u))
                        continue;
                    const uint32_t yw[4] = {yv[q].x, yv[q].y, yv[q].z, yv[q].w};
                    uint32_t r[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        part[j] = __fmaf_rn(bf16lo(yw[h]), df[2 * h], part[j]);
                        part[j] = __fmaf_rn(bf16hi(yw[h]), df[2 * h + 1], part[j]);
                        const __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(w, df[2 * h]),
                                                                       __fmul_rn(w, df[2 * h + 1]));
                        r[h] = *reinterpret_cast<const uint32_t *>(&b);
                    }
                    st_v4(dy + (int64_t)s * C + c, make_uint4(r[0], r[1], r[2], r[3]));
                }
            }
        }
        if (dw) {
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                float v = part[j];
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1)
                    v += __shfl_xor_sync(FULL_MASK, v, o);
                if (lane == 0)
                    red[warp][j] = v;
            }
            __syncthreads();
            if (warp == 0 && lane < k) {
                float v = 0.0f;
#pragma unroll
                for (int w = 0; w < CB_WARPS; ++w)
                    v += red[w][lane];
                dw[t * k + lane] = v;
            }
            __syncthreads();
        }
    }
}

template <int KMAX>
static cudaError_t launch_combine_backward_t(int T, int H, int k, const void *dout, const void *y,
                                             const int32_t *slot_of, const float *topk_w,
                                             void *dy, float *dw, uint32_t *err_word,
                                             cudaStream_t stream)
{
    const int64_t g = T < 65535 * 32 ? T : 65535 * 32;
    return launch_pdl(combine_backward_kernel<KMAX>, dim3((unsigned)g), dim3(32 * CB_WARPS), 0,
                      stream, static_cast<const uint4 *>(dout), static_cast<const uint4 *>(y),
                      slot_of, topk_w, static_cast<uint4 *>(dy), dw, T, k, H / 8, err_word);
}

// Tunables of the small-k kernel (compile-time; the defaults are the shipped
// configuration): vectors per lane per iteration and minimum resident blocks,
// for k <= 2 and for k = 3..4.  Occupancy matters more than loads per lane
// here: 4 (k <= 2) and 3 (k <= 4) resident blocks took a 65536-token k = 2
// batch from 54 % to 98 % of HBM bandwidth, with a few bytes of spills.
#ifndef MOE_CBW2_UC
#define MOE_CBW2_UC 2
#endif
#ifndef MOE_CBW2_MINB
#define MOE_CBW2_MINB 4
#endif
#ifndef MOE_CBW4_UC
#define MOE_CBW4_UC 2
#endif
#ifndef MOE_CBW4_MINB
#define MOE_CBW4_MINB 3
#endif

// Small k (<= 4): too little work per token for a whole CTA.  The same
// arithmetic with WPT warps per token (here 1: each warp owns a token) and two
// vectors per iteration, so that a warp keeps 2 * (1 + k) loads in flight; the
// token's dot products are reduced by its warp's xor tree, then (when WPT > 1)
// by its warps in index order.
template <int KMAX, int UC, int MINB>
__global__ void __launch_bounds__(32 * CB_WARPS, MINB)
    combine_backward_warp_kernel(const uint4 *__restrict__ dout, const uint4 *__restrict__ y,
                            const int32_t *__restrict__ slot_of, const float *__restrict__ topk_w,
                            uint4 *__restrict__ dy, float *__restrict__ dw, int T, int k, int C,
                            int wpt, uint32_t *err_word)
{
    __shared__ float red[CB_WARPS][KMAX];
    wait_prior_grid();
    allow_next_grid();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int N = T * k;
    const int tpc = CB_WARPS / wpt;              // tokens per CTA pass
    const int slice = warp % wpt;
    const int per = (C + wpt - 1) / wpt;
    const int c0 = slice * per, c1 = min(C, c0 + per);
    const int64_t groups = ((int64_t)T + tpc - 1) / tpc;
    for (int64_t g = blockIdx.x; g < groups; g += gridDim.x) {
        const int64_t t = g * tpc + warp / wpt;
        const bool tok = t < T;                  // warp-uniform
        const int32_t ms = tok && lane < k ? ld_nc_s32(slot_of + t * k + lane) : -1;
        const float mw = tok && lane < k ? ld_nc_f32(topk_w + t * k + lane) : 0.0f;
        const unsigned okmask = __ballot_sync(FULL_MASK, lane < k && (unsigned)ms < (unsigned)N);
        if (tok && slice == 0 && lane == 0 &&
            okmask != (k >= 32 ? FULL_MASK : ((1u << k) - 1u)))
            report(err_word, MOE_ERRBIT_BAD_INDEX);
        float part[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
            part[j] = 0.0f;
        // warp-uniform loop (the shuffles below need every lane); a lane past
        // the slice only skips its loads, arithmetic and stores
        for (int cb = c0; tok && cb < c1; cb += 32 * UC) {
            bool act[UC];
            float df[UC][8];
#pragma unroll
            for (int u = 0; u < UC; ++u) {
                const int c = cb + 32 * u + lane;
                act[u] = c < c1;
                const uint4 d = act[u] ? ld_stream_v4(dout + t * C + c) : make_uint4(0, 0, 0, 0);
                const uint32_t d4[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    df[u][2 * h] = bf16lo(d4[h]);
                    df[u][2 * h + 1] = bf16hi(d4[h]);
                }
            }
            constexpr int QG = KMAX < 8 ? KMAX : 8;  // slots whose rows load together
#pragma unroll
            for (int jb = 0; jb < KMAX; jb += QG) {
                if (jb >= k)
                    break;
                uint4 yv[QG][UC];
#pragma unroll
                for (int q = 0; q < QG; ++q) {
                    const int j = jb + q;
                    const int32_t s = __shfl_sync(FULL_MASK, ms, j & 31);
                    const bool okj = y && j < k && ((okmask >> j) & 1u);
#pragma unroll
                    for (int u = 0; u < UC; ++u)
                        yv[q][u] = (okj && act[u])
                                       ? ld_stream_v4(y + (int64_t)s * C + cb + 32 * u + lane)
                                       : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int q = 0; q < QG; ++q) {
                    const int j = jb + q;
                    const int32_t s = __shfl_sync(FULL_MASK, ms, j & 31);
                    const float w = __shfl_sync(FULL_MASK, mw, j & 31);
                    if (j >= k || !((okmask >> j) & 1u))
                        continue;
#pragma unroll
                    for (int u = 0; u < UC; ++u) {
                        if (!act[u])
                            continue;
                        const uint32_t yw[4] = {yv[q][u].x, yv[q][u].y, yv[q][u].z, yv[q][u].w};
                        uint32_t r[4];
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            part[j] = __fmaf_rn(bf16lo(yw[h]), df[u][2 * h], part[j]);
                            part[j] = __fmaf_rn(bf16hi(yw[h]), df[u][2 * h + 1], part[j]);
                            const __nv_bfloat162 bb = __floats2bfloat162_rn(
                                __fmul_rn(w, df[u][2 * h]), __fmul_rn(w, df[u][2 * h + 1]));
                            r[h] = *reinterpret_cast<const uint32_t *>(&bb);
                        }
                        st_v4(dy + (int64_t)s * C + cb + 32 * u + lane, make_uint4(r[0], r[1], r[2], r[3]));
                    }
                }
            }
        }
        if (dw) {
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                float v = part[j];
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1)
                    v += __shfl_xor_sync(FULL_MASK, v, o);
                if (lane == 0)
                    red[warp][j] = v;
            }
            __syncthreads();
            if (tok && slice == 0 && lane < k) {
                float v = 0.0f;
                for (int i = 0; i < wpt; ++i)
                    v += red[warp + i][lane];
                dw[t * k + lane] = v;
            }
            __syncthreads();
        }
    }
}

template <int KMAX, int UC, int MINB>
static cudaError_t launch_combine_backward_warp(int T, int H, int k, const void *dout, const void *y,
                                                const int32_t *slot_of, const float *topk_w,
                                                void *dy, float *dw, uint32_t *err_word,
                                                cudaStream_t stream)
{
    auto kern = combine_backward_warp_kernel<KMAX, UC, MINB>;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * CB_WARPS, 0) !=
            cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t groups = ((int64_t)T + CB_WARPS - 1) / CB_WARPS;  // one warp per token
    const int64_t cap = (int64_t)sm_count() * per_sm * 4;
    const int64_t g = groups < cap ? groups : cap;
    return launch_pdl(kern, dim3((unsigned)g), dim3(32 * CB_WARPS), 0, stream,
                      static_cast<const uint4 *>(dout), static_cast<const uint4 *>(y), slot_of,
                      topk_w, static_cast<uint4 *>(dy), dw, T, k, H / 8, 1, err_word);
}

// ------------------------------------------------- backward through bulk copies
//
// The same gradient as combine_backward_kernel, on the forward combine's
// pipeline: one persistent CTA per SM over a contiguous range of units (unit =
// token t, chunk c of CH bytes).  The producer warp loads dout[t]'s chunk and
// the k chunks of y[slot_of[t, j]] into a stage (one cp.async.bulk each) and
// writes the weights and slots into its header; the stage's consumer group
// stores dy[slot_of[t, j]] = bf16(w[t, j] * dout[t]) for its chunk and folds
// the k dot-product partials of the chunk (per lane, then the group's warps in
// index order).
//
// dw without a workspace, deterministic: each unit's k partials go to a small
// shared-memory ring indexed by token; the group that completes a token's last
// chunk in this CTA sums the token's chunk partials in chunk order and adds
// the sum to dw, which the launch zero-fills.  The grid is at most T CTAs, so a
// token's units lie in at most two CTAs: dw gets at most two additions onto
// zero, and fp32 addition of two values does not depend on their order.  A
// ring slot is reused by token t + CB_RING only after every unit of token t
// was released (the finalisation precedes the release, and the producer
// refills a stage only after its release), which CB_RING >= CT_STAGES makes
// sufficient.  The same release order protects a group's reduction slots and
// counter: its next unit's stage is refilled only after the group's last warp
// has read them and arrived.
constexpr int CB_RING = 8;
static_assert(CB_RING >= CT_STAGES, "ring covers the units in flight");
constexpr int CB_HDR_WORDS = 68;  // [0, 32) weights, [32, 64) slots, 64 valid-slot mask
constexpr int CB_HDR_SLOT = 32, CB_HDR_OK = 64;

template <int KMAX>
__global__ void __launch_bounds__(CT_MAX_THREADS, 1)
    combine_backward_bulk_kernel(const uint8_t *__restrict__ dout, const uint8_t *__restrict__ y,
                                 const int32_t *__restrict__ slot_of,
                                 const float *__restrict__ topk_w, uint8_t *__restrict__ dy,
                                 float *__restrict__ dw, int T, int H, int k, int N, int CH,
                                 int nchunks, int64_t units, int wps, uint32_t *err_word)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t bars = smem_addr(smem);
    uint32_t *hdr = reinterpret_cast<uint32_t *>(smem + CT_BAR_BYTES);  // [CT_STAGES][CB_HDR_WORDS]
    float *red = reinterpret_cast<float *>(hdr + CT_STAGES * CB_HDR_WORDS);  // [CT_CONSUMERS][CT_MAX_WPS][KMAX]
    int32_t *gcnt = reinterpret_cast<int32_t *>(red + CT_CONSUMERS * CT_MAX_WPS * KMAX);  // [CT_CONSUMERS]
    int32_t *cnt = gcnt + CT_CONSUMERS;                      // [CB_RING]
    float *ring = reinterpret_cast<float *>(cnt + CB_RING);  // [CB_RING][nchunks][k]
    const int ring_words = CB_RING * nchunks * k;
    const uint32_t prefix =
        (uint32_t)((CT_BAR_BYTES + 4 * (CT_STAGES * CB_HDR_WORDS + CT_CONSUMERS * CT_MAX_WPS * KMAX +
                                        CT_CONSUMERS + CB_RING + ring_words) + 127) / 128 * 128);
    const uint32_t stages = bars + prefix;
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (CT_STAGES + s); };
    const bool want_dw = dw != nullptr && y != nullptr;
    const uint32_t stage_bytes = (uint32_t)(want_dw ? 1 + k : 1) * CH;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t rowbytes = 2 * (int64_t)H;

    if (threadIdx.x == 0) {
        for (int s = 0; s < CT_STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), (uint32_t)wps);
        }
        mbar_fence_init();
    }
    for (int i = threadIdx.x; i < CT_CONSUMERS + CB_RING; i += blockDim.x)
        gcnt[i] = 0;  // gcnt and cnt are contiguous
    __syncthreads();
    wait_prior_grid();
    allow_next_grid();

    const int64_t u0 = units * blockIdx.x / gridDim.x;
    const int64_t u1 = units * (blockIdx.x + 1) / gridDim.x;
    const int64_t nloc = u1 - u0;
    if (nloc <= 0)
        return;
    const int64_t t_first = u0 / nchunks;

    if (warp == 0) {
        // ---------------- producer
        int64_t t = t_first;
        int c = (int)(u0 - t * nchunks);
        const bool kl = lane < k;
        int32_t cur_s = kl ? ld_nc_s32(slot_of + t * k + lane) : -1;
        float cur_w = kl ? ld_nc_f32(topk_w + t * k + lane) : 0.0f;
        int32_t nxt_s = kl && t + 1 < T ? ld_nc_s32(slot_of + (t + 1) * k + lane) : -1;
        float nxt_w = kl && t + 1 < T ? ld_nc_f32(topk_w + (t + 1) * k + lane) : 0.0f;
        int64_t n = 0;
        bool timed_out = false;
        for (; n < nloc; ++n) {
            if (n > 0 && ++c == nchunks) {
                c = 0;
                ++t;
                cur_s = nxt_s;
                cur_w = nxt_w;
                nxt_s = kl && t + 1 < T ? ld_nc_s32(slot_of + (t + 1) * k + lane) : -1;
                nxt_w = kl && t + 1 < T ? ld_nc_f32(topk_w + (t + 1) * k + lane) : 0.0f;
            }
            const int s = (int)(n % CT_STAGES);
            const uint32_t r = (uint32_t)(n / CT_STAGES);
            if (r > 0 && !mbar_wait(empty(s), (r - 1) & 1)) {
                timed_out = true;
                break;
            }
            const uint32_t cb = (uint32_t)min((int64_t)CH, rowbytes - (int64_t)c * CH);
            const bool ok = kl && (unsigned)cur_s < (unsigned)N;
            const unsigned okmask = __ballot_sync(FULL_MASK, ok);
            uint32_t *h = hdr + s * CB_HDR_WORDS;
            if (kl) {
                h[lane] = __float_as_uint(cur_w);
                h[CB_HDR_SLOT + lane] = (uint32_t)cur_s;
            }
            if (lane == 0)
                h[CB_HDR_OK] = okmask;
            __syncwarp();  // the header is written before lane 0 arrives
            if (lane == 0) {
                const unsigned kmask = k >= 32 ? FULL_MASK : (1u << k) - 1u;
                if (c == 0 && okmask != kmask)
                    report(err_word, MOE_ERRBIT_BAD_INDEX);
                const uint32_t nrows = want_dw ? 1u + (uint32_t)__popc(okmask) : 1u;
                mbar_arrive_expect_tx(full(s), nrows * cb);
                bulk_g2s(stages + (uint32_t)s * stage_bytes,
                         dout + t * rowbytes + (int64_t)c * CH, cb, full(s));
            }
            __syncwarp();
            if (want_dw && ok)
                bulk_g2s(stages + (uint32_t)s * stage_bytes + (uint32_t)(1 + lane) * CH,
                         y + (int64_t)cur_s * rowbytes + (int64_t)c * CH, cb, full(s));
        }
        if (timed_out && lane == 0)
            report(err_word, MOE_ERRBIT_TIMEOUT);
        const int64_t first = n > CT_STAGES ? n - CT_STAGES : 0;
        for (int64_t m = first + lane; m < n; m += 32) {
            if (!mbar_wait(full((int)(m % CT_STAGES)), (uint32_t)(m / CT_STAGES) & 1))
                report(err_word, MOE_ERRBIT_TIMEOUT);
        }
        return;
    }

    // ---------------- consumers: unit n goes to group n % CT_CONSUMERS
    const int cw = (warp - 1) % CT_CONSUMERS;
    const int sub = (warp - 1) / CT_CONSUMERS;
    int64_t t = (u0 + cw) / nchunks;
    int c = (int)(u0 + cw - t * nchunks);
    for (int64_t n = cw; n < nloc; n += CT_CONSUMERS) {
        if (n > cw)
            advance(t, c, CT_CONSUMERS, nchunks);
        const int s = (int)(n % CT_STAGES);
        if (!mbar_wait(full(s), (uint32_t)(n / CT_STAGES) & 1)) {
            if (lane == 0)
                report(err_word, MOE_ERRBIT_TIMEOUT);
            return;
        }
        const uint32_t *h = hdr + s * CB_HDR_WORDS;
        const unsigned okmask = h[CB_HDR_OK];
        float w[KMAX];
        int32_t sl[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            w[j] = j < k ? __uint_as_float(h[j]) : 0.0f;
            sl[j] = j < k ? (int32_t)h[CB_HDR_SLOT + j] : 0;
        }
        const int cb = (int)min((int64_t)CH, rowbytes - (int64_t)c * CH);
        const uint32_t base = stages + (uint32_t)s * stage_bytes;
        float part[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
            part[j] = 0.0f;
        for (int v = lane + 32 * sub; v < cb / 16; v += 32 * wps) {
            const uint4 d = lds128(base + (uint32_t)v * 16);
            const uint32_t d4[4] = {d.x, d.y, d.z, d.w};
            float df[8];
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
                df[2 * hh] = bf16lo(d4[hh]);
                df[2 * hh + 1] = bf16hi(d4[hh]);
            }
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (j >= k || !((okmask >> j) & 1u))
                    continue;
                uint32_t rr[4];
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) {
                    const __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(w[j], df[2 * hh]),
                                                                   __fmul_rn(w[j], df[2 * hh + 1]));
                    rr[hh] = *reinterpret_cast<const uint32_t *>(&b);
                }
                st_v4(dy + (int64_t)sl[j] * rowbytes + (int64_t)c * CH + (int64_t)v * 16,
                      make_uint4(rr[0], rr[1], rr[2], rr[3]));
                if (want_dw) {
                    const uint4 q = lds128(base + (uint32_t)(1 + j) * CH + (uint32_t)v * 16);
                    const uint32_t p[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) {
                        part[j] = __fmaf_rn(bf16lo(p[hh]), df[2 * hh], part[j]);
                        part[j] = __fmaf_rn(bf16hi(p[hh]), df[2 * hh + 1], part[j]);
                    }
                }
            }
        }
        if (want_dw) {
            // the unit's partials: each warp's xor tree; the group's last warp
            // to get here adds the warps' sums in index order and files them in
            // the token's ring entry (no barrier: a warp that gives up on a
            // wait cannot leave the others blocked)
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                float v = part[j];
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1)
                    v += __shfl_xor_sync(FULL_MASK, v, o);
                part[j] = v;
            }
            float *rg = red + (cw * CT_MAX_WPS) * KMAX;
            if (lane == 0) {
#pragma unroll
                for (int j = 0; j < KMAX; ++j)
                    rg[sub * KMAX + j] = part[j];
            }
            __syncwarp();
            __threadfence_block();
            int last = 0;
            if (lane == 0)
                last = atomicAdd(gcnt + cw, 1) + 1 == wps;
            last = __shfl_sync(FULL_MASK, last, 0);
            if (last) {
                __threadfence_block();
                const int ts = (int)((t - t_first) % CB_RING);
                float *acc = ring + (ts * nchunks) * k;
                if (lane < k) {
                    float v = 0.0f;
                    for (int q = 0; q < wps; ++q)
                        v += rg[q * KMAX + lane];
                    acc[c * k + lane] = v;
                }
                __syncwarp();
                __threadfence_block();
                int done = 0;
                if (lane == 0) {
                    gcnt[cw] = 0;
                    const int64_t lo = max(u0, t * nchunks), hi = min(u1, (t + 1) * nchunks);
                    done = atomicAdd(cnt + ts, 1) + 1 == (int)(hi - lo);
                }
                done = __shfl_sync(FULL_MASK, done, 0);
                if (done) {
                    // every chunk of token t in this CTA is filed: their sum in
                    // chunk order
                    __threadfence_block();
                    const int c_lo = (int)(max(u0, t * nchunks) - t * nchunks);
                    const int c_hi = (int)(min(u1, (t + 1) * nchunks) - t * nchunks);
                    if (lane < k && ((okmask >> lane) & 1u)) {
                        float v = 0.0f;
                        for (int q = c_lo; q < c_hi; ++q)
                            v += acc[q * k + lane];
                        atomicAdd(dw + t * k + lane, v);
                    }
                    if (lane == 0)
                        cnt[ts] = 0;
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(empty(s));
    }
}

// Returns cudaErrorNotSupported (nothing launched) when the ring and stages do
// not fit in shared memory; the caller then takes the CTA-per-token kernel.
template <int KMAX>
static cudaError_t launch_combine_backward_bulk(int T, int H, int k, const void *dout,
                                                const void *y, const int32_t *slot_of,
                                                const float *topk_w, void *dy, float *dw,
                                                uint32_t *err_word, cudaStream_t stream)
{
    const bool want_dw = dw != nullptr && y != nullptr;
    const int rows = want_dw ? 1 + k : 1;  // chunks per stage: dout and the k rows of y
    const int rowbytes = 2 * H;
    const int vec = rowbytes / 16;
    int nchunks = (int)(((int64_t)rowbytes * rows + CT_STAGE_TARGET - 1) / CT_STAGE_TARGET);
    nchunks = max(1, min(nchunks, vec));
    const int CH = (vec + nchunks - 1) / nchunks * 16;
    nchunks = (rowbytes + CH - 1) / CH;
    const int64_t units = (int64_t)T * nchunks;
    // must match the kernel's layout: barriers, headers, reduction slots,
    // group counters, ring counters, ring
    const size_t prefix =
        ((size_t)CT_BAR_BYTES + 4 * ((size_t)CT_STAGES * CB_HDR_WORDS + CT_CONSUMERS * CT_MAX_WPS * KMAX +
                                     CT_CONSUMERS + CB_RING + (size_t)CB_RING * nchunks * k) + 127) /
        128 * 128;
    const size_t smem = prefix + (size_t)CT_STAGES * rows * CH;
    int dev = 0, smem_max = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
        return cudaErrorNotSupported;
    if (smem > (size_t)smem_max)
        return cudaErrorNotSupported;
    auto kern = combine_backward_bulk_kernel<KMAX>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    if (want_dw && (e = cudaMemsetAsync(dw, 0, sizeof(float) * (size_t)T * k, stream)) !=
                       cudaSuccess)
        return e;
    const int wps = CT_MAX_WPS;
    const int threads = 32 * (CT_CONSUMERS * wps + 1);
    // at most T CTAs: every CTA holds at least nchunks units, so a token's
    // units lie in at most two CTAs (see above)
    int64_t g = sm_count();
    if (g > T)
        g = T;
    if (g > units)
        g = units;
    return launch_pdl(kern, dim3((unsigned)g), dim3(threads), smem, stream,
                      static_cast<const uint8_t *>(dout), static_cast<const uint8_t *>(y),
                      slot_of, topk_w, static_cast<uint8_t *>(dy), want_dw ? dw : nullptr, T, H,
                      k, T * k, CH, nchunks, units, wps, err_word);
}

cudaError_t launch_combine_backward(int T, int H, int k, const void *dout, const void *y,
                                    const int32_t *slot_of, const float *topk_w, void *dy,
                                    float *dw, uint32_t *err_word, cudaStream_t stream)
{
    if (T == 0)
        return cudaSuccess;
    if (k <= 2)
        return launch_combine_backward_warp<2, MOE_CBW2_UC, MOE_CBW2_MINB>(
            T, H, k, dout, y, slot_of, topk_w, dy, dw, err_word, stream);
    if (k <= 4)
        return launch_combine_backward_warp<4, MOE_CBW4_UC, MOE_CBW4_MINB>(
            T, H, k, dout, y, slot_of, topk_w, dy, dw, err_word, stream);
    if (k <= 8) {
        // the bulk-copy pipeline, unless its ring and stages do not fit (k > 8
        // would hold 3 x k values per lane in registers: it spills)
        const cudaError_t e = launch_combine_backward_bulk<8>(T, H, k, dout, y, slot_of, topk_w,
                                                              dy, dw, err_word, stream);
        if (e != cudaErrorNotSupported)
            return e;
        return launch_combine_backward_t<8>(T, H, k, dout, y, slot_of, topk_w, dy, dw, err_word,
                                            stream);
    }
    if (MOE_CB_K16 && k <= 16)
        return launch_combine_backward_t<16>(T, H, k, dout, y, slot_of, topk_w, dy, dw,
                                             err_word, stream);
    return launch_combine_backward_t<32>(T, H, k, dout, y, slot_of, topk_w, dy, dw, err_word,
                                         stream);
}

cudaError_t launch_combine(int T, int H, int k, const void *y, const int32_t *slot_of,
                           const float *topk_w, void *out, bool out_f32, uint32_t *err_word,
                           cudaStream_t stream)
{
    if (T == 0)
        return cudaSuccess;
    const int N = T * k;
    if (k <= 8)
        return launch_combine_bulk<8, CB_PLAIN>(T, H, k, y, slot_of, topk_w, nullptr, nullptr,
                                                out, out_f32, N, 0, err_word, stream);
    if (k <= 32)
        return launch_combine_bulk<32, CB_PLAIN>(T, H, k, y, slot_of, topk_w, nullptr, nullptr,
                                                 out, out_f32, N, 0, err_word, stream);
    // KC x U ~ 16 independent 16-byte loads in flight per lane.
    return launch_combine_t<MOE_CF_KC, MOE_CF_U>(T, H, k, y, slot_of, topk_w, out, out_f32,
                                                  err_word, stream);
}

// Coalesced combine, one pass: the rank-side pre-reduction into `partial` (one
// bf16 row per coalesced row) and the token-side sum of the rounded rows.
template <int KMAX>
static cudaError_t launch_combine_coalesced_t(int T, int H, int k, const void *y,
                                              const int32_t *slot_of, const float *topk_w,
                                              const int32_t *crow, int rows, void *partial,
                                              void *out, bool out_f32, uint32_t *err_word,
                                              cudaStream_t stream)
{
    return launch_combine_bulk<KMAX, CB_COAL>(T, H, k, y, slot_of, topk_w, crow, partial, out,
                                              out_f32, T * k, rows, err_word, stream);
}

cudaError_t launch_combine_coalesced(int T, int H, int k, const void *y, const int32_t *slot_of,
                                     const float *topk_w, const int32_t *crow, int rows,
                                     void *partial, void *out, bool out_f32, uint32_t *err_word,
                                     cudaStream_t stream)
{
    if (T == 0)
        return cudaSuccess;
    if (k <= 8)
        return launch_combine_coalesced_t<8>(T, H, k, y, slot_of, topk_w, crow, rows, partial,
                                             out, out_f32, err_word, stream);
    return launch_combine_coalesced_t<32>(T, H, k, y, slot_of, topk_w, crow, rows, partial, out,
                                          out_f32, err_word, stream);
}

}  // namespace moe

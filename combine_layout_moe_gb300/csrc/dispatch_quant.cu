// Dispatch with fused FP8-E4M3 block quantisation (sm_103a).
//
// UBEP, Table 3: the DeepSeek-R1 / V3.2 deployments run W8A8; the pages give
// no further recipe.  Reading: per token row, 1 x 128-channel blocks; scale =
// amax / 448 and inv = 448 / amax, each one correctly rounded fp32 division;
// code = e4m3(x * inv), one rounded fp32 multiply then a saturating
// nearest-even conversion.  The token is quantised once and the same codes
// and scales go to all k slots (or, COAL, once per coalesced row).
//
// GPU design: a warp item is one token and 2U blocks of 128 channels (U
// 16-byte vectors of x in flight per lane, in adjacent pairs); eight lanes own
// a block (8 lanes x 16 channels), reduce its amax with xor-shuffles, and
// store 16-byte code words and one fp32 scale per block to every destination
// row.  When the
// items take more than QUANT_DYN_MIN_ROUNDS rounds of the resident warps, the
// warps take QUANT_STATIC_PCT percent of them in interleaved rounds (warp w:
// items w, w + warps, ...), then draw the rest from the launch's pool
// (sched.cuh), the next draw requested while the current items are
// processed; a draw takes enough items to cover SCHED_DRAW_BYTES of traffic,
// which keeps the draws on the pool's one counter far apart.
#include <cuda_fp8.h>

#include "common.cuh"
#include "launch.h"
#include "sched.cuh"

namespace moe {

constexpr int QUANT_THREADS = 256;

// The channel encoding of the quantised dispatch: two fp32 values to two
// E4M3 codes (low byte first), nearest-even, saturating to +-448.  One
// routine for the kernel and for moe_e4m3_encode_bits, the diagnostic entry
// point that lets the tests check it on every fp32 input.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    float2 g;
    g.x = lo;
    g.y = hi;
    return __nv_cvt_float2_to_fp8x2(g, __NV_SATFINITE, __NV_E4M3) & 0xffffu;
}
// 16-lane quantisation blocks per half-warp per item (compile-time tunable;
// the default is the shipped configuration).  Four keep 64 bytes of x in
// flight per lane (measured on one GB300, each launch after a flush: 65536
// tokens, H = 4096, k = 2: 227 us with 2, 204 us with 4; 8192 tokens,
// H = 7168, k = 8: 104-105 us with either; 6 and 8 were slower at H = 7168).
#ifndef MOE_QUANT_U
#define MOE_QUANT_U 4
#endif
constexpr int QUANT_U = MOE_QUANT_U;
#ifndef MOE_QUANT_STATIC_PCT
#define MOE_QUANT_STATIC_PCT 50
#endif
#ifndef MOE_QUANT_DYN_MIN_ROUNDS
#define MOE_QUANT_DYN_MIN_ROUNDS 4
#endif
constexpr int QUANT_STATIC_PCT = MOE_QUANT_STATIC_PCT;
constexpr int QUANT_DYN_MIN_ROUNDS = MOE_QUANT_DYN_MIN_ROUNDS;
__device__ SchedSlot g_quant_sched[SCHED_SLOTS];
static std::atomic<unsigned> g_quant_seq{0};

// FP8: eight lanes own one 128-channel block (8 lanes x 16 channels: two
// adjacent 16-byte vectors of x, whose 16 codes go out in one 16-byte store
// per slot).  The amax is reduced with xor-shuffles inside the eight lanes;
// scale and reciprocal are each one correctly rounded fp32 division; each
// channel is one rounded fp32 multiply followed by a saturating nearest-even
// E4M3 conversion.
template <int U, bool COAL, bool POOL>
__global__ void __launch_bounds__(QUANT_THREADS)
    dispatch_fp8_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ slot_of,
                        uint8_t *__restrict__ recv_q, float *__restrict__ recv_scales, int k,
                        int H, int groups, int64_t items, int64_t pool_from, int grab,
                        int sched_slot, int N, int prefetch_x, uint32_t *err_word)
{
    static_assert(U % 2 == 0, "vectors go in adjacent pairs");
    constexpr int P = U / 2;  // vector pairs per lane per item
    // POOL: items from pool_from on are drawn; else every item is taken in
    // interleaved rounds and the pool code is compiled out
    const int64_t static_items = POOL ? pool_from : items;
    // prefetch_x: the first item's x is loaded and quantised before waiting
    // for the previous grid, and only the slot map and the stores wait.  Only
    // for a launch whose previous grid is this library's layout kernel: that
    // kernel lets dependents launch only after its own wait, so x and the
    // receive buffers are final; the slot map is not.
    bool waited = !prefetch_x;
    if (waited) {
        wait_prior_grid();
        allow_next_grid();
    }
    const int lane = threadIdx.x & 31;
    const int C = H >> 3;    // 16-byte vectors per row
    const int B = H >> 7;    // 128-channel blocks per row
    const int64_t nwarps = (int64_t)gridDim.x * (QUANT_THREADS / 32);
    // the item source (warp-uniform): interleaved rounds below static_items,
    // then ranges drawn from the pool [static_items, items)
    SchedSlot *sched = g_quant_sched + sched_slot;
    unsigned long long drawn = 0;  // lane 0: the pending draw's pool offset
    bool pending = false;
    int64_t d_end = 0;
    auto request = [&]() {
        if (lane == 0)
            drawn = atomicAdd(&sched->taken, (unsigned long long)grab);
        pending = true;
    };
    auto draw = [&]() -> int64_t {
        if (!pending)
            request();
        const int64_t v = static_items + (int64_t)__shfl_sync(FULL_MASK, drawn, 0);
        pending = false;
        if (v >= items)
            return -1;
        d_end = min(v + (int64_t)grab, items);
        return v;
    };
    auto next_item = [&](int64_t it) -> int64_t {
        if (it < static_items) {
            if (it + nwarps < static_items)
                return it + nwarps;
        } else if (it + 1 < d_end) {
            return it + 1;
        }
        return static_items < items ? draw() : -1;
    };
    int64_t it0 = (int64_t)blockIdx.x * (QUANT_THREADS / 32) + (threadIdx.x >> 5);
    if (it0 >= static_items)
        it0 = static_items < items ? draw() : -1;
    for (int64_t it = it0; it >= 0; it = next_item(it)) {
        // the next draw travels while this item is processed
        if (!pending && (it >= static_items ? it + 1 >= d_end : it + nwarps >= static_items) &&
            static_items < items)
            request();
        const int64_t t = it / groups;
        // lane `lane` holds pairs of adjacent vectors (16 channels): pair p is
        // vectors base + 64p + 2 lane + {0, 1}; eight lanes cover a block
        const int base = (int)(it - t * groups) * (32 * U);
        const uint4 *src = x + t * C;
        uint4 v[U];
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int c = base + 64 * p + 2 * lane;
            const bool in = c < C;  // C is a multiple of 16: a pair is whole or absent
            v[2 * p] = in ? ld_stream_v4(src + c) : make_uint4(0, 0, 0, 0);
            v[2 * p + 1] = in ? ld_stream_v4(src + c + 1) : make_uint4(0, 0, 0, 0);
        }

        uint4 code[P];
        float scale[P];
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const uint32_t w[8] = {v[2 * p].x,     v[2 * p].y,     v[2 * p].z,     v[2 * p].w,
                                   v[2 * p + 1].x, v[2 * p + 1].y, v[2 * p + 1].z, v[2 * p + 1].w};
            float f[16];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                f[2 * q] = bf16lo(w[q]);
                f[2 * q + 1] = bf16hi(w[q]);
            }
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
            for (int o = 4; o >= 1; o >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, o));
            bool zero = !(amax > 0.0f);
            float inv = 0.0f, sc = 1.0f;
            if (!zero) {
                inv = __fdiv_rn(448.0f, amax);
                if (isinf(inv))
                    zero = true;
                else
                    sc = __fdiv_rn(amax, 448.0f);
            }
            uint32_t packed[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {  // code word h: channels 4h .. 4h+3
                uint32_t word = 0;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int i = 4 * h + 2 * q;
                    uint32_t pair;
                    if (zero) {
                        const uint32_t src_w = w[2 * h + q];
                        pair = ((src_w >> 15) & 1u) << 7 | ((src_w >> 31) & 1u) << 15;
                    } else {
                        pair = e4m3x2(__fmul_rn(f[i], inv), __fmul_rn(f[i + 1], inv));
                    }
                    word |= (pair & 0xffffu) << (16 * q);
                }
                packed[h] = word;
            }
            code[p] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            scale[p] = sc;
        }

        if (!waited) {
            wait_prior_grid();
            allow_next_grid();
            waited = true;
        }
        const int32_t *so = slot_of + t * k;
        for (int jb = 0; jb < k; jb += 32) {
            const int32_t mine = jb + lane < k ? ld_nc_s32(so + jb + lane) : 0;
            const int jn = min(32, k - jb);
            // COAL (k <= 32): a slot whose coalesced row a lower slot of the
            // token names stores nothing; that row is written once
            bool first = true;
            if (COAL) {
                const unsigned kmask = jn >= 32 ? FULL_MASK : (1u << jn) - 1u;
                first = (__match_any_sync(FULL_MASK, mine) & kmask & lanemask_lt()) == 0;
            }
            for (int q = 0; q < jn; ++q) {
                const int32_t s = __shfl_sync(FULL_MASK, mine, q);
                if (COAL && !__shfl_sync(FULL_MASK, first, q))
                    continue;
                if ((unsigned)s >= (unsigned)N) {
                    if (lane == 0)
                        report(err_word, MOE_ERRBIT_BAD_INDEX);
                    continue;
                }
                uint8_t *dq = recv_q + (int64_t)s * H;
                float *ds = recv_scales + (int64_t)s * B;
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    const int c = base + 64 * p + 2 * lane;
                    if (c < C) {
                        st_v4(dq + (int64_t)c * 8, code[p]);
                        if ((lane & 7) == 0)
                            ds[c >> 4] = scale[p];
                    }
                }
            }
        }
    }
    if (!waited) {  // a warp with no item still lets the next grid launch
        wait_prior_grid();
        allow_next_grid();
    }
    if (static_items < items) {  // the same for every CTA
        __syncthreads();         // every draw of this CTA is done
        if (threadIdx.x == 0)
            sched_finish(sched);
    }
}

template <int U, bool COAL>
static cudaError_t launch_fp8_u(int T, int H, int k, const void *x, const int32_t *slot_of,
                                uint8_t *recv_q, float *recv_scales, int rows, bool prefetch_x,
                                uint32_t *err_word, cudaStream_t stream)
{
    const int C = H / 8;
    const int groups = (C + 32 * U - 1) / (32 * U);
    const int64_t items = (int64_t)T * groups;
    const int grid = warp_item_grid((const void *)dispatch_fp8_kernel<U, COAL, true>,
                                    QUANT_THREADS, 0, items);
    const int64_t warps = (int64_t)grid * (QUANT_THREADS / 32);
    const int64_t rounds = (items + warps - 1) / warps;
    // an item: 2U blocks of 128 channels read once, codes and scales written k times
    const int64_t item_bytes = (int64_t)U * 256 * 2 + (int64_t)k * U * (256 + 8);
    if (rounds > QUANT_DYN_MIN_ROUNDS) {
        const int64_t pool_from = items * QUANT_STATIC_PCT / 100 / warps * warps;
        return launch_pdl(dispatch_fp8_kernel<U, COAL, true>, dim3(grid), dim3(QUANT_THREADS),
                          0, stream, static_cast<const uint4 *>(x), slot_of, recv_q, recv_scales,
                          k, H, groups, items, pool_from, sched_grab(item_bytes),
                          next_sched_slot(g_quant_seq), rows, prefetch_x ? 1 : 0, err_word);
    }
    const int grid_s = warp_item_grid((const void *)dispatch_fp8_kernel<U, COAL, false>,
                                      QUANT_THREADS, 0, items);
    return launch_pdl(dispatch_fp8_kernel<U, COAL, false>, dim3(grid_s), dim3(QUANT_THREADS), 0,
                      stream, static_cast<const uint4 *>(x), slot_of, recv_q, recv_scales, k, H,
                      groups, items, items, 1, 0, rows, prefetch_x ? 1 : 0, err_word);
}

// Rounds of warp items the busiest warp runs, times the blocks per item: the
// item time, in units of one block's work, of a launch with U blocks per item.
template <int U, bool COAL>
static int64_t fp8_rounds(int T, int H)
{
    const int C = H / 8;
    const int64_t items = (int64_t)T * ((C + 32 * U - 1) / (32 * U));
    auto kern = dispatch_fp8_kernel<U, COAL, false>;
    const int64_t warps = (int64_t)warp_item_grid((const void *)kern, QUANT_THREADS, 0,
                                                  items) * (QUANT_THREADS / 32);
    return (items + warps - 1) / warps * U;
}

template <bool COAL>
static cudaError_t launch_fp8(int T, int H, int k, const void *x, const int32_t *slot_of,
                              uint8_t *recv_q, float *recv_scales, int rows, uint32_t *err_word,
                              cudaStream_t stream, bool prefetch_x = false)
{
    if (T == 0)
        return cudaSuccess;
    // QUANT_U blocks per warp item keep the most bytes in flight, but a batch
    // whose items fill the GPU's warps only 1.5 times over (1024 tokens of
    // 7168 channels: 7168 items on 4864 resident warps) leaves the second
    // round half empty; items of half the size then finish sooner (3 rounds
    // of half items, against 2 of whole ones).  Only while the whole items
    // take a few rounds: over many rounds the half items' fixed costs weigh
    // more than the last round's idle warps (measured: 65536 tokens of 4096
    // channels, 203 us with whole items, 227 us with half items).
    const int64_t whole = fp8_rounds<QUANT_U, COAL>(T, H);
    if (QUANT_U == 4 && whole <= 3 * QUANT_U && fp8_rounds<2, COAL>(T, H) < whole)
        return launch_fp8_u<2, COAL>(T, H, k, x, slot_of, recv_q, recv_scales, rows, prefetch_x,
                                     err_word, stream);
    return launch_fp8_u<QUANT_U, COAL>(T, H, k, x, slot_of, recv_q, recv_scales, rows,
                                       prefetch_x, err_word, stream);
}

cudaError_t launch_dispatch_fp8(int T, int H, int k, const void *x, const int32_t *slot_of,
                                uint8_t *recv_q, float *recv_scales, uint32_t *err_word,
                                cudaStream_t stream)
{
    return launch_fp8<false>(T, H, k, x, slot_of, recv_q, recv_scales, T * k, err_word, stream);
}

cudaError_t launch_dispatch_fp8_coalesced(int T, int H, int k, const void *x,
                                          const int32_t *crow, uint8_t *recv_q,
                                          float *recv_scales, int rows, uint32_t *err_word,
                                          cudaStream_t stream)
{
    return launch_fp8<true>(T, H, k, x, crow, recv_q, recv_scales, rows, err_word, stream);
}

cudaError_t launch_layout_dispatch_quant(int T, int H, int k, int E, int R,
                                         const int32_t *topk_idx, const void *x,
                                         int32_t *expert_counts, int32_t *expert_offsets,
                                         int32_t *rank_offsets, int32_t *slot_of,
                                         int32_t *src_of, uint8_t *recv_q, float *recv_scales,
                                         void *workspace, uint32_t *err_word,
                                         cudaStream_t stream)
{
    cudaError_t e = launch_layout(T, k, E, R, topk_idx, expert_counts, expert_offsets,
                                  rank_offsets, slot_of, src_of, workspace, err_word, stream);
    if (e != cudaSuccess || T == 0)
        return e;
    // the layout kernel is the previous grid: x may be read early
    return launch_fp8<false>(T, H, k, x, slot_of, recv_q, recv_scales, T * k, err_word, stream,
                             true);
}

// The encoding of consecutive fp32 bit patterns first, first + 1, ...
// (wrapping past 2^32 - 1), one code per input.
__global__ void e4m3_bits_kernel(uint32_t first, uint32_t count, uint8_t *__restrict__ codes)
{
    // 64-bit index: a count near 2^32 must not wrap the loop
    const uint64_t stride = 2ull * gridDim.x * blockDim.x;
    for (uint64_t i = 2ull * (blockIdx.x * blockDim.x + threadIdx.x); i < count; i += stride) {
        const float a = __uint_as_float((uint32_t)(first + i));
        const float b = __uint_as_float((uint32_t)(first + i + 1));
        const uint32_t pair = e4m3x2(a, b);
        codes[i] = (uint8_t)(pair & 0xffu);
        if (i + 1 < count)
            codes[i + 1] = (uint8_t)(pair >> 8);
    }
}

cudaError_t launch_e4m3_bits(uint32_t first, uint32_t count, uint8_t *codes, cudaStream_t stream)
{
    if (count == 0)
        return cudaSuccess;
    const int threads = 256;
    int64_t blocks = ((int64_t)count / 2 + threads) / threads;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (blocks > cap)
        blocks = cap;
    e4m3_bits_kernel<<<(unsigned)blocks, threads, 0, stream>>>(first, count, codes);
    return cudaGetLastError();
}

}  // namespace moe

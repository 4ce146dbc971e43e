// C ABI entry points of libmoe_ep.so: argument checks, then the launchers.
// Nothing here allocates device memory or synchronises, except
// moe_read_error, whose job is to synchronise and read the error word.
#include <atomic>
#include <cstdint>
#include <cstring>

#include "launch.h"
#include "moe_ep.h"

namespace moe {

// SM count of the current device, cached per device (any host thread may call
// the library; every thread that fills an entry writes the same value).
int sm_count()
{
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 1;
    if (dev >= 0 && dev < 64) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0)
            return c;
    }
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        n = 1;
    if (dev >= 0 && dev < 64)
        cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

int warp_item_grid(const void *kernel, int threads, size_t smem, int64_t items)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) !=
            cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t warps_per_cta = threads / 32;
    const int64_t need = (items + warps_per_cta - 1) / warps_per_cta;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    const int64_t g = need < cap ? need : cap;
    return (int)(g < 1 ? 1 : g);
}

}  // namespace moe

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool pairs_ok(int T, int k)
{
    return T >= 0 && k >= 1 && (int64_t)T * k < ((int64_t)1 << 31);
}

}  // namespace

extern "C" {

int moe_abi_version(void) { return 2; }

const char *moe_status_string(int status)
{
    switch (status) {
    case MOE_OK:
        return "ok";
    case MOE_ERR_INVALID_ARG:
        return "invalid argument";
    case MOE_ERR_BAD_INDEX:
        return "expert id or slot index out of range";
    case MOE_ERR_CUDA:
        return "CUDA error";
    case MOE_ERR_TIMEOUT:
        return "device-side wait timed out";
    case MOE_ERR_UNSUPPORTED:
        return "unsupported configuration";
    case MOE_ERR_INTEGRITY:
        return "payload equals the sentinel, or a checksum does not match the data";
    default:
        return "unknown status";
    }
}

size_t moe_layout_workspace_bytes(int T, int k, int E)
{
    if (!pairs_ok(T, k) || E < 1 || E > MOE_MAX_EXPERTS)
        return 0;
    return moe::layout_workspace_bytes((int64_t)T * k, E);
}

moe_status moe_layout(int T, int k, int E, int R, const int32_t *topk_idx,
                      int32_t *expert_counts, int32_t *expert_offsets, int32_t *rank_offsets,
                      int32_t *slot_of, int32_t *src_of, void *workspace,
                      size_t workspace_bytes, uint32_t *err_word, cudaStream_t stream)
{
    if (!pairs_ok(T, k) || E < 1 || R < 1 || E % R != 0)
        return MOE_ERR_INVALID_ARG;
    if (E > MOE_MAX_EXPERTS)
        return MOE_ERR_UNSUPPORTED;
    if (!expert_counts || !expert_offsets || !rank_offsets)
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !slot_of || !src_of || !workspace))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(topk_idx, 4) || !aligned(expert_counts, 4) || !aligned(expert_offsets, 4) ||
        !aligned(rank_offsets, 4) || !aligned(slot_of, 4) || !aligned(src_of, 4) ||
        !aligned(workspace, 16) || !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && workspace_bytes < moe::layout_workspace_bytes((int64_t)T * k, E))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_layout(T, k, E, R, topk_idx, expert_counts, expert_offsets,
                                        rank_offsets, slot_of, src_of, workspace, err_word,
                                        stream));
}

moe_status moe_dispatch(int T, int H, int k, const void *x, const int32_t *slot_of, void *recv,
                        uint32_t *err_word, cudaStream_t stream)
{
    if (!pairs_ok(T, k) || H < 8 || H % 8 != 0)
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x || !slot_of || !recv))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(recv, 16) || !aligned(slot_of, 4) || !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_dispatch_bf16(T, H, k, x, slot_of, recv, err_word, stream));
}

moe_status moe_layout_coalesced(int T, int k, int E, int R, const int32_t *topk_idx,
                                const int32_t *slot_of, int32_t *rank_counts_c,
                                int32_t *rank_offsets_c, int32_t *crow, int32_t *src_pair_c,
                                int32_t *expand, void *workspace, size_t workspace_bytes,
                                uint32_t *err_word, cudaStream_t stream)
{
    if (!pairs_ok(T, k) || E < 1 || R < 1 || E % R != 0)
        return MOE_ERR_INVALID_ARG;
    if (E > MOE_MAX_EXPERTS)
        return MOE_ERR_UNSUPPORTED;
    if (!rank_counts_c || !rank_offsets_c)
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !slot_of || !crow || !src_pair_c || !expand || !workspace))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(topk_idx, 4) || !aligned(slot_of, 4) || !aligned(rank_counts_c, 4) ||
        !aligned(rank_offsets_c, 4) || !aligned(crow, 4) || !aligned(src_pair_c, 4) ||
        !aligned(expand, 4) || !aligned(workspace, 16) || !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && workspace_bytes < moe::layout_workspace_bytes((int64_t)T * k, R))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_layout_coalesced(T, k, E, R, topk_idx, slot_of, rank_counts_c,
                                                  rank_offsets_c, crow, src_pair_c, expand,
                                                  workspace, err_word, stream));
}

moe_status moe_dispatch_coalesced(int T, int H, int k, const void *x, const int32_t *crow,
                                  int rows, void *recv_c, uint32_t *err_word,
                                  cudaStream_t stream)
{
    if (!pairs_ok(T, k) || H < 8 || H % 8 != 0 || rows < 0)
        return MOE_ERR_INVALID_ARG;
    if (k > 32)
        return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!x || !crow || !recv_c))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(recv_c, 16) || !aligned(crow, 4) || !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_dispatch_coalesced(T, H, k, x, crow, recv_c, rows, err_word,
                                                    stream));
}

moe_status moe_dispatch_quant_coalesced(int T, int H, int k, const void *x, const int32_t *crow,
                                        int rows, uint8_t *recv_q, float *recv_scales,
                                        uint32_t *err_word, cudaStream_t stream)
{
    if (!pairs_ok(T, k) || H < 128 || H % 128 != 0 || rows < 0)
        return MOE_ERR_INVALID_ARG;
    if (k > 32)
        return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!x || !crow || !recv_q || !recv_scales))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(recv_q, 16) || !aligned(recv_scales, 16) ||
        !aligned(crow, 4) || !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_dispatch_fp8_coalesced(T, H, k, x, crow, recv_q, recv_scales,
                                                        rows, err_word, stream));
}

moe_status moe_combine_coalesced(int T, int H, int k, const void *y, const int32_t *slot_of,
                                 const float *topk_w, const int32_t *crow, int rows,
                                 void *partial, void *out, int out_dtype, uint32_t *err_word,
                                 cudaStream_t stream)
{
    if (!pairs_ok(T, k) || H < 8 || H % 8 != 0 || rows < 0)
        return MOE_ERR_INVALID_ARG;
    if (out_dtype != MOE_OUT_BF16 && out_dtype != MOE_OUT_F32)
        return MOE_ERR_INVALID_ARG;
    if (k > 32)
        return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!y || !slot_of || !topk_w || !crow || !partial || !out))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(y, 16) || !aligned(partial, 16) || !aligned(out, 16) || !aligned(slot_of, 4) ||
        !aligned(topk_w, 4) || !aligned(crow, 4) || !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_combine_coalesced(T, H, k, y, slot_of, topk_w, crow, rows,
                                                   partial, out, out_dtype == MOE_OUT_F32,
                                                   err_word, stream));
}

moe_status moe_layout_dispatch(int T, int H, int k, int E, int R, const int32_t *topk_idx,
                               const void *x, int32_t *expert_counts, int32_t *expert_offsets,
                               int32_t *rank_offsets, int32_t *slot_of, int32_t *src_of,
                               void *recv, void *workspace, size_t workspace_bytes,
                               uint32_t *err_word, cudaStream_t stream)
{
    if (!pairs_ok(T, k) || E < 1 || R < 1 || E % R != 0 || H < 8 || H % 8 != 0)
        return MOE_ERR_INVALID_ARG;
    if (E > MOE_MAX_EXPERTS)
        return MOE_ERR_UNSUPPORTED;
    if (!expert_counts || !expert_offsets || !rank_offsets)
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !x || !slot_of || !src_of || !recv || !workspace))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(topk_idx, 4) || !aligned(expert_counts, 4) || !aligned(expert_offsets, 4) ||
        !aligned(rank_offsets, 4) || !aligned(slot_of, 4) || !aligned(src_of, 4) ||
        !aligned(workspace, 16) || !aligned(x, 16) || !aligned(recv, 16) || !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && workspace_bytes < moe::layout_workspace_bytes((int64_t)T * k, E))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_layout_dispatch(T, H, k, E, R, topk_idx, x, expert_counts,
                                                 expert_offsets, rank_offsets, slot_of, src_of,
                                                 recv, workspace, err_word, stream));
}

moe_status moe_layout_dispatch_quant(int T, int H, int k, int E, int R, const int32_t *topk_idx,
                                     const void *x, int32_t *expert_counts,
                                     int32_t *expert_offsets, int32_t *rank_offsets,
                                     int32_t *slot_of, int32_t *src_of, uint8_t *recv_q,
                                     float *recv_scales, void *workspace, size_t workspace_bytes,
                                     uint32_t *err_word, cudaStream_t stream)
{
    if (!pairs_ok(T, k) || E < 1 || R < 1 || E % R != 0 || H < 128 || H % 128 != 0)
        return MOE_ERR_INVALID_ARG;
    if (E > MOE_MAX_EXPERTS)
        return MOE_ERR_UNSUPPORTED;
    if (!expert_counts || !expert_offsets || !rank_offsets)
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !x || !slot_of || !src_of || !recv_q || !recv_scales ||
                  !workspace))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(topk_idx, 4) || !aligned(expert_counts, 4) || !aligned(expert_offsets, 4) ||
        !aligned(rank_offsets, 4) || !aligned(slot_of, 4) || !aligned(src_of, 4) ||
        !aligned(workspace, 16) || !aligned(x, 16) || !aligned(recv_q, 16) ||
        !aligned(recv_scales, 16) || !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && workspace_bytes < moe::layout_workspace_bytes((int64_t)T * k, E))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_layout_dispatch_quant(T, H, k, E, R, topk_idx, x, expert_counts,
                                                       expert_offsets, rank_offsets, slot_of,
                                                       src_of, recv_q, recv_scales, workspace,
                                                       err_word, stream));
}

moe_status moe_dispatch_quant(int T, int H, int k, const void *x, const int32_t *slot_of,
                              uint8_t *recv_q, float *recv_scales, uint32_t *err_word,
                              cudaStream_t stream)
{
    if (!pairs_ok(T, k) || H < 128 || H % 128 != 0)
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x || !slot_of || !recv_q || !recv_scales))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(recv_q, 16) || !aligned(recv_scales, 16) ||
        !aligned(slot_of, 4) || !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_dispatch_fp8(T, H, k, x, slot_of, recv_q, recv_scales, err_word,
                                              stream));
}

moe_status moe_combine(int T, int H, int k, const void *y, const int32_t *slot_of,
                       const float *topk_w, void *out, int out_dtype, uint32_t *err_word,
                       cudaStream_t stream)
{
    if (!pairs_ok(T, k) || H < 8 || H % 8 != 0)
        return MOE_ERR_INVALID_ARG;
    if (out_dtype != MOE_OUT_BF16 && out_dtype != MOE_OUT_F32)
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!y || !slot_of || !topk_w || !out))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(y, 16) || !aligned(out, 16) || !aligned(slot_of, 4) || !aligned(topk_w, 4) ||
        !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_combine(T, H, k, y, slot_of, topk_w, out,
                                         out_dtype == MOE_OUT_F32, err_word, stream));
}

moe_status moe_combine_backward(int T, int H, int k, const void *dout, const void *y,
                                const int32_t *slot_of, const float *topk_w, void *dy, float *dw,
                                uint32_t *err_word, cudaStream_t stream)
{
    if (!pairs_ok(T, k) || H < 8 || H % 8 != 0)
        return MOE_ERR_INVALID_ARG;
    if (k > 32)
        return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!dout || !slot_of || !topk_w || !dy || (dw && !y)))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(dout, 16) || !aligned(y, 16) || !aligned(dy, 16) || !aligned(slot_of, 4) ||
        !aligned(topk_w, 4) || !aligned(dw, 4) || !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_combine_backward(T, H, k, dout, y, slot_of, topk_w, dy, dw,
                                                  err_word, stream));
}

moe_status moe_dispatch_backward(int T, int H, int k, const void *drecv, const int32_t *slot_of,
                                 void *dx, int out_dtype, uint32_t *err_word, cudaStream_t stream)
{
    if (!pairs_ok(T, k) || H < 8 || H % 8 != 0)
        return MOE_ERR_INVALID_ARG;
    if (out_dtype != MOE_OUT_BF16 && out_dtype != MOE_OUT_F32)
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!drecv || !slot_of || !dx))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(drecv, 16) || !aligned(dx, 16) || !aligned(slot_of, 4) || !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    // the combine pipeline with unit weights
    return from_cuda(moe::launch_combine(T, H, k, drecv, slot_of, nullptr, dx,
                                         out_dtype == MOE_OUT_F32, err_word, stream));
}

size_t moe_sync_words(int T, int H, int k, int mode, int block_bytes)
{
    if (!pairs_ok(T, k) || H < 8 || H % 8 != 0)
        return 0;
    return moe::sync_words(T, H, k, mode, block_bytes);
}

moe_status moe_dispatch_combine_flagged(int T, int H, int k, const void *x, const int32_t *slot_of,
                                        const float *topk_w, void *recv, void *y, void *out,
                                        int out_dtype, int mode, int block_bytes, uint32_t *words,
                                        uint32_t epoch, uint64_t spin_limit_ns,
                                        int64_t fault_skip_pair, uint32_t *err_word,
                                        cudaStream_t stream)
{
    if (!pairs_ok(T, k) || H < 8 || H % 8 != 0 || spin_limit_ns == 0)
        return MOE_ERR_INVALID_ARG;
    if (mode < MOE_SYNC_WORD || mode > MOE_SYNC_BARRIER ||
        !moe::sync_granularity_ok(mode, H, block_bytes))
        return MOE_ERR_INVALID_ARG;
    if ((mode == MOE_SYNC_WORD || mode == MOE_SYNC_BATCH) && epoch == 0)
        return MOE_ERR_INVALID_ARG;
    if (k > 32)
        return MOE_ERR_UNSUPPORTED;
    if (out_dtype != MOE_OUT_BF16 && out_dtype != MOE_OUT_F32)
        return MOE_ERR_INVALID_ARG;
    const bool need_words = moe::sync_words(T, H, k, mode, block_bytes) > 0;
    if (T > 0 && (!x || !slot_of || !topk_w || !recv || !y || !out || (need_words && !words)))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(recv, 16) || !aligned(y, 16) || !aligned(out, 16) ||
        !aligned(slot_of, 4) || !aligned(topk_w, 4) || !aligned(words, 8) ||
        !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_dispatch_combine_flagged(
        T, H, k, x, slot_of, topk_w, recv, y, out, out_dtype == MOE_OUT_F32, mode, block_bytes,
        words, epoch, spin_limit_ns, fault_skip_pair, err_word, stream));
}

moe_status moe_ep_reorder(int W, int El, int H, const int32_t *recv_counts, int rows,
                          const void *src, void *dst, int direction,
                          int32_t *local_expert_offsets, uint32_t *err_word, cudaStream_t stream)
{
    if (W < 1 || El < 1 || H < 8 || H % 8 != 0 || rows < 0)
        return MOE_ERR_INVALID_ARG;
    if (direction != MOE_EP_TO_EXPERT && direction != MOE_EP_TO_SOURCE)
        return MOE_ERR_INVALID_ARG;
    if ((int64_t)W * El > MOE_MAX_EXPERTS)
        return MOE_ERR_UNSUPPORTED;
    if (!recv_counts || (rows > 0 && (!src || !dst)))
        return MOE_ERR_INVALID_ARG;
    if (rows > 0 && src == dst)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(src, 16) || !aligned(dst, 16) || !aligned(recv_counts, 4) ||
        !aligned(local_expert_offsets, 4) || !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_ep_reorder(W, El, 2 * (int64_t)H, recv_counts, rows, src, dst,
                                            direction == MOE_EP_TO_SOURCE, local_expert_offsets,
                                            err_word, stream));
}

moe_status moe_ep_reorder_rows(int W, int El, int row_bytes, const int32_t *recv_counts,
                               int rows, const void *src, void *dst, int direction,
                               int32_t *local_expert_offsets, uint32_t *err_word,
                               cudaStream_t stream)
{
    if (W < 1 || El < 1 || row_bytes < 4 || row_bytes % 4 != 0 || rows < 0)
        return MOE_ERR_INVALID_ARG;
    if (direction != MOE_EP_TO_EXPERT && direction != MOE_EP_TO_SOURCE)
        return MOE_ERR_INVALID_ARG;
    if ((int64_t)W * El > MOE_MAX_EXPERTS)
        return MOE_ERR_UNSUPPORTED;
    if (!recv_counts || (rows > 0 && (!src || !dst)))
        return MOE_ERR_INVALID_ARG;
    if (rows > 0 && src == dst)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(src, 4) || !aligned(dst, 4) || !aligned(recv_counts, 4) ||
        !aligned(local_expert_offsets, 4) || !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_ep_reorder(W, El, row_bytes, recv_counts, rows, src, dst,
                                            direction == MOE_EP_TO_SOURCE, local_expert_offsets,
                                            err_word, stream));
}

moe_status moe_e4m3_encode_bits(uint32_t first, uint32_t count, uint8_t *codes,
                                cudaStream_t stream)
{
    if (count > 0 && !codes)
        return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_e4m3_bits(first, count, codes, stream));
}

moe_status moe_read_error(uint32_t *err_word, int clear, cudaStream_t stream, uint32_t *bits_out)
{
    if (!err_word || !aligned(err_word, 4))
        return MOE_ERR_INVALID_ARG;
    uint32_t bits = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaMemcpy(&bits, err_word, sizeof bits, cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (clear && bits != 0) {
        if (cudaMemsetAsync(err_word, 0, sizeof bits, stream) != cudaSuccess ||
            cudaStreamSynchronize(stream) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    if (bits_out)
        *bits_out = bits;
    if (bits & MOE_ERRBIT_LAUNCH)
        return MOE_ERR_CUDA;
    if (bits & MOE_ERRBIT_TIMEOUT)
        return MOE_ERR_TIMEOUT;
    if (bits & MOE_ERRBIT_BAD_INDEX)
        return MOE_ERR_BAD_INDEX;
    if (bits & (MOE_ERRBIT_SENTINEL | MOE_ERRBIT_CHECKSUM))
        return MOE_ERR_INTEGRITY;
    return MOE_OK;
}

}  // extern "C"

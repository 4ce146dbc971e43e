// moe_layout_noalloc: the layout entry point for callers that cannot allocate.
//
// Some callers cannot allocate device memory when they call the layout: code
// handed fixed buffers by a host framework that owns all allocation, or
// runtimes that forbid cudaMalloc once they have started.  They cannot supply
// moe_layout's workspace.  This variant runs the same layout kernel, with
// its per-tile count table in a fixed array compiled into the library
// instead of a caller workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds MOE_NOALLOC_SCRATCH_BYTES of it until the process exits.  Host
// code cannot use the array's name as a device address, so the first call on
// each device (made with that device current) looks the address up with
// cudaGetSymbolAddress and caches it; make that first call before any stream
// capture.  All calls on a device share the one array: calls whose kernels
// overlap on the GPU (different streams, no ordering between them) race on it.
// Only its first 8 bytes (the layout kernel's grid barrier) must start at
// zero, and each call clears them on the stream before launching; the tile
// table is rewritten before it is read.  The entry point allocates nothing,
// frees nothing and calls no allocating library routine.
#include <mutex>

#include "launch.h"
#include "moe_ep.h"

namespace {

static __device__ __align__(256) int32_t g_layout_scratch[MOE_NOALLOC_SCRATCH_BYTES / sizeof(int32_t)];

constexpr int MAX_DEVICES = 64;
std::mutex g_mutex;
void *g_scratch_addr[MAX_DEVICES] = {nullptr};

// Device address of the scratch array on the current device, or nullptr.
void *scratch_on_current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
        return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_layout_scratch) != cudaSuccess)
            return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" MOE_API moe_status moe_layout_noalloc(int T, int k, int E, int R,
                                                 const int32_t *topk_idx,
                                                 int32_t *expert_counts,
                                                 int32_t *expert_offsets,
                                                 int32_t *rank_offsets, int32_t *slot_of,
                                                 int32_t *src_of, uint32_t *err_word,
                                                 cudaStream_t stream)
{
    if (T < 0 || k < 1 || (int64_t)T * k >= ((int64_t)1 << 31) || E < 1 || R < 1 ||
        E % R != 0)
        return MOE_ERR_INVALID_ARG;
    if (E > MOE_MAX_EXPERTS)
        return MOE_ERR_UNSUPPORTED;
    if (!expert_counts || !expert_offsets || !rank_offsets)
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !slot_of || !src_of))
        return MOE_ERR_INVALID_ARG;
    if (!aligned4(topk_idx) || !aligned4(expert_counts) || !aligned4(expert_offsets) ||
        !aligned4(rank_offsets) || !aligned4(slot_of) || !aligned4(src_of) ||
        !aligned4(err_word))
        return MOE_ERR_INVALID_ARG;
    if (moe::layout_workspace_bytes((int64_t)T * k, E) > MOE_NOALLOC_SCRATCH_BYTES)
        return MOE_ERR_UNSUPPORTED;
    void *scratch = scratch_on_current_device();
    if (scratch == nullptr)
        return MOE_ERR_CUDA;
    // The layout kernel's grid barrier (the array's first 8 bytes) must start
    // at zero; clear it on the stream so no earlier failure can leave it set.
    cudaError_t e = cudaMemsetAsync(scratch, 0, 8, stream);
    if (e == cudaSuccess)
        e = moe::launch_layout(T, k, E, R, topk_idx, expert_counts, expert_offsets, rank_offsets,
                               slot_of, src_of, scratch, err_word, stream);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

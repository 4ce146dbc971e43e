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
// cudaGetSymbolAddress and caches it together with the identity of the CUDA
// context it belongs to; a later call that finds another context current on
// that device (after cudaDeviceReset, say) looks it up again.  Make the first
// call before any stream capture.  All calls on a device share the one array:
// calls whose kernels overlap on the GPU (different streams, no ordering
// between them) race on it.  Only its first 8 bytes (the layout kernel's grid
// barrier) must start at zero, and they are cleared on the stream right before
// a launch in the grid-barrier form, the only form that reads them (one tile,
// or one cluster of up to 16, uses no part of the array).  The tile table is
// rewritten before it is read.  The entry point allocates nothing, frees
// nothing and calls no allocating library routine.
#include <cuda.h>
#include <mutex>

#include "launch.h"
#include "moe_ep.h"

namespace {

static __device__ __align__(256) int32_t g_layout_scratch[MOE_NOALLOC_SCRATCH_BYTES / sizeof(int32_t)];

constexpr int MAX_DEVICES = 64;
std::mutex g_mutex;
void *g_scratch_addr[MAX_DEVICES] = {nullptr};
unsigned long long g_scratch_ctx[MAX_DEVICES] = {0};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
std::once_flag g_entry_once;

// Process-unique id of the CUDA context current on this thread (the driver's
// context id, never reused within a process), or 0 when unavailable.
unsigned long long current_context_id()
{
    std::call_once(g_entry_once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f);
        (void)cudaGetLastError();
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr ||
        g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        g_ctx_get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array in the current device's current
// context, or nullptr.
void *scratch_on_current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
        return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    const unsigned long long ctx = current_context_id();
    if (g_scratch_addr[dev] != nullptr && ctx != 0 && ctx == g_scratch_ctx[dev])
        return g_scratch_addr[dev];
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_layout_scratch) != cudaSuccess)
        return nullptr;
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = current_context_id();  // the lookup made a context current if none was
    return p;
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
    // clear_barrier: the grid-barrier form, if it runs, finds its barrier at
    // zero whatever an earlier call left there
    const cudaError_t e = moe::launch_layout(T, k, E, R, topk_idx, expert_counts, expert_offsets,
                                             rank_offsets, slot_of, src_of, scratch, err_word,
                                             stream, true);
    // the same status mapping as every other entry point
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

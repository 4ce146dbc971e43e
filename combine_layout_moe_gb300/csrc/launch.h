// Internal launchers behind the C ABI (abi.cu).  Arguments are already
// validated by the caller; each returns the CUDA status of its launches.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

size_t layout_workspace_bytes(int64_t N, int E);

// clear_barrier: zero the workspace's grid-barrier head on the stream before
// a launch in the grid-barrier form (the only form that reads it).
cudaError_t launch_layout(int T, int k, int E, int R, const int32_t *topk_idx,
                          int32_t *expert_counts, int32_t *expert_offsets,
                          int32_t *rank_offsets, int32_t *slot_of, int32_t *src_of,
                          void *workspace, uint32_t *err_word, cudaStream_t stream,
                          bool clear_barrier = false);

// Records the layout form (MOE_LAYOUT_FORM_*) this host thread launched last.
void note_layout_form(int form);

cudaError_t launch_layout_coalesced(int T, int k, int E, int R, const int32_t *topk_idx,
                                    const int32_t *slot_of, int32_t *rank_counts_c,
                                    int32_t *rank_offsets_c, int32_t *crow, int32_t *src_pair_c,
                                    int32_t *expand, void *workspace, uint32_t *err_word,
                                    cudaStream_t stream);

cudaError_t launch_dispatch_coalesced(int T, int H, int k, const void *x, const int32_t *crow,
                                      void *recv_c, int rows, uint32_t *err_word,
                                      cudaStream_t stream);

cudaError_t launch_dispatch_bf16(int T, int H, int k, const void *x, const int32_t *slot_of,
                                 void *recv, uint32_t *err_word, cudaStream_t stream);

// moe_layout followed by moe_dispatch (bf16) whose first loads of x overlap
// the layout.
cudaError_t launch_layout_dispatch(int T, int H, int k, int E, int R, const int32_t *topk_idx,
                                   const void *x, int32_t *expert_counts,
                                   int32_t *expert_offsets, int32_t *rank_offsets,
                                   int32_t *slot_of, int32_t *src_of, void *recv,
                                   void *workspace, uint32_t *err_word, cudaStream_t stream);

// The single-kernel layout + dispatch for small batches (layout_dispatch.cu):
// whether a batch fits it, and its launch.
bool layout_dispatch_fused_fits(int T, int H, int k, int E);
cudaError_t launch_layout_dispatch_fused(int T, int H, int k, int E, int R,
                                         const int32_t *topk_idx, const void *x,
                                         int32_t *expert_counts, int32_t *expert_offsets,
                                         int32_t *rank_offsets, int32_t *slot_of,
                                         int32_t *src_of, void *recv, uint32_t *err_word,
                                         cudaStream_t stream);

// moe_layout followed by moe_dispatch_quant, whose first items' loads and
// quantisation of x overlap the layout.
cudaError_t launch_layout_dispatch_quant(int T, int H, int k, int E, int R,
                                         const int32_t *topk_idx, const void *x,
                                         int32_t *expert_counts, int32_t *expert_offsets,
                                         int32_t *rank_offsets, int32_t *slot_of,
                                         int32_t *src_of, uint8_t *recv_q, float *recv_scales,
                                         void *workspace, uint32_t *err_word,
                                         cudaStream_t stream);

// The quantised dispatch's channel encoding on consecutive fp32 bit patterns.
cudaError_t launch_e4m3_bits(uint32_t first, uint32_t count, uint8_t *codes, cudaStream_t stream);

cudaError_t launch_dispatch_fp8(int T, int H, int k, const void *x, const int32_t *slot_of,
                                uint8_t *recv_q, float *recv_scales, uint32_t *err_word,
                                cudaStream_t stream);

cudaError_t launch_dispatch_fp8_coalesced(int T, int H, int k, const void *x,
                                          const int32_t *crow, uint8_t *recv_q,
                                          float *recv_scales, int rows, uint32_t *err_word,
                                          cudaStream_t stream);

cudaError_t launch_combine(int T, int H, int k, const void *y, const int32_t *slot_of,
                           const float *topk_w, void *out, bool out_f32,
                           uint32_t *err_word, cudaStream_t stream);

cudaError_t launch_combine_coalesced(int T, int H, int k, const void *y, const int32_t *slot_of,
                                     const float *topk_w, const int32_t *crow, int rows,
                                     void *partial, void *out, bool out_f32, uint32_t *err_word,
                                     cudaStream_t stream);

cudaError_t launch_combine_backward(int T, int H, int k, const void *dout, const void *y,
                                    const int32_t *slot_of, const float *topk_w, void *dy,
                                    float *dw, uint32_t *err_word, cudaStream_t stream);

cudaError_t launch_ep_reorder(int W, int El, int64_t row_bytes, const int32_t *recv_counts,
                              int64_t rows, const void *src, void *dst, bool to_source,
                              int32_t *local_expert_offsets, uint32_t *err_word,
                              cudaStream_t stream);

bool sync_granularity_ok(int mode, int H, int G);

size_t sync_words(int T, int H, int k, int mode, int G);

cudaError_t launch_dispatch_combine_flagged(int T, int H, int k, const void *x,
                                            const int32_t *slot_of, const float *topk_w,
                                            void *recv, void *y, void *out, bool out_f32,
                                            int mode, int G, uint32_t *words, uint32_t epoch,
                                            uint64_t spin_limit_ns, int64_t skip_pair,
                                            uint32_t *err_word, cudaStream_t stream);

// Launches `kernel` on `stream` with programmatic stream serialisation, so it
// may become resident while the previous kernel in the stream is still running
// (the kernel itself waits for that grid before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Number of SMs of the current device (cached per device).
int sm_count();

// Grid size for a warp-per-item kernel: enough CTAs for `items` warp items,
// capped at the number of co-resident CTAs on the whole GPU.
int warp_item_grid(const void *kernel, int threads, size_t smem, int64_t items);

}  // namespace moe

/*
 * moe_ep.h -- C ABI of the GB300 MoE expert-parallel layout / dispatch / combine
 * library (libmoe_ep.so, sm_103a kernels).
 *
 * Problem statement (shared by the pages): T tokens with hidden size H, each
 * routed by a top-k router to k of E experts; the experts are spread over R
 * expert-parallel ranks in contiguous blocks of E/R (expert e lives on rank
 * e / (E/R)).  On one GPU the ranks are contiguous segments of one HBM buffer.
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or keeps a pointer past the call.  The output
 *     arrays of a call may not overlap one another or its inputs (the kernels
 *     are compiled on that promise).
 *   - Every call is asynchronous and ordered on `stream`; none copies data back
 *     to the host.  MOE_OK means the work was enqueued.
 *   - Arguments are checked before anything is launched; a bad argument returns
 *     MOE_ERR_INVALID_ARG and launches nothing.  Payload pointers (x, recv, y,
 *     out, recv_q, recv_scales) must be 16-byte aligned; index/weight arrays
 *     4-byte aligned.
 *   - Problems found on the device (an expert id outside [0, E), a slot outside
 *     [0, T*k)) skip the offending element and OR a bit into `*err_word` (a
 *     device uint32 the caller zero-fills once; NULL disables reporting).
 *     moe_read_error() synchronises the stream and reports it.  Outputs are
 *     undefined after any error.
 *   - A failed CUDA launch returns MOE_ERR_CUDA.
 *   - The dispatch kernels share large launches out at run time: each CTA (or
 *     warp) takes a fixed part of the work and draws the rest from a counter
 *     of the launch.  The counters live in a table of 1024 slots per kernel
 *     family in the library's own device memory (static, allocated when the
 *     library loads); a launch takes the next slot and its last CTA clears
 *     it.  Launches of one family may run concurrently, and a captured CUDA
 *     graph may be replayed, as long as fewer than 1024 of them execute at
 *     the same moment on one device.
 */
#ifndef MOE_EP_H
#define MOE_EP_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1, /* rejected on the host, nothing launched            */
    MOE_ERR_BAD_INDEX = 2,   /* device saw an expert id or slot out of range      */
    MOE_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed              */
    MOE_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up                */
    MOE_ERR_UNSUPPORTED = 5, /* well-formed request outside this build's limits   */
    MOE_ERR_INTEGRITY = 6    /* payload equal to the sentinel, or a checksum that */
                             /* does not match the data                           */
} moe_status;

typedef enum moe_out_dtype { MOE_OUT_BF16 = 0, MOE_OUT_F32 = 1 } moe_out_dtype;

/* bits OR-ed into *err_word by the kernels */
#define MOE_ERRBIT_BAD_INDEX 0x1u
#define MOE_ERRBIT_TIMEOUT 0x2u
#define MOE_ERRBIT_SENTINEL 0x4u
#define MOE_ERRBIT_CHECKSUM 0x8u
#define MOE_ERRBIT_LAUNCH 0x10u /* a kernel found itself launched in a shape it   */
                                /* cannot serve (a cluster of the wrong size);    */
                                /* it wrote no outputs                            */

/* how moe_dispatch_combine_flagged's readers learn that data has arrived */
typedef enum moe_sync_mode {
    MOE_SYNC_WORD = 0,     /* a 32-bit word per (row, block), set after a fence     */
    MOE_SYNC_SENTINEL = 1, /* the reader polls the data itself (sentinel-filled)   */
    MOE_SYNC_BATCH = 2,    /* a 64-bit (epoch, checksum) word per (row, batch)      */
    MOE_SYNC_BARRIER = 3   /* a grid barrier between the phases (stop-and-wait)     */
} moe_sync_mode;

/* largest expert count the layout kernels hold in shared memory */
#define MOE_MAX_EXPERTS 1024

/* ABI revision; bumped on any signature change. */
MOE_API int moe_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
MOE_API const char *moe_status_string(int status);

/*
 * Bytes of device workspace moe_layout needs for (T, k, E); 0 for bad sizes.
 * The first 256 bytes hold the grid barrier of the layout kernel (one
 * cooperative launch): zero-fill the workspace once before its first use.
 * Every successful call leaves the barrier's arrival count at zero again, so
 * it never needs zeroing again (after MOE_ERR_TIMEOUT, zero it again).  The
 * rest holds per-tile expert counts, scratch between calls.  One workspace
 * serves any (T, k, E) whose size fits.
 */
MOE_API size_t moe_layout_workspace_bytes(int T, int k, int E);

/*
 * moe_layout -- count, exclusive scan and stable slot map.
 *
 * UBEP, section 2.3 and Figure 2 (dispatch Phase 5: per-expert token counts give
 * offsets, tokens are reordered contiguously per expert) and section 4 (receive
 * region partitioned by source and expert); StrataCL, Appendix D (per-expert
 * counts, prefix-sum offsets and token-local offsets are the placement metadata
 * that dispatch and combine reuse).
 *
 *   topk_idx        [T, k] int32, row-major; expert id of token t's j-th choice
 *   expert_counts   [E]    out: number of (t, j) pairs routed to expert e
 *   expert_offsets  [E+1]  out: exclusive prefix sum of expert_counts; [E] = T*k
 *   rank_offsets    [R+1]  out: expert_offsets[r * E/R], the start of rank r's
 *                          segment of the receive buffer; [R] = T*k
 *   slot_of         [T, k] out: receive-buffer row of (t, j)
 *   src_of          [T*k]  out: inverse map, src_of[slot_of[t,j]] = t*k + j
 *   workspace       moe_layout_workspace_bytes(T, k, E) bytes of device scratch,
 *                   zero-filled before its first use (see above)
 *
 * Slot order is (rank, expert, token, j): rank-segmented, expert-contiguous,
 * and stable in (t, j), with no padding.  The result is deterministic and
 * does not depend on the launch configuration.  1 <= k, 1 <= E <=
 * MOE_MAX_EXPERTS, E % R == 0, 0 <= T, T*k < 2^31.  T == 0 writes zero counts
 * and offsets.
 */
MOE_API moe_status moe_layout(int T, int k, int E, int R, const int32_t *topk_idx,
                      int32_t *expert_counts, int32_t *expert_offsets,
                      int32_t *rank_offsets, int32_t *slot_of, int32_t *src_of,
                      void *workspace, size_t workspace_bytes, uint32_t *err_word,
                      cudaStream_t stream);

/*
 * moe_dispatch -- bf16 token rows scattered into the packed receive buffer.
 *
 * UBEP, section 2.3 (Phase 2: each token is sent to every expert it chose) and
 * section 4 (senders write directly into the partitioned receive region);
 * RailWave, section 3.2 (payload packed without padding).
 *
 *   x        [T, H]   bf16 hidden states, row-major
 *   slot_of  [T, k]   from moe_layout
 *   recv     [T*k, H] out: recv[slot_of[t, j], :] = x[t, :]  (bit copy)
 *
 * H % 8 == 0 (16-byte rows).
 */
MOE_API moe_status moe_dispatch(int T, int H, int k, const void *x, const int32_t *slot_of,
                        void *recv, uint32_t *err_word, cudaStream_t stream);

/*
 * moe_layout_dispatch -- moe_layout followed by moe_dispatch (bf16), with the
 * dispatch's loads of x overlapping the layout.
 *
 * UBEP, section 3.2 (kernel decomposition: token sending overlaps the count
 * and scan instead of waiting behind them).  Same arguments, outputs, rules
 * and errors as moe_layout and moe_dispatch called in turn on `stream`.
 * Small batches (T*k <= 16384, each SM's share of x within shared memory,
 * k <= 32) run as one kernel: every CTA loads its share of x, counts the
 * whole batch's ids itself while those loads land, and stores its rows to
 * their slots -- no exchange between CTAs and no second launch; the workspace
 * is then not touched.  Larger batches run the layout kernel, then a dispatch
 * kernel that reads x while the layout still runs.  Either way x must be
 * complete before this call, as for moe_dispatch.
 */
MOE_API moe_status moe_layout_dispatch(int T, int H, int k, int E, int R,
                               const int32_t *topk_idx, const void *x,
                               int32_t *expert_counts, int32_t *expert_offsets,
                               int32_t *rank_offsets, int32_t *slot_of, int32_t *src_of,
                               void *recv, void *workspace, size_t workspace_bytes,
                               uint32_t *err_word, cudaStream_t stream);

/*
 * moe_dispatch_quant -- dispatch with fused FP8-E4M3 block quantisation.
 *
 * UBEP, Table 3 (the DeepSeek-R1 / V3.2 deployments run W8A8; the pages give no
 * further recipe).  Reading implemented: per token row, blocks of 128 channels;
 * amax = max |x|; scale = amax / 448 and inv = 448 / amax, each rounded to
 * nearest in fp32; code = e4m3(x * inv) rounded to nearest-even with saturation
 * to +-448.  A block with amax == 0, or whose 448 / amax overflows fp32, stores
 * scale 1 and signed zero codes.  Every one of a token's k slots receives the
 * same codes and scales.
 *
 *   x            [T, H]      bf16
 *   recv_q       [T*k, H]    out: E4M3 codes (one byte each)
 *   recv_scales  [T*k, H/128] out: fp32 dequantisation scales, row-major
 *
 * H % 128 == 0.
 */
MOE_API moe_status moe_dispatch_quant(int T, int H, int k, const void *x, const int32_t *slot_of,
                              uint8_t *recv_q, float *recv_scales, uint32_t *err_word,
                              cudaStream_t stream);

/*
 * moe_layout_dispatch_quant -- moe_layout followed by moe_dispatch_quant, with
 * the dispatch's first loads and quantisation of x overlapping the layout.
 *
 * UBEP, section 3.2 (token sending overlaps the count and scan) and Table 3
 * (W8A8).  Same arguments, outputs, rules and errors as moe_layout and
 * moe_dispatch_quant called in turn on `stream`.  The FP8 dispatch kernel
 * launches while the layout kernel runs, loads and quantises its first token
 * blocks, and waits for the layout only before reading the slot map; x must
 * be complete before this call, as for moe_dispatch_quant.
 */
MOE_API moe_status moe_layout_dispatch_quant(int T, int H, int k, int E, int R,
                                     const int32_t *topk_idx, const void *x,
                                     int32_t *expert_counts, int32_t *expert_offsets,
                                     int32_t *rank_offsets, int32_t *slot_of, int32_t *src_of,
                                     uint8_t *recv_q, float *recv_scales, void *workspace,
                                     size_t workspace_bytes, uint32_t *err_word,
                                     cudaStream_t stream);

/*
 * moe_combine -- gather expert outputs back to token order, router-weighted.
 *
 * HyperParallel-MoE, section 2.2 (expert outputs are weighted by the routing
 * scores and combined) and section 4.1 (Combine accumulates the top-k
 * contributions according to routing scores); RailWave, section 3 (combine
 * uses the saved dispatch metadata to return rows to their token positions).
 *
 *   y        [T*k, H] bf16 expert outputs in receive order
 *   slot_of  [T, k]   from moe_layout
 *   topk_w   [T, k]   fp32 router weights (used as given, not renormalised)
 *   out      [T, H]   out: bf16 (out_dtype MOE_OUT_BF16) or fp32 (MOE_OUT_F32)
 *
 * out[t, h] = round(sum_j w[t, j] * y[slot_of[t, j], h]) with fp32 accumulation:
 * acc = +0, then acc = fma(w[t, j], y, acc) for j = 0 .. k-1, then one rounding
 * to the output type (nearest-even).  H % 8 == 0.
 */
MOE_API moe_status moe_combine(int T, int H, int k, const void *y, const int32_t *slot_of,
                       const float *topk_w, void *out, int out_dtype, uint32_t *err_word,
                       cudaStream_t stream);

/*
 * moe_combine_backward -- gradient of moe_combine (the backward Dispatch).
 *
 * HyperParallel-MoE, section 2.2 / Figure 2(b): the backward Dispatch is the
 * gradient of the forward Combine.  With out[t] = sum_j w[t,j] * y[slot_of[t,j]]:
 *
 *   dout     [T, H]    bf16 gradient of out
 *   y        [T*k, H]  bf16 forward expert outputs (receive order); may be NULL
 *                      when dw is NULL
 *   dy       [T*k, H]  out: bf16, dy[slot_of[t,j]] = w[t,j] * dout[t] (one fp32
 *                      multiply, rounded once to bf16)
 *   dw       [T, k]    out (may be NULL): fp32 <y[slot_of[t,j]], dout[t]>; the
 *                      bf16 products are exact in fp32, the sum is accumulated
 *                      in fp32 in a fixed order (deterministic; within
 *                      (H-1) * 2^-24 * sum|y * dout| of the exact value)
 *
 * 1 <= k <= 32; H % 8 == 0.  For 5 <= k <= 8 the call first zero-fills dw on
 * the stream (an asynchronous memset, then the kernel adds at most two partial
 * sums per element, whose order cannot change the result).
 */
MOE_API moe_status moe_combine_backward(int T, int H, int k, const void *dout, const void *y,
                                const int32_t *slot_of, const float *topk_w, void *dy,
                                float *dw, uint32_t *err_word, cudaStream_t stream);

/*
 * moe_dispatch_backward -- gradient of moe_dispatch (the backward Combine).
 *
 * HyperParallel-MoE, section 2.2 / Figure 2(b): the backward Combine returns
 * the input-activation gradient.  dx[t] = sum_j drecv[slot_of[t,j]]: fp32
 * accumulation from +0 in slot order, rounded once to bf16 (MOE_OUT_BF16) or
 * kept fp32 (MOE_OUT_F32) -- moe_combine with unit weights.
 *
 *   drecv    [T*k, H]  bf16 gradient of recv
 *   dx       [T, H]    out
 */
MOE_API moe_status moe_dispatch_backward(int T, int H, int k, const void *drecv,
                                 const int32_t *slot_of, void *dx, int out_dtype,
                                 uint32_t *err_word, cudaStream_t stream);

/*
 * moe_layout_coalesced -- rank-coalesced row map: one receive row per token
 * and distinct destination rank.
 *
 * RailWave, section 3.1 (token coalescing: a token crosses to a rank once,
 * however many of its experts live there); UBEP, section 2.3 (a token goes to
 * several experts).  Pair (t, j) owns (t, rank(e_tj)) when no earlier slot
 * j' < j of token t chose an expert on the same rank (rank(e) = e / (E / R)).
 * Owners take rows rank by rank, in token order inside a rank, no padding.
 *
 *   topk_idx       [T, k]  int32 expert ids in [0, E)
 *   slot_of        [T, k]  int32 plain slot map from moe_layout (same topk_idx)
 *   rank_counts_c  [R]     out: coalesced rows per destination rank
 *   rank_offsets_c [R+1]   out: exclusive scan of rank_counts_c; [R] = Nc
 *   crow           [T, k]  out: coalesced row of (t, rank(e_tj)), for owners and
 *                          the other slots alike
 *   src_pair_c     [T*k]   out: owner pair t*k+j of row c, for c < Nc (the
 *                          rest is left unwritten)
 *   expand         [T*k]   out: expand[slot_of[t,j]] = crow[t,j], the coalesced
 *                          row that holds the input of each plain slot
 *   workspace      moe_layout_workspace_bytes(T, k, R) bytes, zero-filled once
 *                  (the same rules as moe_layout's; the two may not share one
 *                  workspace concurrently)
 *
 * Ids outside [0, E) set MOE_ERRBIT_BAD_INDEX, get crow -1 and no row.
 * 1 <= R <= E <= MOE_MAX_EXPERTS, E % R == 0.  One launch when k divides 32
 * (every 32-pair warp step then holds whole tokens, so the other slots and
 * expand are resolved in the same pass); otherwise a second launch does that.
 */
MOE_API moe_status moe_layout_coalesced(int T, int k, int E, int R, const int32_t *topk_idx,
                                const int32_t *slot_of, int32_t *rank_counts_c,
                                int32_t *rank_offsets_c, int32_t *crow, int32_t *src_pair_c,
                                int32_t *expand, void *workspace, size_t workspace_bytes,
                                uint32_t *err_word, cudaStream_t stream);

/*
 * moe_dispatch_coalesced -- copy each token's row once per destination rank.
 *
 * RailWave, section 3.1 (coalesced dispatch sends one copy of a token per
 * destination rank).  recv_c[crow[t, j]] = x[t]; each row is written once
 * (by the lowest slot of the token that names it).
 *
 *   x       [T, H]     bf16 token rows (16-byte aligned)
 *   crow    [T, k]     from moe_layout_coalesced
 *   rows    capacity of recv_c in rows (rows named by crow must be below it;
 *           Nc <= T * min(k, R))
 *   recv_c  [rows, H]  out: bf16 (16-byte aligned)
 *
 * 1 <= k <= 32 (larger k: MOE_ERR_UNSUPPORTED); H % 8 == 0.  Row indices
 * outside [0, rows) set MOE_ERRBIT_BAD_INDEX and are skipped.
 */
MOE_API moe_status moe_dispatch_coalesced(int T, int H, int k, const void *x,
                                  const int32_t *crow, int rows, void *recv_c,
                                  uint32_t *err_word, cudaStream_t stream);

/*
 * moe_dispatch_quant_coalesced -- moe_dispatch_quant into the rank-coalesced
 * rows: each token's E4M3 codes and fp32 scales (the moe_dispatch_quant
 * reading: 1x128 blocks, scale = amax / 448) are written once per distinct
 * destination rank.
 *
 * RailWave, section 3.1 (token coalescing); UBEP, Table 3 (W8A8).
 *   crow        [T, k]         from moe_layout_coalesced
 *   rows        capacity of the outputs in rows (as for moe_dispatch_coalesced)
 *   recv_q      [rows, H]      out: E4M3 codes (16-byte aligned)
 *   recv_scales [rows, H/128]  out: fp32 scales (16-byte aligned)
 * 1 <= k <= 32 (larger k: MOE_ERR_UNSUPPORTED); H % 128 == 0.  Row indices
 * outside [0, rows) set MOE_ERRBIT_BAD_INDEX and are skipped.
 */
MOE_API moe_status moe_dispatch_quant_coalesced(int T, int H, int k, const void *x,
                                        const int32_t *crow, int rows, uint8_t *recv_q,
                                        float *recv_scales, uint32_t *err_word,
                                        cudaStream_t stream);

/*
 * moe_combine_coalesced -- the return path of the coalesced dispatch: each
 * destination rank pre-reduces a token's slots it holds into the token's
 * coalesced row, then the token sums its rows.
 *
 * RailWave, section 3.1 (token coalescing) and section 3 (combine reuses the
 * dispatch metadata).  Reading: the returned row is bf16, like the payload.
 *
 *   y        [T*k, H]  bf16 expert outputs in plain receive order
 *   slot_of  [T, k]    from moe_layout
 *   topk_w   [T, k]    fp32 router weights
 *   crow     [T, k]    from moe_layout_coalesced
 *   rows     capacity of partial in rows (crow < rows; T * min(k, R) always
 *            suffices)
 *   partial  [rows, H] out: bf16; partial[c] = bf16(sum over the slots j of
 *            row c's token with crow[t, j] == c, in increasing j, of
 *            w[t, j] * y[slot_of[t, j]]), fp32 fused multiply-adds from +0
 *   out      [T, H]    out: bf16 (MOE_OUT_BF16) or fp32 (MOE_OUT_F32); fp32
 *            sum from +0 of the token's distinct rows, in order of their
 *            first slot, rounded once
 *
 * One token-major launch (each unit folds a token's slots into its rows and
 * sums them for the token in the same pass).  1 <= k <= 32 (larger k:
 * MOE_ERR_UNSUPPORTED); H % 8 == 0.  Rows of crow outside [0, rows) set
 * MOE_ERRBIT_BAD_INDEX and are skipped.  Not bit-identical to moe_combine:
 * each rank's share is rounded to bf16.
 */
MOE_API moe_status moe_combine_coalesced(int T, int H, int k, const void *y,
                                 const int32_t *slot_of, const float *topk_w,
                                 const int32_t *crow, int rows, void *partial, void *out,
                                 int out_dtype, uint32_t *err_word, cudaStream_t stream);

/*
 * moe_dispatch_combine_flagged -- dispatch, an identity expert and combine in
 * one persistent kernel, each hop synchronised by the reader observing the
 * data's readiness instead of a kernel boundary.
 *
 * UBEP, section 3.4 and Figure 6 (Data-as-Flag: Token-Flag Fusion,
 * Data-for-Checksum, Sentinel Polling), section 3.2 (consumers start as soon
 * as their inputs are signalled) and section 6 (without atomic 512-byte
 * writes, fall back to explicit fences).  Three phases per warp, in one
 * cooperative launch:
 *   produce  recv[slot_of[t, j]] = x[t]                     (token order)
 *   expert   y[s] = recv[s], the identity expert     (receive-row order)
 *   combine  out[t] = sum_j w[t, j] * y[slot_of[t, j]]      (token order),
 *            fp32 fused multiply-adds in slot order from +0, one rounding
 * The expert and combine phases read rows written by other SMs; how they know
 * the rows have arrived is `mode`, at granularity `block_bytes` (G):
 *   MOE_SYNC_WORD      a 32-bit word per (row, G-byte block) per hop, set to
 *                      `epoch` after a fence; G a power of two from 16 to
 *                      1024, or a multiple of 512 from 2048 (a warp moves at
 *                      least 2048 bytes of a row between fences, so blocks of
 *                      one such unit are published together)
 *   MOE_SYNC_SENTINEL  no words.  recv and y must hold 0xFFFFFFFF in every
 *                      32-bit word before the call (memset 0xFF); readers
 *                      poll the data until no word is the sentinel and write
 *                      it back after use, so a call that succeeds leaves them
 *                      ready for the next.  After a call that reports an
 *                      error, refill both.  A payload word equal to the
 *                      sentinel (two bf16 0xFFFF NaNs) sets
 *                      MOE_ERRBIT_SENTINEL.  G is ignored (every word is
 *                      checked) but must still be valid as for WORD
 *   MOE_SYNC_BATCH     a 64-bit (epoch, checksum) word per (row, G-byte
 *                      batch) per hop, G a multiple of 512; the checksum is
 *                      the sum of the first 32-bit word of each 512-byte
 *                      block, and a reader that finds a different sum sets
 *                      MOE_ERRBIT_CHECKSUM
 *   MOE_SYNC_BARRIER   no readiness: a grid barrier between the phases
 *
 *   x        [T, H]    bf16 token rows
 *   slot_of  [T, k]    from moe_layout
 *   topk_w   [T, k]    fp32 router weights
 *   recv, y  [T*k, H]  bf16: the dispatched rows and the expert's output
 *   out      [T, H]    bf16 (MOE_OUT_BF16) or fp32 (MOE_OUT_F32)
 *   words    moe_sync_words(T, H, k, mode, block_bytes) uint32 device words,
 *            zero-filled once (may be NULL when that is 0); WORD and BATCH:
 *            none may already hold `epoch`
 *   epoch    non-zero and different on every call that reuses `words`
 *            (WORD and BATCH)
 *   spin_limit_ns   bound on each expert-phase wait; combine-phase waits get
 *            three times as long (one may sit behind an expert wait that ran
 *            out).  A wait that runs out sets MOE_ERRBIT_TIMEOUT and leaves
 *            that unit unwritten; the warp then stops waiting for data that
 *            is not already there, and the kernel returns
 *   fault_skip_pair test hook: the producer of pair t*k+j == fault_skip_pair
 *            publishes nothing for it (WORD, BATCH) or does not write it
 *            (SENTINEL), so the readers of that row time out; -1 in normal
 *            use, ignored by BARRIER
 *
 * Results: recv = moe_dispatch(x, slot_of) and y = recv (WORD, BATCH,
 * BARRIER; SENTINEL leaves both sentinel-filled), out = moe_combine(y,
 * slot_of, topk_w).  1 <= k <= 32 (larger k: MOE_ERR_UNSUPPORTED); H % 8 == 0.
 */
MOE_API size_t moe_sync_words(int T, int H, int k, int mode, int block_bytes);

MOE_API moe_status moe_dispatch_combine_flagged(int T, int H, int k, const void *x,
                                        const int32_t *slot_of, const float *topk_w,
                                        void *recv, void *y, void *out, int out_dtype,
                                        int mode, int block_bytes, uint32_t *words,
                                        uint32_t epoch, uint64_t spin_limit_ns,
                                        int64_t fault_skip_pair, uint32_t *err_word,
                                        cudaStream_t stream);

/*
 * moe_ep_reorder -- the receiver's reorder of expert-parallel dispatch across
 * real ranks, and its inverse on the combine's return path.
 *
 * UBEP, section 2.3 and Figure 2 (the receive region is partitioned by source
 * rank and expert; in Phase 5 the receiver computes offsets from every
 * source's per-expert counts and reorders the tokens contiguously per
 * expert) and section 4 (receive address space partitioned in advance);
 * StrataCL, Appendix D (the same counts return the rows on the combine path).
 *
 * With experts spread over W ranks (El = E / W local experts each), every
 * rank runs moe_layout with R = W over its own tokens and moe_dispatch; the
 * rank segments of its receive buffer are its sends.  After the exchange
 * (an all-to-all of those segments) a receiver holds the rows source by
 * source -- for source s, its rows for local expert 0, 1, ... in s's (token,
 * slot) order.  This call places them expert-major: for local expert el the
 * rows of source 0, then 1, ..., each in its source's order.
 *
 *   recv_counts  [W, El] int32 device: rows source s sent for local expert
 *                el (the El counts of this rank's experts in s's
 *                expert_counts)
 *   rows         the sum of recv_counts; src and dst hold `rows` rows
 *   src, dst     [rows, H] bf16, 16-byte aligned, not the same buffer
 *   direction    MOE_EP_TO_EXPERT: dst[expert-major(q)] = src[q] (dispatch);
 *                MOE_EP_TO_SOURCE: dst[q] = src[expert-major(q)] (the return
 *                path: expert outputs back to source-major order)
 *   local_expert_offsets  [El+1] int32 device out, may be NULL: first row of
 *                each local expert in the expert-major order; [El] = rows
 *
 * Counts that are negative or do not add up to `rows` set
 * MOE_ERRBIT_BAD_INDEX and copy nothing.  W * El <= MOE_MAX_EXPERTS
 * (larger: MOE_ERR_UNSUPPORTED); H % 8 == 0.
 */
#define MOE_EP_TO_EXPERT 0
#define MOE_EP_TO_SOURCE 1

MOE_API moe_status moe_ep_reorder(int W, int El, int H, const int32_t *recv_counts, int rows,
                                  const void *src, void *dst, int direction,
                                  int32_t *local_expert_offsets, uint32_t *err_word,
                                  cudaStream_t stream);

/*
 * moe_ep_reorder_rows -- moe_ep_reorder for rows of any payload: `row_bytes`
 * bytes per row (a multiple of 4; src and dst 4-byte aligned, 16-byte aligned
 * rows of a multiple of 16 bytes move as 16-byte vectors).  With the FP8
 * dispatch across ranks (UBEP Table 3: W8A8) a receiver reorders the E4M3
 * code rows (H bytes) and the scale rows (H / 128 fp32) with two calls on the
 * same counts.  Same counts, directions, offsets and errors as
 * moe_ep_reorder.
 */
MOE_API moe_status moe_ep_reorder_rows(int W, int El, int row_bytes, const int32_t *recv_counts,
                                       int rows, const void *src, void *dst, int direction,
                                       int32_t *local_expert_offsets, uint32_t *err_word,
                                       cudaStream_t stream);

/*
 * moe_layout_noalloc -- moe_layout for callers that cannot allocate device
 * memory.  The pages have no counterpart: this is a deployment convenience.
 *
 * Some callers cannot call cudaMalloc (or an allocator built on it) when they
 * run the layout -- for example code handed fixed buffers by a host framework
 * that owns all allocation, or a runtime that forbids allocation after start-
 * up -- so they cannot supply moe_layout's workspace.  This entry point takes
 * the same arguments minus the workspace and produces the same outputs as
 * moe_layout; the per-tile count table lives in a fixed device array of
 * MOE_NOALLOC_SCRATCH_BYTES compiled into the library, which every GPU that
 * loads the library holds until the process exits.
 *
 * The first call on a device (with that device current) looks up the array's
 * device address; make that first call before any stream capture.  All calls
 * on one device share the array and its contents persist between calls:
 * calls whose work overlaps on the GPU (unordered streams) race on it.
 * Each call clears the part that must start at zero (8 bytes, on the
 * stream), so the caller never clears anything.  Requests whose count table would exceed
 * MOE_NOALLOC_SCRATCH_BYTES (more than 512 experts with the largest token
 * counts) return MOE_ERR_UNSUPPORTED without launching; moe_layout handles
 * them.  The call allocates and frees nothing.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (256u * 1024u)

MOE_API moe_status moe_layout_noalloc(int T, int k, int E, int R, const int32_t *topk_idx,
                              int32_t *expert_counts, int32_t *expert_offsets,
                              int32_t *rank_offsets, int32_t *slot_of, int32_t *src_of,
                              uint32_t *err_word, cudaStream_t stream);

/*
 * moe_read_error -- synchronise `stream`, read the device error word into
 * *bits_out (may be NULL), clear it when `clear` is non-zero, and return the
 * status of the most serious bit set, in this order:
 *   MOE_ERRBIT_LAUNCH                        -> MOE_ERR_CUDA
 *   MOE_ERRBIT_TIMEOUT                       -> MOE_ERR_TIMEOUT
 *   MOE_ERRBIT_BAD_INDEX                     -> MOE_ERR_BAD_INDEX
 *   MOE_ERRBIT_SENTINEL, MOE_ERRBIT_CHECKSUM -> MOE_ERR_INTEGRITY
 * and MOE_OK when no bit is set.  MOE_ERR_CUDA also if the synchronisation or
 * the copy fails.  The error word is a separate argument of every call, not a
 * part of a workspace: the dispatch and combine calls take no workspace, and
 * one word can collect the errors of a whole step of calls.
 */
MOE_API moe_status moe_read_error(uint32_t *err_word, int clear, cudaStream_t stream,
                          uint32_t *bits_out);

/*
 * moe_e4m3_encode_bits -- diagnostic: the channel encoding moe_dispatch_quant
 * applies (after scaling by 448 / amax), on the fp32 values whose bit patterns
 * are first, first + 1, ..., first + count - 1 (modulo 2^32): codes[i] =
 * E4M3 code of that value, nearest-even, saturating to +-448, infinities to
 * +-448.  The pages have no counterpart; the call exists so that the kernel's
 * encoding can be checked against the format's definition on every fp32
 * input.  codes: count device bytes.  NaN inputs give a NaN code whose sign
 * is not specified.
 */
MOE_API moe_status moe_e4m3_encode_bits(uint32_t first, uint32_t count, uint8_t *codes,
                                        cudaStream_t stream);

/*
 * moe_layout_last_form -- diagnostic: which form of the layout kernel the most
 * recent moe_layout, moe_layout_dispatch, moe_layout_coalesced or
 * moe_layout_noalloc call made by this host thread launched.  The pages have
 * no counterpart; tests use it to check that a given shape took the form
 * they mean to exercise.
 *   MOE_LAYOUT_FORM_NONE         nothing launched (T == 0, or no call yet)
 *   MOE_LAYOUT_FORM_SINGLE       one CTA (at most one tile of pairs)
 *   MOE_LAYOUT_FORM_CLUSTER      one thread-block cluster of 2..16 CTAs
 *   MOE_LAYOUT_FORM_COOPERATIVE  a cooperative grid with a grid barrier in the
 *                                workspace (more than 16 tiles, or a cluster
 *                                the GPU could not place)
 *   MOE_LAYOUT_FORM_FUSED        moe_layout_dispatch's single kernel, in
 *                                which every CTA computes the whole layout
 *                                itself (small batches; see there)
 */
#define MOE_LAYOUT_FORM_NONE 0
#define MOE_LAYOUT_FORM_SINGLE 1
#define MOE_LAYOUT_FORM_CLUSTER 2
#define MOE_LAYOUT_FORM_COOPERATIVE 3
#define MOE_LAYOUT_FORM_FUSED 4

MOE_API int moe_layout_last_form(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_EP_H */

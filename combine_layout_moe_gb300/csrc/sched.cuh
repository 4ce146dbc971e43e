// Dynamic tail for the dispatch kernels (sm_103a).
//
// A static split gives each CTA (or warp) an equal share of the units, but
// the CTAs of one launch do not move bytes at equal rates: six one-warp CTAs
// of the bulk dispatch share each SM, and on GB300 their rates differ by more
// than half between the slowest and the fastest tenth, so a static split
// ends when the slowest CTA ends while the SMs of the others idle.  Each CTA
// (bulk dispatch) or warp (FP8 dispatch) therefore takes a fixed part of the
// work as its own and then draws the rest, a few units at a time, from a pool
// shared by the launch: those that run ahead take more.
//
// The pool counter lives in a slot of a file-scope table in device memory
// (the library allocates nothing per call).  The host hands out slots round
// robin, one per launch; the last CTA of a launch to finish zeroes its slot,
// so the slot is clean for its next user -- including the next replay of a
// captured CUDA graph, which reuses the slot it was captured with (replays of
// one graph are ordered, so they never share a slot at the same time).  Two
// launches share a slot at the same time only if SCHED_SLOTS launches of the
// same kernel run concurrently on one device, far more than the hardware
// runs at once.
#pragma once

#include <atomic>
#include <cstdint>

namespace moe {

constexpr int SCHED_SLOTS = 1024;

struct SchedSlot {
    unsigned long long taken;  // units drawn from the pool so far
    unsigned int done;         // CTAs that have finished
    unsigned int pad;
};

// One thread per CTA, once, after the CTA's last draw: counts the CTA out;
// the last one zeroes the slot.  The fence orders every draw of this CTA
// before its count, so the reset follows every draw of the launch.
__device__ __forceinline__ void sched_finish(SchedSlot *s)
{
    __threadfence();
    if (atomicAdd(&s->done, 1u) == gridDim.x - 1) {
        atomicExch(&s->taken, 0ull);
        atomicExch(&s->done, 0u);
    }
}

// Host: units per draw so that each draw covers at least SCHED_DRAW_BYTES of
// the launch's HBM traffic.  Draws on one counter are serialised where the
// counter lives; at this spacing a launch moving bytes near the HBM's rate
// asks for one draw every few nanoseconds at most, well inside what the
// counter sustains (measured on one GB300: one-item draws of 4 KB items on
// 65536 tokens slowed the FP8 dispatch from 206 to 253 us).
constexpr int64_t SCHED_DRAW_BYTES = 16384;
inline int sched_grab(int64_t unit_bytes)
{
    const int64_t g = (SCHED_DRAW_BYTES + unit_bytes - 1) / (unit_bytes > 0 ? unit_bytes : 1);
    return (int)(g < 1 ? 1 : g);
}

// Host: the slot for the next launch of one kernel family.
inline int next_sched_slot(std::atomic<unsigned> &seq)
{
    return (int)(seq.fetch_add(1u, std::memory_order_relaxed) % (unsigned)SCHED_SLOTS);
}

}  // namespace moe

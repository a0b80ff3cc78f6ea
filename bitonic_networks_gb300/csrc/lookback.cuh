// lookback.cuh -- warp-wide decoupled look-back over one state word per tile
// ([CUDA3] "Stream Compaction", single pass with decoupled look-back), shared
// by the compaction and the 2-way split kernels.
//
// Tile t publishes its own count first (AGG, or PREFIX for tile 0), then lane
// l of the calling warp inspects tile t-1-l: one round reads 32 predecessors;
// the nearest PREFIX ends the walk and the AGG counts after it are summed.
// An empty word means a predecessor has not published: the whole window is
// re-read after a back-off, at most spin_limit times.  The state words sit
// `stride` words apart (a 128-byte line each), so the polling of many waiting
// tiles spreads over many L2 lines.
#pragma once

#include "gsort_internal.cuh"

namespace gsort {
namespace {

// Called by all 32 lanes of one warp.  Returns the exclusive prefix of the
// tile (0 for tile 0) in every lane; ok = false when a wait gave up or the
// abort flag was raised.  stall_tile (testing): that tile publishes nothing.
__device__ __forceinline__ uint32_t warp_look_back(uint32_t *states, uint32_t stride, uint32_t tile,
                                                   uint32_t total, uint32_t stall_tile,
                                                   uint32_t spin_limit, const uint32_t *abort_flag,
                                                   bool &ok) {
    const uint32_t lane = threadIdx.x & 31;
    uint32_t prefix = 0;
    ok = true;
    if (lane == 0 && tile != stall_tile)
        st_relaxed(states + tile * stride, (tile == 0 ? kFlagPrefix : kFlagAgg) | total);
    if (tile == 0 || tile == stall_tile) return 0;
    int32_t t = static_cast<int32_t>(tile) - 1 - static_cast<int32_t>(lane);
    uint32_t polls = 0, ns = 32;
    while (true) {
        const uint32_t s = (t >= 0) ? ld_relaxed(states + t * stride) : kFlagPrefix;   // empty prefix before tile 0
        const uint32_t flag = s & ~kValueMask;
        const uint32_t pmask = __ballot_sync(kFullMask, flag == kFlagPrefix);
        const uint32_t zmask = __ballot_sync(kFullMask, flag == 0);
        // lanes up to and including the nearest published prefix matter
        const uint32_t need = pmask ? (((pmask & (0u - pmask)) << 1) - 1u) : kFullMask;
        if (zmask & need) {
            ++polls;
            if (__any_sync(kFullMask, polls >= spin_limit || ld_relaxed(abort_flag) != 0)) {
                ok = false;
                return prefix;
            }
            backoff(ns);
            continue;   // re-read the whole window
        }
        prefix += __reduce_add_sync(kFullMask, ((need >> lane) & 1u) ? (s & kValueMask) : 0u);
        if (pmask != 0) break;
        t -= 32;
    }
    if (lane == 0) st_relaxed(states + tile * stride, kFlagPrefix | (prefix + total));
    return prefix;
}

}  // namespace
}  // namespace gsort

// bitonic.cu -- batched bitonic sort of independent segments of <= 1024 keys
// ([GPUSORT] sort of up to 1024 elements per block, padded with 0xFFFFFFFF;
// [PMPP10] 10.2: for block size k = 2, 4, ..., N and distance j = k/2, ..., 1,
// element i is compare-exchanged with i^j, ascending when bit k of i is
// clear).
//
// One warp sorts one segment, padded to Lp = 32 * R keys (R = 1..32 keys per
// lane).  Lane l holds elements l*R .. l*R + R-1 in registers, so the low
// log2(R) bits of an element index are register bits and the top five are
// lane bits:
//   - steps on a register bit are compare-exchanges between two registers of
//     one thread (no communication);
//   - steps on a lane bit pair a register with the same register of lane
//     l ^ (j/R), exchanged with one shuffle; the lower lane keeps the minimum.
// For stages whose direction bit is a lane bit, a descending lane complements
// its keys for the stage (min and max swap roles under complement), so every
// compare-exchange in registers is an ascending one.  The page kernels run
// the same network in shared memory with a barrier per step.
//
// Global traffic: each key is read once and written once, coalesced; shared
// memory (padded to avoid bank conflicts) turns the coalesced order into the
// per-lane blocked order and back.
#include <algorithm>

#include "gsort_internal.cuh"

namespace gsort {
namespace {

constexpr int kSegWarps = 4;   // segments per block

// Compare-exchange of registers r and r | (1 << b) for every r with bit b
// clear; ascending unless the compile-time direction bit says otherwise.
template <int LOG_R, int S, int B>
__device__ __forceinline__ void register_step(uint32_t (&x)[1 << LOG_R]) {
    constexpr int R = 1 << LOG_R;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (r & (1 << B)) continue;
        const int r2 = r | (1 << B);
        // direction bit S of the element index is a register bit only for S < LOG_R
        const bool asc = (S >= LOG_R) || ((r >> S) & 1) == 0;
        const uint32_t lo = min(x[r], x[r2]);
        const uint32_t hi = max(x[r], x[r2]);
        x[r] = asc ? lo : hi;
        x[r2] = asc ? hi : lo;
    }
}

// All register steps of stage S (b = min(S, LOG_R) - 1 .. 0).
template <int LOG_R, int S, int B>
__device__ __forceinline__ void register_steps_down(uint32_t (&x)[1 << LOG_R]) {
    if constexpr (B >= 0) {
        register_step<LOG_R, S, B>(x);
        register_steps_down<LOG_R, S, B - 1>(x);
    }
}

// Stages 1 .. LOG_R: every step is a register step.  Stage LOG_R's direction
// bit is lane bit 0: a descending lane holds its keys complemented.
template <int LOG_R, int S>
__device__ __forceinline__ void early_stages(uint32_t (&x)[1 << LOG_R], uint32_t lane) {
    if constexpr (S <= LOG_R) {
        if constexpr (S == LOG_R) {
            const uint32_t f = 0u - (lane & 1u);
#pragma unroll
            for (int r = 0; r < (1 << LOG_R); ++r) x[r] ^= f;
        }
        register_steps_down<LOG_R, S, S - 1>(x);
        early_stages<LOG_R, S + 1>(x, lane);
    }
}

template <int LOG_R>
__device__ __forceinline__ void bitonic_registers(uint32_t (&x)[1 << LOG_R], uint32_t lane) {
    constexpr int R = 1 << LOG_R;
    constexpr int LOG_LP = LOG_R + 5;
    if constexpr (LOG_R > 0) early_stages<LOG_R, 1>(x, lane);
    // Stages LOG_R+1 .. LOG_LP: lane steps on bits s-1 .. LOG_R, then the
    // register steps.  The direction bit s is lane bit s - LOG_R (none in the
    // last stage); the keys are complemented by the change of direction from
    // the previous stage.  A runtime loop keeps the code small.
#pragma unroll 1
    for (int s = (LOG_R > 0 ? LOG_R + 1 : 1); s <= LOG_LP; ++s) {
        const uint32_t want = (s < LOG_LP) ? (0u - ((lane >> (s - LOG_R)) & 1u)) : 0u;
        const uint32_t prev = (s - 1 >= LOG_R && s - 1 >= 1)
                                  ? (0u - ((lane >> (s - 1 - LOG_R)) & 1u)) : 0u;
        const uint32_t f = want ^ prev;
#pragma unroll
        for (int r = 0; r < R; ++r) x[r] ^= f;
#pragma unroll 1
        for (int b = s - 1; b >= LOG_R; --b) {
            const uint32_t m = 1u << (b - LOG_R);
            const bool lower = (lane & m) == 0;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t y = __shfl_xor_sync(kFullMask, x[r], m);
                x[r] = lower ? min(x[r], y) : max(x[r], y);
            }
        }
        register_steps_down<LOG_R, LOG_LP, LOG_R - 1>(x);   // ascending (complement handles direction)
    }
}

template <int LOG_R>
__global__ void __launch_bounds__(kSegWarps * 32)
k_bitonic_segments(uint32_t *keys, uint32_t num_segments, uint32_t len) {
    constexpr int R = 1 << LOG_R;
    constexpr int LP = 32 * R;
    constexpr int PADDED = LP + LP / 32;
    __shared__ uint32_t s_all[kSegWarps * PADDED];
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t seg = blockIdx.x * kSegWarps + warp;
    if (seg >= num_segments) return;   // whole warp: no block-wide barrier below
    uint32_t *sw = s_all + warp * PADDED;
    uint32_t *g = keys + static_cast<size_t>(seg) * len;

    // coalesced load, padded to Lp with 0xFFFFFFFF; shared index e + e/32
#pragma unroll
    for (int c = 0; c < R; ++c) {
        const uint32_t e = c * 32 + lane;
        sw[e + (e >> 5)] = e < len ? g[e] : 0xFFFFFFFFu;
    }
    __syncwarp();
    uint32_t x[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint32_t e = lane * R + r;
        x[r] = sw[e + (e >> 5)];
    }

    bitonic_registers<LOG_R>(x, lane);

    __syncwarp();
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint32_t e = lane * R + r;
        sw[e + (e >> 5)] = x[r];
    }
    __syncwarp();
#pragma unroll
    for (int c = 0; c < R; ++c) {
        const uint32_t e = c * 32 + lane;
        if (e < len) g[e] = sw[e + (e >> 5)];
    }
}

template <int LOG_R>
cudaError_t launch_seg(uint32_t *keys, uint32_t num_segments, uint32_t len, cudaStream_t s) {
    const uint32_t grid = (num_segments + kSegWarps - 1) / kSegWarps;
    k_bitonic_segments<LOG_R><<<grid, kSegWarps * 32, 0, s>>>(keys, num_segments, len);
    return cudaGetLastError();
}

}  // namespace

int launch_segmented_bitonic(uint32_t *keys, int64_t num_segments, int segment_len,
                             cudaStream_t stream) {
    if (num_segments == 0 || segment_len <= 1) return GSORT_OK;
    int log_lp = 5;
    while ((1 << log_lp) < segment_len) ++log_lp;
    const uint32_t ns = static_cast<uint32_t>(num_segments);
    const uint32_t len = static_cast<uint32_t>(segment_len);
    cudaError_t e;
    switch (log_lp - 5) {
        case 0: e = launch_seg<0>(keys, ns, len, stream); break;
        case 1: e = launch_seg<1>(keys, ns, len, stream); break;
        case 2: e = launch_seg<2>(keys, ns, len, stream); break;
        case 3: e = launch_seg<3>(keys, ns, len, stream); break;
        case 4: e = launch_seg<4>(keys, ns, len, stream); break;
        default: e = launch_seg<5>(keys, ns, len, stream); break;
    }
    return e == cudaSuccess ? GSORT_OK : GSORT_ECUDA;
}

}  // namespace gsort

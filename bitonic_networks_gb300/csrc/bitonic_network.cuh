// bitonic_network.cuh -- the register bitonic network of one warp, shared by
// the fixed-length batched sort (bitonic.cu) and the small segments of the
// variable-length segmented sort (segsort.cu).  Elements are 32-bit keys or
// 64-bit composites; the network is the one of [PMPP10] 10.2 (block size k =
// 2 .. Lp, distance j = k/2 .. 1, element i compare-exchanged with i^j,
// ascending when bit k of i is clear).
//
// One warp sorts Lp = 32 * R elements (R = 2^LOG_R = 1..32 per lane).  Lane l
// holds elements l*R .. l*R + R-1 in registers, so the low log2(R) bits of an
// element index are register bits and the top five are lane bits:
//   - steps on a register bit are compare-exchanges between two registers of
//     one thread (no communication);
//   - steps on a lane bit pair a register with the same register of lane
//     l ^ (j/R), exchanged with one shuffle; the lower lane keeps the minimum.
// For stages whose direction bit is a lane bit, a descending lane complements
// its elements for the stage (min and max swap roles under complement), so
// every compare-exchange in registers is an ascending one.
#pragma once

#include "gsort_internal.cuh"

namespace gsort {
namespace {

// Compare-exchange of registers r and r | (1 << b) for every r with bit b
// clear; ascending unless the compile-time direction bit says otherwise.
template <int LOG_R, int S, int B, class T>
__device__ __forceinline__ void register_step(T (&x)[1 << LOG_R]) {
    constexpr int R = 1 << LOG_R;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (r & (1 << B)) continue;
        const int r2 = r | (1 << B);
        // direction bit S of the element index is a register bit only for S < LOG_R
        const bool asc = (S >= LOG_R) || ((r >> S) & 1) == 0;
        const T lo = min(x[r], x[r2]);
        const T hi = max(x[r], x[r2]);
        x[r] = asc ? lo : hi;
        x[r2] = asc ? hi : lo;
    }
}

// All register steps of stage S (b = min(S, LOG_R) - 1 .. 0).
template <int LOG_R, int S, int B, class T>
__device__ __forceinline__ void register_steps_down(T (&x)[1 << LOG_R]) {
    if constexpr (B >= 0) {
        register_step<LOG_R, S, B>(x);
        register_steps_down<LOG_R, S, B - 1>(x);
    }
}

// Stages 1 .. LOG_R: every step is a register step.  Stage LOG_R's direction
// bit is lane bit 0: a descending lane holds its keys complemented.
template <int LOG_R, int S, class T>
__device__ __forceinline__ void early_stages(T (&x)[1 << LOG_R], uint32_t lane) {
    if constexpr (S <= LOG_R) {
        if constexpr (S == LOG_R) {
            const T f = T(0) - T(lane & 1u);
#pragma unroll
            for (int r = 0; r < (1 << LOG_R); ++r) x[r] ^= f;
        }
        register_steps_down<LOG_R, S, S - 1>(x);
        early_stages<LOG_R, S + 1>(x, lane);
    }
}

// Stage s >= LOG_R + 1 with every step on a lane bit done by shuffles:
// complement for the stage's direction, lane steps on bits s-1 .. LOG_R, then
// the register steps.
template <int LOG_R, class T>
__device__ __forceinline__ void lane_stage(T (&x)[1 << LOG_R], uint32_t lane, int s) {
    constexpr int R = 1 << LOG_R;
    constexpr int LOG_LP = LOG_R + 5;
    // The direction bit s is lane bit s - LOG_R (none in the last stage); the
    // keys are complemented by the change of direction from the previous stage.
    const uint32_t want = (s < LOG_LP) ? (0u - ((lane >> (s - LOG_R)) & 1u)) : 0u;
    const uint32_t prev = (s - 1 >= LOG_R && s - 1 >= 1) ? (0u - ((lane >> (s - 1 - LOG_R)) & 1u)) : 0u;
    const T f = T(0) - T((want ^ prev) & 1u);
#pragma unroll
    for (int r = 0; r < R; ++r) x[r] ^= f;
#pragma unroll 1
    for (int b = s - 1; b >= LOG_R; --b) {
        const uint32_t m = 1u << (b - LOG_R);
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const T y = __shfl_xor_sync(kFullMask, x[r], m);
            // the lower lane keeps the minimum, the upper the maximum.  With 32
            // keys per lane: take the partner's key when it is on the kept side
            // (one compare, one select; measured 4.6 % faster on 1024-key
            // segments, slower with fewer keys per lane)
            if constexpr (LOG_R == 5) x[r] = ((x[r] > y) != upper) ? y : x[r];
            else x[r] = upper ? max(x[r], y) : min(x[r], y);
        }
    }
    register_steps_down<LOG_R, LOG_LP, LOG_R - 1>(x);   // ascending (complement handles direction)
}

// 32 x 32 transposes through the warp's padded shared buffer (element e at
// word e + e / 32, so both directions touch 32 banks): layout A holds element
// lane * 32 + r in register r, layout B element r * 32 + lane.
template <class T>
__device__ __forceinline__ void transpose_a_to_b(T (&x)[32], T *sw, uint32_t lane) {
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 32; ++r) sw[lane * 33 + r] = x[r];
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 32; ++r) x[r] = sw[r * 33 + lane];
}

template <class T>
__device__ __forceinline__ void transpose_b_to_a(T (&x)[32], T *sw, uint32_t lane) {
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 32; ++r) sw[r * 33 + lane] = x[r];
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 32; ++r) x[r] = sw[lane * 33 + r];
}

// Stage S (8 .. 10) of the 1024-element network: after the complement for
// the stage's direction (in layout A, where the direction bit is a lane bit),
// the steps on element bits S-1 .. 5 run in layout B, where those bits are
// register bits S-6 .. 0 (two-instruction compare-exchanges instead of a
// shuffle, a compare and a select per key); then the steps on bits 4 .. 0 in
// layout A.  The complemented keys travel with their elements, so every
// compare-exchange stays ascending in both layouts.
template <int S, class T>
__device__ __forceinline__ void transposed_stage(T (&x)[32], uint32_t lane, T *sw) {
    constexpr int LOG_LP = 10;
    const uint32_t want = (S < LOG_LP) ? (0u - ((lane >> (S - 5)) & 1u)) : 0u;
    const uint32_t prev = 0u - ((lane >> (S - 6)) & 1u);
    const T f = T(0) - T((want ^ prev) & 1u);
#pragma unroll
    for (int r = 0; r < 32; ++r) x[r] ^= f;
    transpose_a_to_b(x, sw, lane);
    register_steps_down<5, LOG_LP, S - 6>(x);
    transpose_b_to_a(x, sw, lane);
    register_steps_down<5, LOG_LP, 4>(x);
}

// The whole network.  sw: the warp's padded shared buffer of 32 * R + R
// elements (used, by the 1024-element network of 32-bit keys only, for the
// transposes of stages 8 .. 10; its contents are overwritten).  Measured on
// 1024-key segments: 13 % faster with the transposes for 32-bit keys, 25 %
// slower for 64-bit composites, which keep the shuffles.
template <int LOG_R, class T>
__device__ __forceinline__ void bitonic_registers(T (&x)[1 << LOG_R], uint32_t lane, T *sw) {
    constexpr int LOG_LP = LOG_R + 5;
    constexpr bool kTransposed = LOG_R == 5 && sizeof(T) == 4;
    if constexpr (LOG_R > 0) early_stages<LOG_R, 1>(x, lane);
    // Stages LOG_R+1 .. LOG_LP: lane steps on bits s-1 .. LOG_R, then the
    // register steps.  A runtime loop keeps the code small.
    constexpr int kLaneStages = kTransposed ? 7 : LOG_LP;   // last stage done with shuffles
#pragma unroll 1
    for (int s = (LOG_R > 0 ? LOG_R + 1 : 1); s <= kLaneStages; ++s) lane_stage<LOG_R>(x, lane, s);
    if constexpr (kTransposed) {
        transposed_stage<8>(x, lane, sw);
        transposed_stage<9>(x, lane, sw);
        transposed_stage<10>(x, lane, sw);
    }
}

}  // namespace
}  // namespace gsort

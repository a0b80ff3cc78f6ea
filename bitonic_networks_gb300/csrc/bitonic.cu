// bitonic.cu -- batched bitonic sort of independent segments of <= 1024 keys
// ([GPUSORT] sort of up to 1024 elements per block, padded with 0xFFFFFFFF;
// [PMPP10] 10.2: for block size k = 2, 4, ..., N and distance j = k/2, ..., 1,
// element i is compare-exchanged with i^j, ascending when bit k of i is
// clear).
//
// One warp sorts one segment, padded to Lp = 32 * R keys (R = 1..32 keys per
// lane), with the register network of bitonic_network.cuh.  The page kernels
// run the same network in shared memory with a barrier per step.
//
// Global traffic: each key is read once and written once, coalesced; shared
// memory (padded to avoid bank conflicts) turns the coalesced order into the
// per-lane blocked order and back.
#include <algorithm>

#include "bitonic_network.cuh"

namespace gsort {
namespace {

constexpr int kSegWarps = 4;   // segments per block

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

    bitonic_registers<LOG_R>(x, lane, sw);

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

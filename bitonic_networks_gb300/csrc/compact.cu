// compact.cu -- stream compaction of the positive floats, the 1-bit special
// case of the radix sort's scatter ([CUDA3] "Stream Compaction": predicate,
// exclusive scan of the predicate, scatter; single pass with decoupled
// look-back and a warp-wide look-back window).
//
// One kernel reads every tile once: predicate, block scan of the per-thread
// counts, publish the tile count, look back (warp 0 inspects 32 earlier tiles
// per step, while the other warps stage the tile's kept values contiguously in
// shared memory) and copy the kept values out as one run.  The output ends in
// +0.0 from m to n (the pages' worked example shows a zero tail; their kernels
// leave it unwritten): a tile with K kept values before it and z dropped ones
// of its own writes its z zeros just below the zeros of the tiles before it,
// at [n - (base - K) - z, n - (base - K)), so the tail fills from the end
// without waiting for m.  The last tile records m.  Traffic: read 4n, write 4n.
#include <algorithm>
#include <mutex>

#include "lookback.cuh"

namespace gsort {
namespace {

constexpr int kCompactThreads = 512;
constexpr int kCompactItems = 16;          // per thread, a multiple of 4
constexpr uint32_t kCompactTile = kCompactThreads * kCompactItems;
// One look-back word per 128-byte line: hundreds of waiting tiles poll their
// predecessors' words at once, and packing the words densely puts all of that
// polling on a few L2 lines.  Spread out, the polls of one window hit 32 lines.
constexpr uint32_t kStateStride = 32;      // words

__global__ void k_zero_words(uint32_t *p, uint32_t nwords) {
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < nwords;
         i += gridDim.x * blockDim.x)
        p[i] = 0;
}

// +0.0 into out[a, a + count): a head up to a 16-byte boundary, 16-byte
// streaming stores, a tail.  Called by every thread of a block of T.
template <int T>
__device__ __forceinline__ void zero_run(uint32_t *out, uint32_t a, uint32_t count, uint32_t tid) {
    uint32_t head = static_cast<uint32_t>(((16 - (reinterpret_cast<uintptr_t>(out + a) & 15)) & 15) >> 2);
    head = min(head, count);
    const uint32_t nvec = (count - head) >> 2;
    uint4 *vec = reinterpret_cast<uint4 *>(out + a + head);
    for (uint32_t v = tid; v < nvec; v += T) __stcs(vec + v, make_uint4(0, 0, 0, 0));
    if (tid < head) out[a + tid] = 0;
    const uint32_t tail0 = head + nvec * 4;
    if (tid < count - tail0) out[a + tail0 + tid] = 0;
}

// x > 0 under IEEE comparison, on the bit pattern: sign clear, not +0, not
// NaN (0 < bits <= 0x7F800000).  Positive subnormals count as positive.
__device__ __forceinline__ uint32_t is_positive(uint32_t bits) {
    return (bits - 1u) < 0x7F800000u ? 1u : 0u;
}

template <int T, int IPT>
__global__ void __launch_bounds__(T, 4)
k_compact(const uint32_t *__restrict__ in, uint32_t *__restrict__ out, uint32_t n,
          uint32_t *states, uint32_t *tile_counter, uint32_t *status, uint32_t *abort_flag,
          unsigned long long *kept, int64_t *num_kept, uint32_t num_tiles, uint32_t spin_limit,
          uint32_t stall_tile, int vec_ok) {
    constexpr uint32_t TILE = T * IPT;
    constexpr int WARPS = T / 32;
    __shared__ uint32_t s_buf[TILE];
    __shared__ uint32_t s_warp[WARPS];
    __shared__ uint32_t s_misc[4];

    const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_misc[0] = atomicAdd(tile_counter, 1u);
        s_misc[1] = ld_relaxed(abort_flag);
    }
    __syncthreads();
    const uint32_t tile = s_misc[0];
    if (s_misc[1]) return;
    const uint32_t base = tile * TILE;
    const uint32_t tile_n = min(TILE, n - base);

    // blocked arrangement: thread t owns items [t*IPT, t*IPT + IPT) of the tile
    uint32_t x[IPT];
    const uint32_t first = tid * IPT;
    if (tile_n == TILE && vec_ok) {
        const uint4 *src = reinterpret_cast<const uint4 *>(in + base + first);
#pragma unroll
        for (int q = 0; q < IPT / 4; ++q) {
            const uint4 v = __ldcs(src + q);
            x[4 * q + 0] = v.x;
            x[4 * q + 1] = v.y;
            x[4 * q + 2] = v.z;
            x[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < IPT; ++j) x[j] = (first + j < tile_n) ? in[base + first + j] : 0u;
    }
    uint32_t flags = 0;
#pragma unroll
    for (int j = 0; j < IPT; ++j) flags |= is_positive(x[j]) << j;
    const uint32_t cnt = __popc(flags);

    // block exclusive scan of the per-thread counts: warp scans, then every
    // thread adds up the totals of the warps before its own (one barrier)
    const uint32_t incl = warp_inclusive_scan(cnt, lane);
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    uint32_t warp_excl = 0, total = 0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
        const uint32_t c = s_warp[w];
        warp_excl += (static_cast<uint32_t>(w) < warp) ? c : 0u;
        total += c;
    }
    uint32_t pos = warp_excl + incl - cnt;

    if (warp == 0) {
        // publish the tile count at once, then look back over 32 predecessors per round
        bool ok;
        const uint32_t prefix = warp_look_back(states, kStateStride, tile, total, stall_tile,
                                               spin_limit, abort_flag, ok);
        if (lane == 0) {
            s_misc[1] = ok ? 0u : 1u;
            s_misc[3] = prefix;
            if (!ok) record_error(status, abort_flag, GSORT_ETIMEOUT);
        }
    }

    // stage the kept values contiguously (overlaps warp 0's look-back)
#pragma unroll
    for (int j = 0; j < IPT; ++j)
        if ((flags >> j) & 1u) s_buf[pos++] = x[j];
    __syncthreads();
    if (s_misc[1] || tile == stall_tile) return;
    const uint32_t prefix = s_misc[3];

    // copy them out as one run
    for (uint32_t i = tid; i < total; i += T) {
        const uint32_t g = prefix + i;
        if (g < n) out[g] = s_buf[i];
    }
    // this tile's share of the zero tail, below the shares of the tiles before it
    if (prefix <= base) {   // guards the writes should a count ever be corrupt
        const uint32_t dropped_before = base - prefix, dropped = tile_n - total;
        if (static_cast<uint64_t>(dropped_before) + dropped <= n)
            zero_run<T>(out, n - dropped_before - dropped, dropped, tid);
    }
    if (tile == num_tiles - 1 && tid == 0) {
        const unsigned long long m = static_cast<unsigned long long>(prefix) + total;
        *kept = m;
        if (num_kept != nullptr) *num_kept = static_cast<int64_t>(m);
    }
}

void record(cudaEvent_t *ev, int num, int idx, cudaStream_t s) {
    if (ev != nullptr && idx < num && ev[idx] != nullptr) cudaEventRecord(ev[idx], s);
}

}  // namespace

CompactLayout compact_layout(uint32_t n) {
    CompactLayout L{};
    L.tiles = (n + kCompactTile - 1) / kCompactTile;
    L.states = kHdrBytes;
    L.total = kHdrBytes + align_up(static_cast<size_t>(L.tiles) * kStateStride * sizeof(uint32_t), kWsAlign);
    return L;
}

int launch_compact(const CompactLaunch &L) {
    const CompactLayout lay = compact_layout(L.n);
    cudaStream_t s = L.stream;
    uint32_t *words = reinterpret_cast<uint32_t *>(L.ws);
    uint32_t *status = reinterpret_cast<uint32_t *>(L.ws + kHdrStatus);
    uint32_t *abort_flag = reinterpret_cast<uint32_t *>(L.ws + kHdrAbort);
    uint32_t *counter = reinterpret_cast<uint32_t *>(L.ws + kHdrCounters);
    unsigned long long *kept = reinterpret_cast<unsigned long long *>(L.ws + kHdrKept);
    uint32_t *states = reinterpret_cast<uint32_t *>(L.ws + lay.states);

    record(L.events, L.num_events, 0, s);
    const uint32_t init_words = static_cast<uint32_t>(kHdrBytes / 4) + lay.tiles * kStateStride;
    const uint32_t init_grid = std::min<uint32_t>((init_words + 1023) / 1024, 4u * L.sm_count);
    k_zero_words<<<init_grid, 256, 0, s>>>(words, init_words);
    if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
    record(L.events, L.num_events, 1, s);

    const int vec_ok = (reinterpret_cast<uintptr_t>(L.in) & 15) == 0;
    k_compact<kCompactThreads, kCompactItems><<<lay.tiles, kCompactThreads, 0, s>>>(
        L.in, L.out, L.n, states, counter, status, abort_flag, kept, L.num_kept, lay.tiles,
        L.spin_limit, L.stall_tile, vec_ok);
    if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
    record(L.events, L.num_events, 2, s);   // the zero tail is written by the same kernel
    record(L.events, L.num_events, 3, s);
    return GSORT_OK;
}

}  // namespace gsort

// ------------------------------------------------ allocation-free variant
// Some callers cannot hand this library a workspace: code that runs where
// device allocation is forbidden or too costly, such as the execute step of a
// plugin whose host framework owns all device memory, a real-time loop that
// cannot afford cudaMalloc's device-wide synchronisation and unbounded
// latency, or a handler that runs while the caller's own allocator is busy.
// For them, gsort_compact_positive_noalloc keeps its scratch (status words,
// tile counter, kept count and one look-back line per tile) in the static
// device array below (about 4 MiB), sized for GSORT_COMPACT_NOALLOC_MAX_N elements.  Every
// GPU that loads the library holds this array until the process exits.
namespace {

constexpr uint32_t kNoAllocMaxN = GSORT_COMPACT_NOALLOC_MAX_N;
// the compaction workspace for kNoAllocMaxN elements: header + one 128-byte
// look-back line per tile
constexpr size_t kNoAllocScratchBytes =
    gsort::kHdrBytes +
    ((kNoAllocMaxN + gsort::kCompactTile - 1) / gsort::kCompactTile * gsort::kStateStride * 4u + 255u) /
        256u * 256u;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 256;
std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the static scratch on device `dev` (the current device).
// The first call on a device asks the runtime for it; later calls reuse it.
int noalloc_scratch(int dev, void **out) {
    if (dev < 0 || dev >= kMaxDevices) return GSORT_EINVAL;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return GSORT_ECUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return GSORT_OK;
}

}  // namespace

extern "C" int gsort_compact_positive_noalloc(const float *d_in, float *d_out, int64_t n,
                                              int64_t *d_num_kept, cudaStream_t stream) {
    using namespace gsort;
    if (n < 0) return GSORT_EINVAL;
    if (n > static_cast<int64_t>(kNoAllocMaxN)) return GSORT_ETOOBIG;
    if (d_num_kept != nullptr && (reinterpret_cast<uintptr_t>(d_num_kept) & 7) != 0)
        return GSORT_EALIGN;
    if (n > 0) {
        if (d_in == nullptr || d_out == nullptr) return GSORT_EINVAL;
        if ((reinterpret_cast<uintptr_t>(d_in) & 3) != 0 || (reinterpret_cast<uintptr_t>(d_out) & 3) != 0)
            return GSORT_EALIGN;
        const uintptr_t a = reinterpret_cast<uintptr_t>(d_in), b = reinterpret_cast<uintptr_t>(d_out);
        const uintptr_t bytes = static_cast<uintptr_t>(n) * 4;
        if (a < b + bytes && b < a + bytes) return GSORT_EINVAL;
    }
    DeviceInfo dev;
    if (device_info(&dev) != GSORT_OK) return GSORT_ECUDA;
    if (compact_layout(static_cast<uint32_t>(n)).total > kNoAllocScratchBytes) return GSORT_ETOOBIG;
    void *scratch = nullptr;
    const int rc = noalloc_scratch(dev.device, &scratch);
    if (rc != GSORT_OK) return rc;
    if (n == 0) {
        if (d_num_kept != nullptr &&
            cudaMemsetAsync(d_num_kept, 0, sizeof(int64_t), stream) != cudaSuccess)
            return GSORT_ECUDA;
        return GSORT_OK;
    }
    // the compaction's own init kernel clears the header and the look-back
    // words at the start of the call, so the array's old contents do not matter
    CompactLaunch L;
    L.in = reinterpret_cast<const uint32_t *>(d_in);
    L.out = reinterpret_cast<uint32_t *>(d_out);
    L.n = static_cast<uint32_t>(n);
    L.num_kept = d_num_kept;
    L.ws = static_cast<unsigned char *>(scratch);
    L.spin_limit = kDefaultSpinLimit;
    L.stall_tile = kNoStall;
    L.events = nullptr;
    L.num_events = 0;
    L.stream = stream;
    L.sm_count = dev.sm_count;
    return launch_compact(L);
}

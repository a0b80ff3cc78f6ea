// Internal declarations of libgsort: workspace layout, look-back state
// encoding, device primitives and the host launchers each .cu file defines.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "gsort.h"

namespace gsort {

// ----------------------------------------------------------- workspace header
// Byte offsets from the start of every workspace.  The header is cleared by
// the init kernel at the start of each call.
constexpr size_t kHdrStatus = 0;      // u32: 0, or a gsort_status a kernel recorded
constexpr size_t kHdrAbort = 4;       // u32: non-zero once a wait gave up; later tiles bail out
constexpr size_t kHdrCounters = 128;  // u32 tile counters, one per 128-byte line
constexpr int kNumCounters = 8;
constexpr size_t kHdrKept = kHdrCounters + 128 * kNumCounters;  // u64 kept count (compaction)
constexpr size_t kHdrHistDone = kHdrKept + 128;   // u32 finished CTAs of the histogram kernel (radix)
constexpr size_t kHdrHist = 2048;     // u32[4][256] digit histograms (radix, 32-bit keys)
constexpr size_t kHdrCursor = kHdrHist + 4096;   // u32[256] bin cursors of an order-free first pass (radix)
constexpr size_t kHdrHot = kHdrCursor + 1024;    // u32[8] most frequent digit of each pass (radix)
constexpr size_t kHdrBytes = 8192;    // header size, keeps what follows 256-byte aligned
constexpr size_t kWsAlign = 256;

// ------------------------------------------------------------ look-back words
// Three states per tile ([CUDA3] decoupled look-back): 0 = nothing published
// yet; AGG = the tile's own count is published; PREFIX = the count over this
// tile and every earlier tile is published.  The state sits in the top two
// bits of a 32-bit word whose low 30 bits hold the count (hence n <= 2^30 - 1):
// one word per tile (compaction) or per tile and digit (radix sort).
constexpr uint32_t kFlagAgg = 1u << 30;
constexpr uint32_t kFlagPrefix = 2u << 30;
constexpr uint32_t kValueMask = (1u << 30) - 1;
constexpr uint32_t kDefaultSpinLimit = 1u << 20;  // polls; with back-off about a second
constexpr uint32_t kNoStall = 0xFFFFFFFFu;

// Smallest tile of any digit-pass variant; sizes the look-back regions.
constexpr uint32_t kMinRadixTile = 4096;

constexpr uint32_t kFullMask = 0xFFFFFFFFu;

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(uint32_t *p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Atomic add with release semantics: every write that precedes it (in this
// thread, or in threads ordered before it by a barrier) is visible to a
// thread that observes the new value with an acquire load.
__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Inclusive warp scan (Kogge-Stone over shuffles).
__device__ __forceinline__ uint32_t warp_inclusive_scan(uint32_t v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t t = __shfl_up_sync(kFullMask, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Records a device-side error once and raises the abort flag.
__device__ __forceinline__ void record_error(uint32_t *status, uint32_t *abort_flag, int code) {
    atomicCAS(status, 0u, static_cast<uint32_t>(code));
    atomicExch(abort_flag, 1u);
}

// Back-off between polls of a look-back word.
__device__ __forceinline__ void backoff(uint32_t &ns) {
    __nanosleep(ns);
    if (ns < 1024) ns <<= 1;
}

// ------------------------------------------- mbarrier + TMA bulk copies
// One-dimensional bulk copies global -> shared through the tensor memory
// accelerator, completed on an mbarrier (transaction-count based).  Both
// addresses and the size must be multiples of 16 bytes.
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for phase `parity` of the barrier, at most `limit` polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Orders this thread's earlier generic-proxy accesses of shared memory before
// later async-proxy (TMA) writes to it.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// -------------------------------------------------------- host-side helpers
struct DeviceInfo {
    int device;
    int sm_count;
};
int device_info(DeviceInfo *out);  // returns GSORT_OK or GSORT_ECUDA; cached per device

// Per-device caches of kernel properties, so that a call costs no more host
// time than its launches: the dynamic shared-memory limit of a kernel (set
// once per device and size) and its resident CTAs per SM.
cudaError_t set_smem_limit(const void *kernel, size_t bytes);
cudaError_t blocks_per_sm(const void *kernel, int threads, size_t smem, int *out);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------ launch plans
// Order map of a key kind and direction: ordered = (float ? float_map(bits)
// : bits) ^ flip, on key words of key_bytes bytes.
struct KeyOrder {
    int key_bytes;
    uint64_t fmask;   // all ones for float kinds, else 0
    uint64_t flip;    // sign bit for signed kinds, complemented for descending order
};
KeyOrder key_order(int kind, int flags);

// Bytes of one key of `kind` (4 or 8), 0 for an unknown kind.
inline int key_kind_bytes(int kind) {
    switch (kind) {
        case GSORT_KEY_U32: case GSORT_KEY_F32: case GSORT_KEY_I32: return 4;
        case GSORT_KEY_U64: case GSORT_KEY_F64: case GSORT_KEY_I64: return 8;
        default: return 0;
    }
}

struct RadixLaunch {
    const void *keys_in;
    void *keys_out;
    const uint32_t *vals_in;  // null: keys only
    uint32_t *vals_out;
    uint32_t n;
    int kind;
    int flags;
    int begin_bit, end_bit;
    unsigned char *ws;
    uint32_t spin_limit;
    uint32_t stall_tile;
    cudaEvent_t *events;
    int num_events;
    int variant;
    cudaStream_t stream;
    int sm_count;
};

// Layout of the radix workspace after the header.
struct RadixLayout {
    uint32_t tiles_max;   // tiles of the smallest tile size any variant uses
    size_t starts;        // u32[8][256] bin starts of every pass (exclusive scans of the histograms)
    size_t hist;          // u32[passes][256] digit histograms
    size_t look_a, look_b;  // [tiles_max][256] look-back words, alternating between passes
    size_t tmp_keys, tmp_vals;
    size_t small_counts;  // 32-bit keys, n <= 2^18: the small-input sort's count buffers
    size_t total;
};
RadixLayout radix_layout(uint32_t n, bool with_values, int key_bytes);

int radix_num_variants();
const char *radix_variant_name(int v);
uint32_t radix_variant_tile(int v);

// Launchers (each returns GSORT_OK or GSORT_ECUDA).
int launch_radix(const RadixLaunch &L);
int launch_digit_histograms(const void *keys, uint32_t n, int kind, int flags, int begin_bit,
                            int end_bit, uint32_t *hist_out, cudaStream_t stream, int sm_count);

struct CompactLayout {
    uint32_t tiles;
    size_t states;
    size_t total;
};
CompactLayout compact_layout(uint32_t n);

struct CompactLaunch {
    const uint32_t *in;
    uint32_t *out;
    uint32_t n;
    int64_t *num_kept;
    unsigned char *ws;
    uint32_t spin_limit;
    uint32_t stall_tile;
    cudaEvent_t *events;
    int num_events;
    cudaStream_t stream;
    int sm_count;
};
int launch_compact(const CompactLaunch &L);

int launch_segmented_bitonic(uint32_t *keys, int64_t num_segments, int segment_len,
                             cudaStream_t stream);

// Small inputs (small.cu): every pass of a 32-bit key sort in one cooperative
// launch.  launch_small_sort returns 1 (and launches nothing) when the grid
// cannot be resident at once; the caller then takes the large-input path.
struct SmallSortLaunch {
    const uint32_t *keys_in;
    uint32_t *keys_out;
    const uint32_t *vals_in;
    uint32_t *vals_out;
    uint32_t *tmp_k, *tmp_v;
    uint32_t n;
    int passes, begin_bit;
    uint32_t last_mask, fmask, flip;
    bool alias;
    uint32_t *counts;            // 3 x [ceil(n / small_sort_tile())][256]
    uint32_t *bar_count;         // zero before the launch
    uint32_t *status, *abort_flag;
    uint32_t spin_limit, stall_tile;
    cudaStream_t stream;
    int sm_count;
};
bool small_sort_applies(uint32_t n, int key_bytes, int variant);
uint32_t small_sort_tile();
int launch_small_sort(const SmallSortLaunch &L);

// Inputs of at most 65,536 32-bit keys (cluster_sort.cu): every pass inside
// one thread-block cluster, keys resident in shared memory; no header clear.
// launch_cluster_sort returns 1 (and launches nothing) when no cluster of its
// shapes can be resident; counts, bar_count, spin_limit and stall_tile of the
// launch description are not used.
bool cluster_sort_applies(uint32_t n, int key_bytes, int variant, uint32_t stall_tile, int passes);
int launch_cluster_sort(const SmallSortLaunch &L);

// 2-way split (split.cu): partition by a predicate, and the 1-bit split sort.
struct SplitLayout {
    uint32_t tiles;
    size_t states_a, states_b;   // one look-back word per tile, 128 bytes apart; b: sort only
    size_t tmp_keys, tmp_vals;   // sort only
    size_t total;
};
SplitLayout split_layout(uint32_t n, bool with_values, bool sort);

struct PartitionLaunch {
    const uint32_t *in;
    uint32_t *out;
    const uint32_t *vals_in;   // null: no values
    uint32_t *vals_out;
    uint32_t n;
    int pred, kind;
    uint32_t param;
    const uint8_t *flags;
    int64_t *num_true;         // may be null
    unsigned char *ws;
    uint32_t spin_limit;
    cudaStream_t stream;
    int sm_count;
};
int launch_partition(const PartitionLaunch &L);

struct SplitSortLaunch {
    const uint32_t *keys_in;
    uint32_t *keys_out;
    const uint32_t *vals_in;
    uint32_t *vals_out;
    uint32_t n;
    int begin_bit, end_bit;
    unsigned char *ws;
    uint32_t spin_limit;
    cudaStream_t stream;
    int sm_count;
};
int launch_split_sort(const SplitSortLaunch &L);

// Variable-length segmented sort (segsort.cu): workspace layout and launch.
struct SegLayout {
    uint32_t small_max;   // segments of 2..1024 keys, at most
    uint32_t large_max;   // segments of more than 1024 keys, at most
    uint32_t tiles_max;   // tiles of the large segments, at most
    size_t small_list, large_start, large_len, tile_base, tiles, hist, look_a, look_b;
    size_t tmp_keys, tmp_vals, total;
};
SegLayout seg_layout(uint32_t n, uint32_t num_segments, bool with_values);

struct SegLaunch {
    const uint32_t *keys_in;
    uint32_t *keys_out;
    const uint32_t *vals_in;   // null: keys only
    uint32_t *vals_out;
    uint32_t n;
    const uint32_t *offsets;   // num_segments + 1 entries
    uint32_t num_segments;
    int kind, flags;
    unsigned char *ws;
    uint32_t spin_limit;
    cudaEvent_t *events;
    int num_events;
    cudaStream_t stream;
    int sm_count;
};
int launch_segmented_sort(const SegLaunch &L);

}  // namespace gsort

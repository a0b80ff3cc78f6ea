// api.cu -- the extern "C" boundary of libgsort: argument validation,
// workspace sizing and launch dispatch.  Validation happens before any CUDA
// call, so every argument error is reported without touching the device.
#include <atomic>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "gsort_internal.cuh"

namespace gsort {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];   // 0: not yet queried

struct KernelKey {
    const void *kernel;
    int device, threads;
    size_t smem;
    bool operator==(const KernelKey &o) const {
        return kernel == o.kernel && device == o.device && threads == o.threads && smem == o.smem;
    }
};
struct KernelKeyHash {
    size_t operator()(const KernelKey &k) const {
        return std::hash<const void *>()(k.kernel) ^ (static_cast<size_t>(k.device) << 48) ^
               (static_cast<size_t>(k.threads) << 32) ^ k.smem;
    }
};
std::mutex g_cache_mutex;
std::unordered_map<KernelKey, int, KernelKeyHash> g_smem_set;    // value unused
std::unordered_map<KernelKey, int, KernelKeyHash> g_occupancy;
}  // namespace

int device_info(DeviceInfo *out) {
    if (cudaGetDevice(&out->device) != cudaSuccess) return GSORT_ECUDA;
    if (out->device >= 0 && out->device < kMaxDevices) {
        const int c = g_sm_count[out->device].load(std::memory_order_relaxed);
        if (c > 0) {
            out->sm_count = c;
            return GSORT_OK;
        }
    }
    if (cudaDeviceGetAttribute(&out->sm_count, cudaDevAttrMultiProcessorCount, out->device) !=
        cudaSuccess)
        return GSORT_ECUDA;
    if (out->device >= 0 && out->device < kMaxDevices)
        g_sm_count[out->device].store(out->sm_count, std::memory_order_relaxed);
    return GSORT_OK;
}

cudaError_t set_smem_limit(const void *kernel, size_t bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const KernelKey key{kernel, dev, 0, bytes};
    {
        std::lock_guard<std::mutex> lock(g_cache_mutex);
        if (g_smem_set.count(key)) return cudaSuccess;
    }
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess) {
        std::lock_guard<std::mutex> lock(g_cache_mutex);
        g_smem_set.emplace(key, 1);
    }
    return e;
}

cudaError_t blocks_per_sm(const void *kernel, int threads, size_t smem, int *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const KernelKey key{kernel, dev, threads, smem};
    {
        std::lock_guard<std::mutex> lock(g_cache_mutex);
        auto it = g_occupancy.find(key);
        if (it != g_occupancy.end()) {
            *out = it->second;
            return cudaSuccess;
        }
    }
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, kernel, threads, smem);
    if (e == cudaSuccess) {
        std::lock_guard<std::mutex> lock(g_cache_mutex);
        g_occupancy.emplace(key, *out);
    }
    return e;
}

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Two ranges of `bytes` each: identical, disjoint, or (bad) partially overlapping.
bool partial_overlap(const void *a, const void *b, size_t bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    if (x == y) return false;
    return x < y + bytes && y < x + bytes;
}

bool ranges_overlap(const void *a, size_t a_bytes, const void *b, size_t b_bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + b_bytes && y < x + a_bytes;
}

bool overlap(const void *a, const void *b, size_t bytes) { return ranges_overlap(a, bytes, b, bytes); }

const gsort_options kDefaults = {0, -1, nullptr, 0, 0};

int radix_args(const void *keys_in, void *keys_out, const uint32_t *vals_in, uint32_t *vals_out,
               int64_t n, int kind, int flags, int begin_bit, int end_bit, const gsort_options *o) {
    if (n < 0) return GSORT_EINVAL;
    if (n > GSORT_MAX_N) return GSORT_ETOOBIG;
    const int kb = key_kind_bytes(kind);
    if (kb == 0) return GSORT_EINVAL;
    if ((flags & ~GSORT_DESCENDING) != 0) return GSORT_EINVAL;
    if (begin_bit < 0 || end_bit > 8 * kb || begin_bit > end_bit) return GSORT_EINVAL;
    if ((vals_in == nullptr) != (vals_out == nullptr)) return GSORT_EINVAL;
    if (kb == 8 ? o->variant != 0 : (o->variant < 0 || o->variant >= radix_num_variants()))
        return GSORT_EINVAL;
    if (o->num_events < 0 || (o->num_events > 0 && o->events == nullptr)) return GSORT_EINVAL;
    if (n == 0) return GSORT_OK;
    if (keys_in == nullptr || keys_out == nullptr) return GSORT_EINVAL;
    if (!aligned(keys_in, kb) || !aligned(keys_out, kb)) return GSORT_EALIGN;
    if (vals_in != nullptr && (!aligned(vals_in, 4) || !aligned(vals_out, 4))) return GSORT_EALIGN;
    const size_t kbytes = static_cast<size_t>(n) * kb, vbytes = static_cast<size_t>(n) * 4;
    if (partial_overlap(keys_in, keys_out, kbytes)) return GSORT_EINVAL;
    if (vals_in != nullptr) {
        if (partial_overlap(vals_in, vals_out, vbytes)) return GSORT_EINVAL;
        if (ranges_overlap(keys_out, kbytes, vals_out, vbytes) ||
            ranges_overlap(keys_in, kbytes, vals_out, vbytes) ||
            ranges_overlap(keys_out, kbytes, vals_in, vbytes))
            return GSORT_EINVAL;
    }
    return GSORT_OK;
}

int radix_sort(const void *d_keys_in, void *d_keys_out, const uint32_t *d_vals_in,
               uint32_t *d_vals_out, int64_t n, int kind, int flags, int begin_bit, int end_bit,
               void *d_ws, size_t ws_bytes, cudaStream_t stream, const gsort_options *options) {
    const gsort_options *o = options ? options : &kDefaults;
    int rc = radix_args(d_keys_in, d_keys_out, d_vals_in, d_vals_out, n, kind, flags, begin_bit,
                        end_bit, o);
    if (rc != GSORT_OK || n == 0) return rc;
    const bool pairs = d_vals_in != nullptr;
    const int kb = key_kind_bytes(kind);
    if (d_ws == nullptr) return GSORT_EWORKSPACE;
    if (!aligned(d_ws, kWsAlign)) return GSORT_EALIGN;
    if (ws_bytes < radix_layout(static_cast<uint32_t>(n), pairs, kb).total) return GSORT_EWORKSPACE;
    const size_t kbytes = static_cast<size_t>(n) * kb, vbytes = static_cast<size_t>(n) * 4;
    if (ranges_overlap(d_ws, ws_bytes, d_keys_in, kbytes) ||
        ranges_overlap(d_ws, ws_bytes, d_keys_out, kbytes) ||
        (pairs && (ranges_overlap(d_ws, ws_bytes, d_vals_in, vbytes) ||
                   ranges_overlap(d_ws, ws_bytes, d_vals_out, vbytes))))
        return GSORT_EINVAL;
    if (begin_bit == end_bit) {   // no key bits: the stable order is the input order
        if (d_keys_out != d_keys_in &&
            cudaMemcpyAsync(d_keys_out, d_keys_in, kbytes, cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
            return GSORT_ECUDA;
        if (pairs && d_vals_out != d_vals_in &&
            cudaMemcpyAsync(d_vals_out, d_vals_in, vbytes, cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
            return GSORT_ECUDA;
        return GSORT_OK;
    }
    DeviceInfo dev;
    if (device_info(&dev) != GSORT_OK) return GSORT_ECUDA;
    RadixLaunch L;
    L.keys_in = d_keys_in;
    L.keys_out = d_keys_out;
    L.vals_in = d_vals_in;
    L.vals_out = d_vals_out;
    L.n = static_cast<uint32_t>(n);
    L.kind = kind;
    L.flags = flags;
    L.begin_bit = begin_bit;
    L.end_bit = end_bit;
    L.ws = static_cast<unsigned char *>(d_ws);
    L.spin_limit = o->spin_limit ? o->spin_limit : kDefaultSpinLimit;
    L.stall_tile = (o->stall_tile >= 0 && o->stall_tile < 0xFFFFFFFFll)
                       ? static_cast<uint32_t>(o->stall_tile) : kNoStall;
    L.events = reinterpret_cast<cudaEvent_t *>(o->events);
    L.num_events = o->num_events;
    L.variant = o->variant;
    L.stream = stream;
    L.sm_count = dev.sm_count;
    return launch_radix(L);
}

}  // namespace
}  // namespace gsort

using namespace gsort;

extern "C" {

const char *gsort_status_string(int status) {
    switch (status) {
        case GSORT_OK: return "GSORT_OK";
        case GSORT_EINVAL: return "GSORT_EINVAL: invalid argument";
        case GSORT_EALIGN: return "GSORT_EALIGN: misaligned pointer";
        case GSORT_EWORKSPACE: return "GSORT_EWORKSPACE: workspace missing or too small";
        case GSORT_ETOOBIG:
            return "GSORT_ETOOBIG: n (or the segment count) exceeds the entry point's maximum (GSORT_MAX_N; "
                   "GSORT_COMPACT_NOALLOC_MAX_N for the allocation-free compaction)";
        case GSORT_ECUDA: return "GSORT_ECUDA: CUDA error";
        case GSORT_ETIMEOUT: return "GSORT_ETIMEOUT: a device-side look-back wait gave up";
        default: return "unknown gsort status";
    }
}

int gsort_version(void) { return 100; }

size_t gsort_radix_workspace_bytes(int64_t n, int with_values) {
    if (n < 0 || n > GSORT_MAX_N) return 0;
    return radix_layout(static_cast<uint32_t>(n), with_values != 0, 4).total;
}

size_t gsort_radix_sort_workspace_bytes(int64_t n, int kind, int with_values) {
    const int kb = key_kind_bytes(kind);
    if (n < 0 || n > GSORT_MAX_N || kb == 0) return 0;
    return radix_layout(static_cast<uint32_t>(n), with_values != 0, kb).total;
}

int gsort_radix_sort_ex(const void *d_keys_in, void *d_keys_out, const uint32_t *d_vals_in,
                        uint32_t *d_vals_out, int64_t n, int kind, int flags, int begin_bit,
                        int end_bit, void *d_ws, size_t ws_bytes, cudaStream_t stream,
                        const gsort_options *options) {
    return radix_sort(d_keys_in, d_keys_out, d_vals_in, d_vals_out, n, kind, flags, begin_bit,
                      end_bit, d_ws, ws_bytes, stream, options);
}

int gsort_radix_sort(const void *d_keys_in, void *d_keys_out, const uint32_t *d_vals_in,
                     uint32_t *d_vals_out, int64_t n, int kind, int flags, int begin_bit,
                     int end_bit, void *d_ws, size_t ws_bytes, cudaStream_t stream) {
    return radix_sort(d_keys_in, d_keys_out, d_vals_in, d_vals_out, n, kind, flags, begin_bit,
                      end_bit, d_ws, ws_bytes, stream, nullptr);
}

int gsort_radix_pairs_ex(const void *d_keys_in, void *d_keys_out, const uint32_t *d_vals_in,
                         uint32_t *d_vals_out, int64_t n, int kind, int begin_bit, int end_bit,
                         void *d_ws, size_t ws_bytes, cudaStream_t stream,
                         const gsort_options *options) {
    if (key_kind_bytes(kind) != 4) return GSORT_EINVAL;   // 64-bit kinds: gsort_radix_sort
    return radix_sort(d_keys_in, d_keys_out, d_vals_in, d_vals_out, n, kind, 0, begin_bit, end_bit,
                      d_ws, ws_bytes, stream, options);
}

int gsort_radix_pairs(const void *d_keys_in, void *d_keys_out, const uint32_t *d_vals_in,
                      uint32_t *d_vals_out, int64_t n, int kind, int begin_bit, int end_bit,
                      void *d_ws, size_t ws_bytes, cudaStream_t stream) {
    return gsort_radix_pairs_ex(d_keys_in, d_keys_out, d_vals_in, d_vals_out, n, kind, begin_bit,
                                end_bit, d_ws, ws_bytes, stream, nullptr);
}

int gsort_radix_keys(const void *d_keys_in, void *d_keys_out, int64_t n, int kind, void *d_ws,
                     size_t ws_bytes, cudaStream_t stream) {
    return gsort_radix_pairs_ex(d_keys_in, d_keys_out, nullptr, nullptr, n, kind, 0, 32, d_ws,
                                ws_bytes, stream, nullptr);
}

int gsort_digit_histograms(const void *d_keys, int64_t n, int kind, int begin_bit, int end_bit,
                           uint32_t *d_hist_out, cudaStream_t stream) {
    if (n < 0) return GSORT_EINVAL;
    if (n > GSORT_MAX_N) return GSORT_ETOOBIG;
    const int kb = key_kind_bytes(kind);
    if (kb == 0) return GSORT_EINVAL;
    if (begin_bit < 0 || end_bit > 8 * kb || begin_bit > end_bit) return GSORT_EINVAL;
    if (begin_bit == end_bit) return GSORT_OK;
    if (d_hist_out == nullptr || (n > 0 && d_keys == nullptr)) return GSORT_EINVAL;
    if (!aligned(d_hist_out, 4) || (n > 0 && !aligned(d_keys, kb))) return GSORT_EALIGN;
    const int passes = (end_bit - begin_bit + 7) / 8;
    if (n > 0 && ranges_overlap(d_keys, static_cast<size_t>(n) * kb, d_hist_out,
                                static_cast<size_t>(passes) * 256 * 4))
        return GSORT_EINVAL;
    DeviceInfo dev;
    if (device_info(&dev) != GSORT_OK) return GSORT_ECUDA;
    return launch_digit_histograms(d_keys, static_cast<uint32_t>(n), kind, 0, begin_bit, end_bit,
                                   d_hist_out, stream, dev.sm_count);
}

size_t gsort_compact_workspace_bytes(int64_t n) {
    if (n < 0 || n > GSORT_MAX_N) return 0;
    return compact_layout(static_cast<uint32_t>(n)).total;
}

int gsort_compact_positive_ex(const float *d_in, float *d_out, int64_t n, int64_t *d_num_kept,
                              void *d_ws, size_t ws_bytes, cudaStream_t stream,
                              const gsort_options *options) {
    const gsort_options *o = options ? options : &kDefaults;
    if (n < 0) return GSORT_EINVAL;
    if (n > GSORT_MAX_N) return GSORT_ETOOBIG;
    if (o->num_events < 0 || (o->num_events > 0 && o->events == nullptr)) return GSORT_EINVAL;
    if (d_num_kept != nullptr && !aligned(d_num_kept, 8)) return GSORT_EALIGN;
    if (n > 0) {
        if (d_in == nullptr || d_out == nullptr) return GSORT_EINVAL;
        if (!aligned(d_in, 4) || !aligned(d_out, 4)) return GSORT_EALIGN;
        if (overlap(d_in, d_out, static_cast<size_t>(n) * 4)) return GSORT_EINVAL;
    }
    if (d_ws == nullptr) return GSORT_EWORKSPACE;
    if (!aligned(d_ws, kWsAlign)) return GSORT_EALIGN;
    const CompactLayout lay = compact_layout(static_cast<uint32_t>(n));
    if (ws_bytes < lay.total) return GSORT_EWORKSPACE;
    if (n > 0 && (ranges_overlap(d_ws, ws_bytes, d_in, static_cast<size_t>(n) * 4) ||
                  ranges_overlap(d_ws, ws_bytes, d_out, static_cast<size_t>(n) * 4)))
        return GSORT_EINVAL;
    if (n == 0) {
        if (d_num_kept != nullptr &&
            cudaMemsetAsync(d_num_kept, 0, sizeof(int64_t), stream) != cudaSuccess)
            return GSORT_ECUDA;
        return GSORT_OK;
    }
    DeviceInfo dev;
    if (device_info(&dev) != GSORT_OK) return GSORT_ECUDA;
    CompactLaunch L;
    L.in = reinterpret_cast<const uint32_t *>(d_in);
    L.out = reinterpret_cast<uint32_t *>(d_out);
    L.n = static_cast<uint32_t>(n);
    L.num_kept = d_num_kept;
    L.ws = static_cast<unsigned char *>(d_ws);
    L.spin_limit = o->spin_limit ? o->spin_limit : kDefaultSpinLimit;
    L.stall_tile = (o->stall_tile >= 0 && o->stall_tile < 0xFFFFFFFFll)
                       ? static_cast<uint32_t>(o->stall_tile) : kNoStall;
    L.events = reinterpret_cast<cudaEvent_t *>(o->events);
    L.num_events = o->num_events;
    L.stream = stream;
    L.sm_count = dev.sm_count;
    return launch_compact(L);
}

int gsort_compact_positive(const float *d_in, float *d_out, int64_t n, int64_t *d_num_kept,
                           void *d_ws, size_t ws_bytes, cudaStream_t stream) {
    return gsort_compact_positive_ex(d_in, d_out, n, d_num_kept, d_ws, ws_bytes, stream, nullptr);
}

int gsort_segmented_bitonic(uint32_t *d_keys, int64_t num_segments, int segment_len,
                            cudaStream_t stream) {
    if (num_segments < 0 || segment_len < 1 || segment_len > 1024) return GSORT_EINVAL;
    if (num_segments > 0x7FFFFFFFll) return GSORT_ETOOBIG;
    if (num_segments == 0 || segment_len == 1) return GSORT_OK;
    if (d_keys == nullptr) return GSORT_EINVAL;
    if (!aligned(d_keys, 4)) return GSORT_EALIGN;
    return launch_segmented_bitonic(d_keys, num_segments, segment_len, stream);
}

int gsort_check(const void *d_ws, cudaStream_t stream) {
    if (d_ws == nullptr) return GSORT_EINVAL;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GSORT_ECUDA;
    uint32_t status = 0;
    if (cudaMemcpy(&status, static_cast<const unsigned char *>(d_ws) + kHdrStatus, sizeof(status),
                   cudaMemcpyDeviceToHost) != cudaSuccess)
        return GSORT_ECUDA;
    return static_cast<int>(status);
}

size_t gsort_segmented_sort_workspace_bytes(int64_t n, int64_t num_segments, int with_values) {
    if (n < 0 || n > GSORT_MAX_N || num_segments < 0 || num_segments > GSORT_MAX_N) return 0;
    return seg_layout(static_cast<uint32_t>(n), static_cast<uint32_t>(num_segments), with_values != 0)
        .total;
}

int gsort_segmented_sort_ex(const void *d_keys_in, void *d_keys_out, const uint32_t *d_vals_in,
                            uint32_t *d_vals_out, int64_t n, const uint32_t *d_offsets,
                            int64_t num_segments, int kind, int flags, void *d_ws, size_t ws_bytes,
                            cudaStream_t stream, const gsort_options *options) {
    const gsort_options *o = options ? options : &kDefaults;
    if (n < 0 || num_segments < 0) return GSORT_EINVAL;
    if (n > GSORT_MAX_N || num_segments > GSORT_MAX_N) return GSORT_ETOOBIG;
    if (key_kind_bytes(kind) != 4) return GSORT_EINVAL;
    if ((flags & ~GSORT_DESCENDING) != 0) return GSORT_EINVAL;
    if ((d_vals_in == nullptr) != (d_vals_out == nullptr)) return GSORT_EINVAL;
    if (o->num_events < 0 || (o->num_events > 0 && o->events == nullptr)) return GSORT_EINVAL;
    if (n == 0) return GSORT_OK;
    if (num_segments == 0) return GSORT_EINVAL;   // n > 0 keys need at least one segment
    if (d_keys_in == nullptr || d_keys_out == nullptr || d_offsets == nullptr) return GSORT_EINVAL;
    if (!aligned(d_keys_in, 4) || !aligned(d_keys_out, 4) || !aligned(d_offsets, 4)) return GSORT_EALIGN;
    if (d_vals_in != nullptr && (!aligned(d_vals_in, 4) || !aligned(d_vals_out, 4))) return GSORT_EALIGN;
    const bool pairs = d_vals_in != nullptr;
    const size_t bytes = static_cast<size_t>(n) * 4;
    const size_t obytes = (static_cast<size_t>(num_segments) + 1) * 4;
    if (partial_overlap(d_keys_in, d_keys_out, bytes)) return GSORT_EINVAL;
    if (ranges_overlap(d_offsets, obytes, d_keys_out, bytes)) return GSORT_EINVAL;
    if (pairs) {
        if (partial_overlap(d_vals_in, d_vals_out, bytes)) return GSORT_EINVAL;
        if (overlap(d_keys_out, d_vals_out, bytes) || overlap(d_keys_in, d_vals_out, bytes) ||
            overlap(d_keys_out, d_vals_in, bytes) || ranges_overlap(d_offsets, obytes, d_vals_out, bytes))
            return GSORT_EINVAL;
    }
    if (d_ws == nullptr) return GSORT_EWORKSPACE;
    if (!aligned(d_ws, kWsAlign)) return GSORT_EALIGN;
    const SegLayout lay = seg_layout(static_cast<uint32_t>(n), static_cast<uint32_t>(num_segments), pairs);
    if (ws_bytes < lay.total) return GSORT_EWORKSPACE;
    if (ranges_overlap(d_ws, ws_bytes, d_keys_in, bytes) || ranges_overlap(d_ws, ws_bytes, d_keys_out, bytes) ||
        ranges_overlap(d_ws, ws_bytes, d_offsets, obytes) ||
        (pairs && (ranges_overlap(d_ws, ws_bytes, d_vals_in, bytes) ||
                   ranges_overlap(d_ws, ws_bytes, d_vals_out, bytes))))
        return GSORT_EINVAL;
    DeviceInfo dev;
    if (device_info(&dev) != GSORT_OK) return GSORT_ECUDA;
    SegLaunch L;
    L.keys_in = static_cast<const uint32_t *>(d_keys_in);
    L.keys_out = static_cast<uint32_t *>(d_keys_out);
    L.vals_in = d_vals_in;
    L.vals_out = d_vals_out;
    L.n = static_cast<uint32_t>(n);
    L.offsets = d_offsets;
    L.num_segments = static_cast<uint32_t>(num_segments);
    L.kind = kind;
    L.flags = flags;
    L.ws = static_cast<unsigned char *>(d_ws);
    L.spin_limit = o->spin_limit ? o->spin_limit : kDefaultSpinLimit;
    L.events = reinterpret_cast<cudaEvent_t *>(o->events);
    L.num_events = o->num_events;
    L.stream = stream;
    L.sm_count = dev.sm_count;
    return launch_segmented_sort(L);
}

int gsort_segmented_sort(const void *d_keys_in, void *d_keys_out, const uint32_t *d_vals_in,
                         uint32_t *d_vals_out, int64_t n, const uint32_t *d_offsets,
                         int64_t num_segments, int kind, int flags, void *d_ws, size_t ws_bytes,
                         cudaStream_t stream) {
    return gsort_segmented_sort_ex(d_keys_in, d_keys_out, d_vals_in, d_vals_out, n, d_offsets,
                                   num_segments, kind, flags, d_ws, ws_bytes, stream, nullptr);
}

size_t gsort_partition_workspace_bytes(int64_t n) {
    if (n < 0 || n > GSORT_MAX_N) return 0;
    return split_layout(static_cast<uint32_t>(n), false, false).total;
}

int gsort_partition(const uint32_t *d_in, uint32_t *d_out, const uint32_t *d_vals_in,
                    uint32_t *d_vals_out, int64_t n, int pred, int kind, uint32_t param,
                    const uint8_t *d_flags, int64_t *d_num_true, void *d_ws, size_t ws_bytes,
                    cudaStream_t stream) {
    if (n < 0) return GSORT_EINVAL;
    if (n > GSORT_MAX_N) return GSORT_ETOOBIG;
    if (pred < GSORT_PRED_FLAGS || pred > GSORT_PRED_POSITIVE) return GSORT_EINVAL;
    if ((pred == GSORT_PRED_BIT_SET || pred == GSORT_PRED_BIT_CLEAR) && param >= 32) return GSORT_EINVAL;
    if (pred == GSORT_PRED_LESS && key_kind_bytes(kind) != 4) return GSORT_EINVAL;
    if ((d_vals_in == nullptr) != (d_vals_out == nullptr)) return GSORT_EINVAL;
    if (d_num_true != nullptr && !aligned(d_num_true, 8)) return GSORT_EALIGN;
    const bool pairs = d_vals_in != nullptr;
    if (n > 0) {
        if (d_in == nullptr || d_out == nullptr) return GSORT_EINVAL;
        if (pred == GSORT_PRED_FLAGS && d_flags == nullptr) return GSORT_EINVAL;
        if (!aligned(d_in, 4) || !aligned(d_out, 4)) return GSORT_EALIGN;
        if (pairs && (!aligned(d_vals_in, 4) || !aligned(d_vals_out, 4))) return GSORT_EALIGN;
        const size_t bytes = static_cast<size_t>(n) * 4;
        if (overlap(d_in, d_out, bytes)) return GSORT_EINVAL;
        if (pairs && (overlap(d_vals_in, d_vals_out, bytes) || overlap(d_in, d_vals_out, bytes) ||
                      overlap(d_vals_in, d_out, bytes) || overlap(d_out, d_vals_out, bytes)))
            return GSORT_EINVAL;
        if (pred == GSORT_PRED_FLAGS &&
            (ranges_overlap(d_flags, static_cast<size_t>(n), d_out, bytes) ||
             (pairs && ranges_overlap(d_flags, static_cast<size_t>(n), d_vals_out, bytes))))
            return GSORT_EINVAL;
    }
    if (d_ws == nullptr) return GSORT_EWORKSPACE;
    if (!aligned(d_ws, kWsAlign)) return GSORT_EALIGN;
    const SplitLayout lay = split_layout(static_cast<uint32_t>(n), pairs, false);
    if (ws_bytes < lay.total) return GSORT_EWORKSPACE;
    if (n == 0) {
        if (d_num_true != nullptr && cudaMemsetAsync(d_num_true, 0, sizeof(int64_t), stream) != cudaSuccess)
            return GSORT_ECUDA;
        return GSORT_OK;
    }
    const size_t bytes = static_cast<size_t>(n) * 4;
    if (ranges_overlap(d_ws, ws_bytes, d_in, bytes) || ranges_overlap(d_ws, ws_bytes, d_out, bytes) ||
        (pairs && (ranges_overlap(d_ws, ws_bytes, d_vals_in, bytes) ||
                   ranges_overlap(d_ws, ws_bytes, d_vals_out, bytes))))
        return GSORT_EINVAL;
    DeviceInfo dev;
    if (device_info(&dev) != GSORT_OK) return GSORT_ECUDA;
    PartitionLaunch L;
    L.in = d_in;
    L.out = d_out;
    L.vals_in = d_vals_in;
    L.vals_out = d_vals_out;
    L.n = static_cast<uint32_t>(n);
    L.pred = pred;
    L.kind = kind;
    L.param = param;
    L.flags = d_flags;
    L.num_true = d_num_true;
    L.ws = static_cast<unsigned char *>(d_ws);
    L.spin_limit = kDefaultSpinLimit;
    L.stream = stream;
    L.sm_count = dev.sm_count;
    return launch_partition(L);
}

size_t gsort_split_sort_workspace_bytes(int64_t n, int with_values) {
    if (n < 0 || n > GSORT_MAX_N) return 0;
    return split_layout(static_cast<uint32_t>(n), with_values != 0, true).total;
}

int gsort_split_sort(const uint32_t *d_keys_in, uint32_t *d_keys_out, const uint32_t *d_vals_in,
                     uint32_t *d_vals_out, int64_t n, int begin_bit, int end_bit, void *d_ws,
                     size_t ws_bytes, cudaStream_t stream) {
    int rc = radix_args(d_keys_in, d_keys_out, d_vals_in, d_vals_out, n, GSORT_KEY_U32, 0, begin_bit,
                        end_bit, &kDefaults);
    if (rc != GSORT_OK || n == 0) return rc;
    const bool pairs = d_vals_in != nullptr;
    if (d_ws == nullptr) return GSORT_EWORKSPACE;
    if (!aligned(d_ws, kWsAlign)) return GSORT_EALIGN;
    if (ws_bytes < split_layout(static_cast<uint32_t>(n), pairs, true).total) return GSORT_EWORKSPACE;
    const size_t bytes = static_cast<size_t>(n) * 4;
    if (ranges_overlap(d_ws, ws_bytes, d_keys_in, bytes) || ranges_overlap(d_ws, ws_bytes, d_keys_out, bytes) ||
        (pairs && (ranges_overlap(d_ws, ws_bytes, d_vals_in, bytes) ||
                   ranges_overlap(d_ws, ws_bytes, d_vals_out, bytes))))
        return GSORT_EINVAL;
    if (begin_bit == end_bit) {
        if (d_keys_out != d_keys_in &&
            cudaMemcpyAsync(d_keys_out, d_keys_in, bytes, cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
            return GSORT_ECUDA;
        if (pairs && d_vals_out != d_vals_in &&
            cudaMemcpyAsync(d_vals_out, d_vals_in, bytes, cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
            return GSORT_ECUDA;
        return GSORT_OK;
    }
    DeviceInfo dev;
    if (device_info(&dev) != GSORT_OK) return GSORT_ECUDA;
    SplitSortLaunch L;
    L.keys_in = d_keys_in;
    L.keys_out = d_keys_out;
    L.vals_in = d_vals_in;
    L.vals_out = d_vals_out;
    L.n = static_cast<uint32_t>(n);
    L.begin_bit = begin_bit;
    L.end_bit = end_bit;
    L.ws = static_cast<unsigned char *>(d_ws);
    L.spin_limit = kDefaultSpinLimit;
    L.stream = stream;
    L.sm_count = dev.sm_count;
    return launch_split_sort(L);
}

int gsort_radix_num_variants(void) { return radix_num_variants(); }

const char *gsort_radix_variant_name(int variant) { return radix_variant_name(variant); }

int gsort_radix_launch_count(int64_t n, int begin_bit, int end_bit, int in_place) {
    return gsort_radix_sort_launch_count(n, GSORT_KEY_U32, begin_bit, end_bit, in_place);
}

int gsort_radix_sort_launch_count(int64_t n, int kind, int begin_bit, int end_bit, int in_place) {
    const int kb = key_kind_bytes(kind);
    if (n <= 0 || begin_bit >= end_bit || kb == 0) return 0;
    if (kb == 4 && n <= 65536)
        return 1;   // one cluster kernel for every pass (where such a cluster fits the device)
    if (n <= GSORT_MAX_N && small_sort_applies(static_cast<uint32_t>(n), kb, 0))
        return 2;   // header clear + one cooperative kernel for every pass
    const int passes = (end_bit - begin_bit + 7) / 8;
    // header clear, histogram, the passes [, the copy back of an odd pass
    // count in place] [, the 64-bit histogram clear]
    return 2 + passes + ((in_place && (passes & 1)) ? 1 : 0) + (kb == 8 ? 1 : 0);
}

}  // extern "C"

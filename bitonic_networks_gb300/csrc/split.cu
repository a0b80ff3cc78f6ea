// split.cu -- stable 2-way split (partition) by a predicate, and the 1-bit
// split LSD radix sort built on it ([CUDA3] "Radix Sort": per bit, a
// predicate (is the bit 0), an exclusive scan of it and a scatter of the
// zeros before the ones; the pages run three kernels per bit).
//
// A split moves every element whose predicate holds, in input order, to
// out[0 .. m), and every other element, in input order, to out[m .. n).  m
// is counted before the split: for the sort, one upfront histogram read
// gives the zero count of every bit at once (a bit's count does not change
// when the keys move); for a partition, one counting read.  The split itself
// is one kernel per pass: each tile evaluates the predicate, scans the
// per-thread counts, finds the true count of all earlier tiles with a
// warp-wide decoupled look-back, stages its true and false elements as two
// runs in shared memory and writes both runs out (the pages' "dense output"
// staging).  Traffic per pass: read 4 B and write 4 B per element (+ 4 + 4
// for a value).
#include <algorithm>

#include "lookback.cuh"
#include "radix_kernels.cuh"

namespace gsort {
namespace {

constexpr int kSplitThreads = 512;
constexpr int kSplitItems = 16;                // per thread, a multiple of 4
constexpr uint32_t kSplitTile = kSplitThreads * kSplitItems;
constexpr uint32_t kSplitStride = 32;          // state words one 128-byte line apart
constexpr size_t kHdrSplitTrue = kHdrKept;     // u32 [0] true count (partition)
constexpr size_t kHdrSplitZeros = kHdrHist + 4096;   // u32 [32] zero count per bit (sort)
constexpr size_t kHdrSplitCounters = kHdrSplitZeros + 1024;   // u32 [32] tile counter per bit pass (sort)
static_assert(kHdrSplitCounters + 32 * 4 <= kHdrBytes, "split counters outside the header");

// ------------------------------------------------------------- predicates
// test(x, g): the predicate of element g (global index) whose word is x.
struct PredFlags {          // flags[g] != 0
    const uint8_t *flags;
    __device__ bool test(uint32_t, uint32_t g) const { return flags[g] != 0; }
};
struct PredBit {            // bit `bit` of the word equals `want`
    uint32_t bit, want;
    __device__ bool test(uint32_t x, uint32_t) const { return ((x >> bit) & 1u) == want; }
};
struct PredLess {           // order_in(x) < order_in(pivot), the sort order of a 32-bit kind
    uint32_t fmask, flip, pivot;   // pivot already mapped
    __device__ bool test(uint32_t x, uint32_t) const { return order_in<uint32_t>(x, fmask, flip) < pivot; }
};
struct PredPositive {       // IEEE x > 0 on the bit pattern (0 < bits <= 0x7F800000)
    __device__ bool test(uint32_t x, uint32_t) const { return (x - 1u) < 0x7F800000u; }
};

// --------------------------------------------------------------- counting
// Grid-stride count of the elements whose predicate holds: 16-byte loads,
// four in flight per thread (a flags predicate reads 4 flag bytes per group
// of 4 elements instead of the words).  vec: the source is suitably aligned
// (16 bytes for words, 4 for flags); otherwise one element at a time.
template <class Pred> struct PredReadsFlags { static constexpr bool value = false; };
template <> struct PredReadsFlags<PredFlags> { static constexpr bool value = true; };

template <class Pred>
__device__ __forceinline__ uint32_t count_group(const uint32_t *in, const Pred &pred, uint32_t g) {
    // elements g .. g+3
    if constexpr (PredReadsFlags<Pred>::value) {
        const uint32_t f = *reinterpret_cast<const uint32_t *>(pred.flags + g);
        return ((f & 0xFFu) != 0) + ((f & 0xFF00u) != 0) + ((f & 0xFF0000u) != 0) + ((f >> 24) != 0);
    } else {
        const uint4 q = __ldcs(reinterpret_cast<const uint4 *>(in + g));
        return pred.test(q.x, g) + pred.test(q.y, g + 1) + pred.test(q.z, g + 2) + pred.test(q.w, g + 3);
    }
}

template <class Pred>
__global__ void __launch_bounds__(256)
k_count_true(const uint32_t *__restrict__ in, uint32_t n, Pred pred, uint32_t *total, int vec) {
    constexpr int U = 4;
    __shared__ uint32_t s_w[8];
    const uint32_t gtid = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t gstride = gridDim.x * blockDim.x;
    uint32_t c = 0;
    const uint32_t groups = vec ? n / 4 : 0;
    for (uint32_t q = gtid; q < groups; q += U * gstride) {
        uint32_t part[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t qq = q + u * gstride;
            part[u] = qq < groups ? count_group(in, pred, 4 * qq) : 0u;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) c += part[u];
    }
    for (uint32_t i = 4 * groups + gtid; i < n; i += gstride)   // the tail, or everything when !vec
        c += pred.test(PredReadsFlags<Pred>::value ? 0u : in[i], i) ? 1u : 0u;
    c = __reduce_add_sync(kFullMask, c);
    if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = 0;
        for (int w = 0; w < 8; ++w) t += s_w[w];
        if (t) atomicAdd(total, t);
    }
}

// Zero count of every bit from the 4 x 256 byte histograms of the keys.
__global__ void k_bit_zeros(const uint32_t *hist, uint32_t *zeros) {
    const uint32_t b = threadIdx.x;   // 32 threads, one bit each
    const uint32_t *h = hist + (b >> 3) * 256;
    uint32_t z = 0;
    for (uint32_t v = 0; v < 256; ++v)
        if (((v >> (b & 7)) & 1u) == 0) z += h[v];
    zeros[b] = z;
}

// ----------------------------------------------------------------- split
template <class Pred, bool PAIRS>
__global__ void __launch_bounds__(kSplitThreads, PAIRS ? 2 : 3)
k_split(const uint32_t *__restrict__ in, const uint32_t *__restrict__ vin, uint32_t *__restrict__ out,
        uint32_t *__restrict__ vout, uint32_t n, Pred pred, const uint32_t *num_true,
        uint32_t *states, uint32_t *states_clear, uint32_t *tile_counter, uint32_t *status,
        uint32_t *abort_flag, uint32_t spin_limit, uint32_t stall_tile, int vec_ok) {
    constexpr int T = kSplitThreads, IPT = kSplitItems, WARPS = T / 32;
    constexpr uint32_t TILE = kSplitTile;
    extern __shared__ __align__(128) uint32_t smem[];
    uint32_t *s_buf = smem;                    // [TILE] true run, then false run
    uint32_t *s_vbuf = smem + TILE;            // [TILE] their values (pairs)
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
    if (states_clear != nullptr && tid == 0) states_clear[tile * kSplitStride] = 0;

    // blocked arrangement: thread t owns items [t*IPT, t*IPT + IPT) of the tile
    uint32_t x[IPT], v[PAIRS ? IPT : 1];
    const uint32_t first = tid * IPT;
    if (tile_n == TILE && vec_ok) {
        const uint4 *src = reinterpret_cast<const uint4 *>(in + base + first);
        const uint4 *vsrc = reinterpret_cast<const uint4 *>(vin + base + first);
#pragma unroll
        for (int q = 0; q < IPT / 4; ++q) {
            const uint4 a = __ldcs(src + q);
            x[4 * q + 0] = a.x;
            x[4 * q + 1] = a.y;
            x[4 * q + 2] = a.z;
            x[4 * q + 3] = a.w;
            if (PAIRS) {
                const uint4 b = __ldcs(vsrc + q);
                v[4 * q + 0] = b.x;
                v[4 * q + 1] = b.y;
                v[4 * q + 2] = b.z;
                v[4 * q + 3] = b.w;
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < IPT; ++j) {
            const bool in_range = first + j < tile_n;
            x[j] = in_range ? in[base + first + j] : 0u;
            if (PAIRS) v[j] = in_range ? vin[base + first + j] : 0u;
        }
    }
    uint32_t flags = 0;
#pragma unroll
    for (int j = 0; j < IPT; ++j)
        if (first + j < tile_n && pred.test(x[j], base + first + j)) flags |= 1u << j;
    const uint32_t cnt = __popc(flags);

    // block exclusive scan of the per-thread true counts (one barrier)
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
    uint32_t pos_t = warp_excl + incl - cnt;            // true items before this thread's
    uint32_t pos_f = total + min(first, tile_n) - pos_t;   // false run follows the true run

    if (warp == 0) {
        bool ok;
        const uint32_t prefix = warp_look_back(states, kSplitStride, tile, total, stall_tile,
                                               spin_limit, abort_flag, ok);
        if (lane == 0) {
            s_misc[1] = ok ? 0u : 1u;
            s_misc[3] = prefix;
            if (!ok) record_error(status, abort_flag, GSORT_ETIMEOUT);
        }
    }

    // stage both runs (overlaps warp 0's look-back)
#pragma unroll
    for (int j = 0; j < IPT; ++j) {
        if (first + j < tile_n) {
            const uint32_t slot = ((flags >> j) & 1u) ? pos_t++ : pos_f++;
            s_buf[slot] = x[j];
            if (PAIRS) s_vbuf[slot] = v[j];
        }
    }
    __syncthreads();
    if (s_misc[1] || tile == stall_tile) return;
    const uint32_t prefix = s_misc[3];                 // true items in earlier tiles
    const uint32_t m = *num_true;                      // true items in all tiles
    // slot i < total goes to prefix + i; slot i >= total to m + (falses before the tile) + (i - total)
    const uint32_t false_base = m + (base - prefix) - total;
    for (uint32_t i = tid; i < tile_n; i += T) {
        const uint32_t g = (i < total) ? prefix + i : false_base + i;
        if (g < n) {
            out[g] = s_buf[i];
            if (PAIRS) vout[g] = s_vbuf[i];
        }
    }
}

template <class Pred, bool PAIRS>
cudaError_t launch_split_kernel(const uint32_t *in, const uint32_t *vin, uint32_t *out, uint32_t *vout,
                                uint32_t n, const Pred &pred, const uint32_t *num_true,
                                uint32_t *states, uint32_t *states_clear, uint32_t *counter,
                                uint32_t *status, uint32_t *abort_flag, uint32_t spin_limit,
                                uint32_t stall_tile, cudaStream_t s) {
    const uint32_t tiles = (n + kSplitTile - 1) / kSplitTile;
    const int vec_ok = (reinterpret_cast<uintptr_t>(in) & 15) == 0 &&
                       (!PAIRS || (reinterpret_cast<uintptr_t>(vin) & 15) == 0);
    const size_t smem = static_cast<size_t>(kSplitTile) * (PAIRS ? 2 : 1) * sizeof(uint32_t);
    auto k = k_split<Pred, PAIRS>;
    cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(k), smem);
    if (e != cudaSuccess) return e;
    k<<<tiles, kSplitThreads, smem, s>>>(in, vin, out, vout, n, pred, num_true, states, states_clear,
                                         counter, status, abort_flag, spin_limit, stall_tile, vec_ok);
    return cudaGetLastError();
}

template <class Pred>
cudaError_t launch_split_any(bool pairs, const uint32_t *in, const uint32_t *vin, uint32_t *out,
                             uint32_t *vout, uint32_t n, const Pred &pred, const uint32_t *num_true,
                             uint32_t *states, uint32_t *states_clear, uint32_t *counter,
                             uint32_t *status, uint32_t *abort_flag, uint32_t spin_limit,
                             uint32_t stall_tile, cudaStream_t s) {
    return pairs ? launch_split_kernel<Pred, true>(in, vin, out, vout, n, pred, num_true, states,
                                                   states_clear, counter, status, abort_flag,
                                                   spin_limit, stall_tile, s)
                 : launch_split_kernel<Pred, false>(in, vin, out, vout, n, pred, num_true, states,
                                                    states_clear, counter, status, abort_flag,
                                                    spin_limit, stall_tile, s);
}

template <class Pred>
cudaError_t launch_count(const uint32_t *in, uint32_t n, const Pred &pred, uint32_t *total,
                         int sm_count, cudaStream_t s) {
    int vec;
    if constexpr (PredReadsFlags<Pred>::value) vec = (reinterpret_cast<uintptr_t>(pred.flags) & 3) == 0;
    else vec = (reinterpret_cast<uintptr_t>(in) & 15) == 0;
    const uint32_t grid = std::max(1u, std::min((n / 4 + 255) / 256, static_cast<uint32_t>(sm_count) * 8));
    k_count_true<Pred><<<grid, 256, 0, s>>>(in, n, pred, total, vec);
    return cudaGetLastError();
}

__global__ void k_store_count(const uint32_t *total, int64_t *num_true) {
    *num_true = static_cast<int64_t>(*total);
}

}  // namespace

SplitLayout split_layout(uint32_t n, bool with_values, bool sort) {
    SplitLayout L{};
    L.tiles = (n + kSplitTile - 1) / kSplitTile;
    size_t off = kHdrBytes;
    const size_t region = align_up(static_cast<size_t>(std::max(L.tiles, 1u)) * kSplitStride * 4, kWsAlign);
    L.states_a = off;
    off += region;
    L.states_b = off;
    if (sort) off += region;
    L.tmp_keys = off;
    if (sort) off += align_up(static_cast<size_t>(n) * 4, kWsAlign);
    L.tmp_vals = off;
    if (sort && with_values) off += align_up(static_cast<size_t>(n) * 4, kWsAlign);
    L.total = off;
    return L;
}

int launch_partition(const PartitionLaunch &L) {
    const SplitLayout lay = split_layout(L.n, L.vals_in != nullptr, false);
    cudaStream_t s = L.stream;
    unsigned char *ws = L.ws;
    uint32_t *status = reinterpret_cast<uint32_t *>(ws + kHdrStatus);
    uint32_t *abort_flag = reinterpret_cast<uint32_t *>(ws + kHdrAbort);
    uint32_t *counter = reinterpret_cast<uint32_t *>(ws + kHdrCounters);
    uint32_t *num_true = reinterpret_cast<uint32_t *>(ws + kHdrSplitTrue);
    uint32_t *states = reinterpret_cast<uint32_t *>(ws + lay.states_a);
    const bool pairs = L.vals_in != nullptr;
    const uint32_t init_words = static_cast<uint32_t>((lay.states_a + static_cast<size_t>(lay.tiles) * kSplitStride * 4) / 4);
    const uint32_t init_grid = std::max(1u, std::min<uint32_t>((init_words + 1023) / 1024, 4u * L.sm_count));
    k_zero_words<<<init_grid, 256, 0, s>>>(reinterpret_cast<uint32_t *>(ws), init_words);
    if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
    cudaError_t e = cudaSuccess;
    switch (L.pred) {
        case GSORT_PRED_FLAGS: {
            const PredFlags p{L.flags};
            e = launch_count(L.in, L.n, p, num_true, L.sm_count, s);
            if (e == cudaSuccess)
                e = launch_split_any(pairs, L.in, L.vals_in, L.out, L.vals_out, L.n, p, num_true, states,
                                     nullptr, counter, status, abort_flag, L.spin_limit, kNoStall, s);
            break;
        }
        case GSORT_PRED_BIT_SET:
        case GSORT_PRED_BIT_CLEAR: {
            const PredBit p{L.param, L.pred == GSORT_PRED_BIT_SET ? 1u : 0u};
            e = launch_count(L.in, L.n, p, num_true, L.sm_count, s);
            if (e == cudaSuccess)
                e = launch_split_any(pairs, L.in, L.vals_in, L.out, L.vals_out, L.n, p, num_true, states,
                                     nullptr, counter, status, abort_flag, L.spin_limit, kNoStall, s);
            break;
        }
        case GSORT_PRED_LESS: {
            const KeyOrder o = key_order(L.kind, 0);
            const uint32_t fm = static_cast<uint32_t>(o.fmask), fl = static_cast<uint32_t>(o.flip);
            // the pivot through the same map, on the host
            uint32_t pv = L.param;
            if (fm) pv ^= (pv >> 31) ? 0xFFFFFFFFu : 0x80000000u;
            pv ^= fl;
            const PredLess p{fm, fl, pv};
            e = launch_count(L.in, L.n, p, num_true, L.sm_count, s);
            if (e == cudaSuccess)
                e = launch_split_any(pairs, L.in, L.vals_in, L.out, L.vals_out, L.n, p, num_true, states,
                                     nullptr, counter, status, abort_flag, L.spin_limit, kNoStall, s);
            break;
        }
        default: {   // GSORT_PRED_POSITIVE_F32
            const PredPositive p{};
            e = launch_count(L.in, L.n, p, num_true, L.sm_count, s);
            if (e == cudaSuccess)
                e = launch_split_any(pairs, L.in, L.vals_in, L.out, L.vals_out, L.n, p, num_true, states,
                                     nullptr, counter, status, abort_flag, L.spin_limit, kNoStall, s);
            break;
        }
    }
    if (e != cudaSuccess) return GSORT_ECUDA;
    if (L.num_true != nullptr) {
        k_store_count<<<1, 1, 0, s>>>(num_true, L.num_true);
        if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
    }
    return GSORT_OK;
}

int launch_split_sort(const SplitSortLaunch &L) {
    const bool pairs = L.vals_in != nullptr;
    const SplitLayout lay = split_layout(L.n, pairs, true);
    cudaStream_t s = L.stream;
    unsigned char *ws = L.ws;
    uint32_t *status = reinterpret_cast<uint32_t *>(ws + kHdrStatus);
    uint32_t *abort_flag = reinterpret_cast<uint32_t *>(ws + kHdrAbort);
    uint32_t *hist = reinterpret_cast<uint32_t *>(ws + kHdrHist);
    uint32_t *zeros = reinterpret_cast<uint32_t *>(ws + kHdrSplitZeros);
    uint32_t *states[2] = {reinterpret_cast<uint32_t *>(ws + lay.states_a),
                           reinterpret_cast<uint32_t *>(ws + lay.states_b)};
    uint32_t *tmp_k = reinterpret_cast<uint32_t *>(ws + lay.tmp_keys);
    uint32_t *tmp_v = pairs ? reinterpret_cast<uint32_t *>(ws + lay.tmp_vals) : nullptr;
    const int bits = L.end_bit - L.begin_bit;

    // header and the first pass's states cleared; later passes clear their
    // successor's states tile by tile
    const uint32_t init_words = static_cast<uint32_t>((lay.states_a + static_cast<size_t>(lay.tiles) * kSplitStride * 4) / 4);
    const uint32_t init_grid = std::max(1u, std::min<uint32_t>((init_words + 1023) / 1024, 4u * L.sm_count));
    k_zero_words<<<init_grid, 256, 0, s>>>(reinterpret_cast<uint32_t *>(ws), init_words);
    if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
    if (launch_hist_kernel<uint32_t>(L.keys_in, L.n, false, 0u, 0u, 0, 4, 0xFFu, hist, nullptr, 0, s,
                                     L.sm_count) != cudaSuccess)
        return GSORT_ECUDA;
    k_bit_zeros<<<1, 32, 0, s>>>(hist, zeros);
    if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;

    // in -> tmp -> out -> tmp ...; an odd bit count ends in tmp and is copied
    // back.  Even counts end in out; in place works the same way.
    const uint32_t *src_k = L.keys_in;
    const uint32_t *src_v = L.vals_in;
    uint32_t *dst_k = nullptr, *dst_v = nullptr;
    for (int p = 0; p < bits; ++p) {
        dst_k = (p % 2 == 0) ? tmp_k : L.keys_out;
        dst_v = pairs ? ((p % 2 == 0) ? tmp_v : L.vals_out) : nullptr;
        const uint32_t b = static_cast<uint32_t>(L.begin_bit + p);
        const PredBit pred{b, 0u};   // zeros first
        uint32_t *counter = reinterpret_cast<uint32_t *>(ws + kHdrSplitCounters) + p;
        if (launch_split_any(pairs, src_k, src_v, dst_k, dst_v, L.n, pred, zeros + b, states[p & 1],
                             (p + 1 < bits) ? states[(p + 1) & 1] : nullptr, counter, status,
                             abort_flag, L.spin_limit, kNoStall, s) != cudaSuccess)
            return GSORT_ECUDA;
        src_k = dst_k;
        src_v = dst_v;
    }
    if (dst_k != L.keys_out) {
        if (cudaMemcpyAsync(L.keys_out, dst_k, static_cast<size_t>(L.n) * 4, cudaMemcpyDeviceToDevice, s) !=
            cudaSuccess)
            return GSORT_ECUDA;
        if (pairs && cudaMemcpyAsync(L.vals_out, dst_v, static_cast<size_t>(L.n) * 4,
                                     cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return GSORT_ECUDA;
    }
    return GSORT_OK;
}

}  // namespace gsort

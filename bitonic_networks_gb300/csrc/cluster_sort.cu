// cluster_sort.cu -- the whole LSD radix sort of a small input (up to 65,536
// 32-bit keys) inside one thread-block cluster, with the keys resident in the
// CTAs' shared memory between passes.
//
// CTA r of the cluster holds keys [r * TC, (r + 1) * TC) of the current
// order (TC keys per CTA).  Per digit pass ([CUDA3] several bits at once;
// [PMPP10] 10.3):
//   each CTA counts its keys' digits (per-warp tables) and publishes the 256
//   counts in its shared memory; cluster barrier;
//   every CTA reads the counts of all CTAs through distributed shared memory
//   and forms, per digit, the bin start (exclusive scan of the digit totals,
//   [CUDA3] kernel 2) plus the count in lower-ranked CTAs -- the complete
//   prefix, so no look-back is needed;
//   each CTA ranks its keys stably with the warp multisplit, reorders them in
//   its own shared memory ([PMPP10] 10.4), and writes each key (and value) to
//   its place in the next pass's distribution: word g % TC of CTA g / TC,
//   through distributed shared memory (the global output after the last
//   pass); cluster barrier.
// So a sort is one launch with 2 cluster barriers per pass (hardware
// barriers: no waits in software, no grid barrier, no round trip through L2)
// and one read and one write of global memory.  The kernel clears the
// status words itself, so no header-clear launch precedes it.
#include <cooperative_groups.h>

#include <mutex>

#include "radix_kernels.cuh"

namespace gsort {
namespace {

namespace cg = cooperative_groups;

constexpr int kClusterThreads = 512;
constexpr int kClusterWarps = kClusterThreads / 32;
constexpr int kClusterIpt = 8;                    // 4096 keys per CTA
constexpr uint32_t kClusterSortMaxN = 1u << 16;   // 16 CTAs

struct ClusterSortArgs {
    const uint32_t *keys_in;
    uint32_t *keys_out;
    const uint32_t *vals_in;   // null: keys only
    uint32_t *vals_out;
    uint32_t n;
    int passes;
    uint32_t begin_bit, last_mask;
    uint32_t fmask, flip;
    int alias;                 // keys or values sorted in place
    uint32_t *status, *abort_flag;
};

template <int IPT, bool PAIRS>
constexpr size_t cluster_smem_words() {
    // two key buffers [+ two value buffers], per-warp counts, tile counts,
    // per-digit global offsets, misc
    return static_cast<size_t>(kClusterThreads) * IPT * (PAIRS ? 4 : 2) + kClusterWarps * kRow + 256 + 256 + 32;
}

template <int IPT, bool PAIRS>
__global__ void __launch_bounds__(kClusterThreads, 1) k_cluster_sort(const ClusterSortArgs a) {
    constexpr int T = kClusterThreads, WARPS = kClusterWarps;
    constexpr uint32_t TC = T * IPT;   // keys per CTA
    extern __shared__ __align__(128) uint32_t smem[];
    uint32_t *const buf_k0 = smem;
    uint32_t *const buf_k1 = smem + TC;
    uint32_t *const buf_v0 = smem + 2 * TC;   // pairs only
    uint32_t *const buf_v1 = smem + 3 * TC;
    uint32_t *const s_cnt = smem + TC * (PAIRS ? 4 : 2);   // [WARPS][256] counts, then next free slots
    uint32_t *const s_tc = s_cnt + WARPS * kRow;           // [256] this CTA's digit counts (read by all)
    uint32_t *const s_goff = s_tc + 256;                   // [256] global index - tile slot
    uint32_t *const s_misc = s_goff + 256;                 // [32]

    cg::cluster_group cluster = cg::this_cluster();
    const uint32_t rank = cluster.block_rank(), csize = cluster.num_blocks();
    const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t base = rank * TC;
    const uint32_t tile_n = base < a.n ? min(TC, a.n - base) : 0u;
    const uint32_t item0 = warp * (32 * IPT) + lane;   // item k at item0 + 32k (warp-contiguous runs)
    if (rank == 0 && tid == 0) {   // this path has no header-clear launch
        *a.status = 0u;
        *a.abort_flag = 0u;
    }

    for (int p = 0; p < a.passes; ++p) {
        const bool first = p == 0, last = p == a.passes - 1;
        const uint32_t shift = a.begin_bit + 8 * p;
        const uint32_t mask = last ? a.last_mask : 0xFFu;
        uint32_t *cur_k = (p & 1) ? buf_k1 : buf_k0;
        uint32_t *nxt_k = (p & 1) ? buf_k0 : buf_k1;
        uint32_t *cur_v = (p & 1) ? buf_v1 : buf_v0;
        uint32_t *nxt_v = (p & 1) ? buf_v0 : buf_v1;

        // ---- this CTA's keys into registers
        uint32_t key[IPT], val[PAIRS ? IPT : 1];
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            const uint32_t i = item0 + 32 * k;
            const bool ok = i < tile_n;
            if (first) {
                key[k] = ok ? order_in<uint32_t>(a.keys_in[base + i], a.fmask, a.flip) : 0u;
                if (PAIRS) val[k] = ok ? a.vals_in[base + i] : 0u;
            } else {
                key[k] = ok ? cur_k[i] : 0u;
                if (PAIRS) val[k] = ok ? cur_v[i] : 0u;
            }
        }
        // one pass in place: nobody writes the output before every CTA has read its input
        if (first && last && a.alias) cluster.sync();
        for (uint32_t i = tid; i < WARPS * kRow; i += T) s_cnt[i] = 0;
        __syncthreads();
        {
            uint32_t *wc = s_cnt + warp * kRow;
#pragma unroll
            for (int k = 0; k < IPT; ++k)
                if (item0 + 32 * k < tile_n) atomicAdd(&wc[digit_at<false>(key[k], shift, mask)], 1u);
        }
        __syncthreads();
        uint32_t cnt = 0;
        if (tid < 256) {
#pragma unroll
            for (int w = 0; w < WARPS; ++w) {
                const uint32_t cw = s_cnt[w * kRow + tid];
                s_cnt[w * kRow + tid] = cnt;   // exclusive over warps
                cnt += cw;
            }
            s_tc[tid] = cnt;
        }
        cluster.sync();   // every CTA's counts are visible to the whole cluster

        // ---- per digit: bin start + count in lower-ranked CTAs; tile offsets
        if (tid < 256) {
            // every CTA's count of digit tid, all 16 loads in flight at once
            uint32_t c[16];
#pragma unroll
            for (uint32_t r = 0; r < 16; ++r) c[r] = r < csize ? cluster.map_shared_rank(s_tc, r)[tid] : 0u;
            uint32_t before = 0, total = 0;
#pragma unroll
            for (uint32_t r = 0; r < 16; ++r) {
                total += c[r];
                before += r < rank ? c[r] : 0u;
            }
            const uint32_t it = warp_inclusive_scan(total, lane);
            const uint32_t ic = warp_inclusive_scan(cnt, lane);
            // the largest digit total of this warp's 32 digits, and that digit
            const uint32_t wmax = __reduce_max_sync(kFullMask, total);
            const uint32_t at = __ffs(__ballot_sync(kFullMask, total == wmax)) - 1;
            if (lane == 31) {
                s_misc[4 + warp] = it;
                s_misc[12 + warp] = ic;
            }
            if (lane == 0) s_misc[20 + warp] = (wmax << 8) | (warp * 32 + at);   // totals < 2^17
            s_goff[tid] = it - total + before;
            cnt = ic - cnt;   // now: the exclusive scan of this tile's counts (within the warp)
        }
        __syncthreads();
        if (tid < 256) {
            uint32_t bt = 0, bc = 0;
            for (uint32_t w = 0; w < warp; ++w) {
                bt += s_misc[4 + w];
                bc += s_misc[12 + w];
            }
            const uint32_t tex = cnt + bc;
            s_goff[tid] += bt - tex;   // global index of tile slot i holding digit d: s_goff[d] + i
#pragma unroll
            for (int w = 0; w < WARPS; ++w) s_cnt[w * kRow + tid] += tex;
        }
        __syncthreads();

        // ---- the slot of each key in the tile-sorted order; the keys are in
        // registers, so the input buffer is free.  First pass of a keys-only
        // sort over every bit: keys of one digit may take any order, so each
        // takes the next free slot of its digit in its warp's range with one
        // shared atomic (one per warp for a warp whose keys share one digit,
        // and warp-aggregated for a digit that holds over 1/8 of the keys);
        // otherwise the stable warp multisplit.
        if (!PAIRS && first && a.begin_bit == 0 && a.passes == 4 && a.last_mask == 0xFFu) {
            uint32_t hot = 256u, hmax = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const uint32_t m = s_misc[20 + w];
                if ((m >> 8) > hmax) {
                    hmax = m >> 8;
                    hot = m & 0xFFu;
                }
            }
            if (hmax <= a.n / 8) hot = 256u;
            uint32_t *wc = s_cnt + warp * kRow;
            bool same = true;
            const uint32_t d0 = __shfl_sync(kFullMask, digit_at<false>(key[0], shift, mask), 0);
#pragma unroll
            for (int k = 0; k < IPT; ++k)
                same &= item0 + 32 * k < tile_n && digit_at<false>(key[k], shift, mask) == d0;
            const bool one_digit = __all_sync(kFullMask, same);
            if (hot < 256u && !one_digit) {
                // keys of other digits take their slots; the warp counts its
                // keys of the hot digit, reserves their slots with one atomic,
                // then places them
                const uint32_t ltm = lanemask_lt();
                uint32_t run = 0;
#pragma unroll
                for (int k = 0; k < IPT; ++k) {
                    const bool valid = item0 + 32 * k < tile_n;
                    const uint32_t d = digit_at<false>(key[k], shift, mask);
                    const bool h = valid && d == hot;
                    run += __popc(__ballot_sync(kFullMask, h));
                    if (valid && !h) cur_k[atomicAdd(&wc[d], 1u)] = key[k];
                }
                uint32_t b = 0;
                if (lane == 0 && run != 0) b = atomicAdd(&wc[hot], run);
                b = __shfl_sync(kFullMask, b, 0);
#pragma unroll
                for (int k = 0; k < IPT; ++k) {
                    const bool h = item0 + 32 * k < tile_n && digit_at<false>(key[k], shift, mask) == hot;
                    const uint32_t hm = __ballot_sync(kFullMask, h);
                    if (h) cur_k[b + __popc(hm & ltm)] = key[k];
                    b += __popc(hm);
                }
            } else {
#pragma unroll
                for (int k = 0; k < IPT; ++k) {
                    const bool valid = item0 + 32 * k < tile_n;
                    const uint32_t d = digit_at<false>(key[k], shift, mask);
                    const uint32_t slot = one_digit ? take_slot(wc, d, lane, true) : (valid ? atomicAdd(&wc[d], 1u) : 0u);
                    if (valid) cur_k[slot] = key[k];
                }
            }
        } else {
            uint32_t *wc = s_cnt + warp * kRow;
            const uint32_t ltm = lanemask_lt();
            const LaneConsts c = lane_consts(lane);
#pragma unroll
            for (int k = 0; k < IPT; ++k) {
                const bool valid = item0 + 32 * k < tile_n;
                const uint32_t d = valid ? digit_at<false>(key[k], shift, mask) : 0u;
                const uint32_t peers = digit_peers<kMatchTable>(d, c) & __ballot_sync(kFullMask, valid);
                const uint32_t leader = highest_bit(peers);   // empty only for padding lanes
                uint32_t b = 0;
                if (valid && lane == leader) b = atomicAdd(&wc[d], static_cast<uint32_t>(__popc(peers)));
                b = __shfl_sync(kFullMask, b, leader);
                if (valid) {
                    const uint32_t slot = b + __popc(peers & ltm);
                    cur_k[slot] = key[k];
                    if (PAIRS) cur_v[slot] = val[k];
                }
            }
        }
        __syncthreads();

        // ---- every key to its place: the owning CTA's next buffer, or the output
        for (uint32_t i = tid; i < tile_n; i += T) {
            const uint32_t kk = cur_k[i];
            const uint32_t g = s_goff[digit_at<false>(kk, shift, mask)] + i;
            if (g < a.n) {
                if (last) {
                    a.keys_out[g] = order_out<uint32_t>(kk, a.fmask, a.flip);
                    if (PAIRS) a.vals_out[g] = cur_v[i];
                } else {
                    cluster.map_shared_rank(nxt_k, g / TC)[g % TC] = kk;
                    if (PAIRS) cluster.map_shared_rank(nxt_v, g / TC)[g % TC] = cur_v[i];
                }
            }
        }
        cluster.sync();   // every key has arrived; this pass's buffers and counts are free
    }
}

// Per-device cache: can a cluster of `size` CTAs of this kernel be resident?
struct ClusterFit {
    const void *kernel;
    int device, size, fits;
};
ClusterFit g_fit[64];
int g_fit_n = 0;
std::mutex g_fit_mutex;

template <int IPT, bool PAIRS>
cudaError_t launch_one(const ClusterSortArgs &a, int csize, cudaStream_t s, bool *launched) {
    auto k = k_cluster_sort<IPT, PAIRS>;
    const size_t smem = cluster_smem_words<IPT, PAIRS>() * sizeof(uint32_t);
    cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(k), smem);
    if (e != cudaSuccess) return e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(csize));
    cfg.blockDim = dim3(kClusterThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(csize);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int fits = -1;
    std::lock_guard<std::mutex> lock(g_fit_mutex);
    for (int i = 0; i < g_fit_n; ++i)
        if (g_fit[i].kernel == reinterpret_cast<const void *>(k) && g_fit[i].device == dev && g_fit[i].size == csize)
            fits = g_fit[i].fits;
    if (fits < 0) {
        if (csize > 8 &&
            (e = cudaFuncSetAttribute(reinterpret_cast<const void *>(k),
                                      cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
            return e;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, reinterpret_cast<const void *>(k), &cfg) != cudaSuccess) {
            cudaGetLastError();   // a refused query only means: no
            clusters = 0;
        }
        fits = clusters > 0 ? 1 : 0;
        if (g_fit_n < 64) g_fit[g_fit_n++] = ClusterFit{reinterpret_cast<const void *>(k), dev, csize, fits};
    }
    *launched = fits == 1;
    if (!*launched) return cudaSuccess;
    return cudaLaunchKernelEx(&cfg, k, a);
}

}  // namespace

bool cluster_sort_applies(uint32_t n, int key_bytes, int variant, uint32_t stall_tile, int passes) {
    return key_bytes == 4 && variant == 0 && n > 0 && n <= kClusterSortMaxN && stall_tile == kNoStall &&
           passes > 0;
}

// The smallest power of two of 4096-key CTAs that holds the input (1 .. 16;
// 16 is above the portable cluster size).  Returns GSORT_OK when the sort was
// launched, GSORT_ECUDA on a launch error, and 1 when such a cluster cannot be
// resident here (the caller takes another path).
int launch_cluster_sort(const SmallSortLaunch &L) {
    ClusterSortArgs a;
    a.keys_in = L.keys_in;
    a.keys_out = L.keys_out;
    a.vals_in = L.vals_in;
    a.vals_out = L.vals_out;
    a.n = L.n;
    a.passes = L.passes;
    a.begin_bit = static_cast<uint32_t>(L.begin_bit);
    a.last_mask = L.last_mask;
    a.fmask = L.fmask;
    a.flip = L.flip;
    a.alias = L.alias ? 1 : 0;
    a.status = L.status;
    a.abort_flag = L.abort_flag;
    const bool pairs = L.vals_in != nullptr;
    constexpr uint32_t kTc = kClusterThreads * kClusterIpt;
    int csize = 1;
    while (static_cast<uint32_t>(csize) * kTc < L.n) csize *= 2;
    bool launched = false;
    const cudaError_t e = pairs ? launch_one<kClusterIpt, true>(a, csize, L.stream, &launched)
                                : launch_one<kClusterIpt, false>(a, csize, L.stream, &launched);
    if (e != cudaSuccess) return GSORT_ECUDA;
    return launched ? GSORT_OK : 1;
}

}  // namespace gsort

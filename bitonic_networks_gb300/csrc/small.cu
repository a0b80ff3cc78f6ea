// small.cu -- the whole LSD radix sort of a small input (up to 2^18 32-bit
// keys) in one cooperative launch.  Each CTA owns one 2048-key tile for all
// passes:
//   count the tile's digits of pass 0, publish the 256 counts, grid barrier
//   then per pass: every CTA reads the counts of all tiles for its digits
//   (complete: no look-back), computes the bin starts (the exclusive scan of
//   the digit totals, [CUDA3] kernel 2) and the prefix over earlier tiles,
//   ranks its keys with the warp multisplit and writes per-digit runs
//   ([CUDA3] kernel 3, [PMPP10] 10.4 buffering); every key written also adds
//   one to the next pass's count of its digit in the tile it lands in, so the
//   next pass needs no counting barrier; grid barrier
// That is passes + 1 grid barriers and one launch in place of the histogram
// kernel, the per-pass launches and the chained look-back of the
// large-input path: at these sizes the sort is bound by launch and
// dependency latency, not by bandwidth.  The barriers are bounded waits (a
// CTA that gives up records GSORT_ETIMEOUT and leaves), and the cooperative
// launch guarantees that every CTA is resident.
#include "radix_kernels.cuh"

namespace gsort {
namespace {

constexpr int kSmallSortThreads = 512;
constexpr int kSmallSortIpt = 4;
constexpr int kSmallSortWarps = kSmallSortThreads / 32;
constexpr uint32_t kSmallSortTile = kSmallSortThreads * kSmallSortIpt;   // 2048 keys
constexpr uint32_t kSmallSortMaxN = 1u << 18;
constexpr uint32_t kBarrierSpinFree = 256;   // polls before the first back-off sleep

struct SmallSortArgs {
    const uint32_t *keys_in;
    uint32_t *keys_out;
    const uint32_t *vals_in;   // null: keys only
    uint32_t *vals_out;
    uint32_t *tmp_k, *tmp_v;
    uint32_t n;
    int passes;
    uint32_t begin_bit, last_mask;
    uint32_t fmask, flip;
    int alias;                 // keys or values sorted in place
    uint32_t *counts;          // 3 x [tiles][256] digit counts (see count_buf)
    uint32_t *bar_count;
    uint32_t *status, *abort_flag;
    uint32_t spin_limit, stall_tile;
};

__device__ __forceinline__ void red_release_add_gpu(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid barrier over all CTAs of the launch: a counter that only grows (zeroed
// by the header clear before the launch); barrier k is passed when it
// reaches k * gridDim.x.  The arrival is a release and the poll an acquire,
// so the writes of the whole CTA before the barrier (ordered by the CTA
// barrier) are visible to every CTA after it.  Returns false in every thread
// of the CTA if the wait gave up or the abort flag is up.  `gen` counts the
// barriers this CTA has passed.
__device__ bool grid_barrier(const SmallSortArgs &a, uint32_t &gen, uint32_t *s_flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t target = (gen + 1) * gridDim.x;
        red_release_add_gpu(a.bar_count, 1u);
        bool ok = true;
        uint32_t polls = 0, ns = 32;
        while (ld_acquire(a.bar_count) < target) {
            ++polls;
            if (polls >= a.spin_limit || ((polls & 63u) == 0 && ld_relaxed(a.abort_flag))) {
                ok = false;
                break;
            }
            if (polls > kBarrierSpinFree) backoff(ns);
        }
        if (!ok) record_error(a.status, a.abort_flag, GSORT_ETIMEOUT);
        *s_flag = ok ? 1u : 0u;
    }
    ++gen;
    __syncthreads();
    return *s_flag != 0;
}

// The three count buffers rotate: pass p reads buffer p % 3, its scatter
// fills buffer (p + 1) % 3, and it clears its own row of buffer (p + 2) % 3.
__device__ __forceinline__ uint32_t *count_buf(const SmallSortArgs &a, uint32_t tiles, int p) {
    return a.counts + static_cast<uint32_t>(p % 3) * tiles * 256;
}

template <bool PAIRS, bool MAPPED>
__global__ void __launch_bounds__(kSmallSortThreads, 1) k_small_sort(const SmallSortArgs a) {
    constexpr int T = kSmallSortThreads, IPT = kSmallSortIpt, WARPS = kSmallSortWarps;
    constexpr uint32_t TILE = kSmallSortTile;
    __shared__ uint32_t s_keys[TILE];
    __shared__ uint32_t s_vals[PAIRS ? TILE : 1];
    __shared__ uint32_t s_cnt[WARPS * kRow];   // per-warp digit counts, then next free slots
    __shared__ uint32_t s_goff[256];
    __shared__ uint32_t s_tex[256];            // exclusive scan of this tile's counts over digits
    __shared__ uint32_t s_misc[32];

    const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t tile = blockIdx.x, tiles = gridDim.x;
    if (tile == a.stall_tile) return;   // testing: never arrives, the others' waits run out
    const uint32_t base = tile * TILE;
    const uint32_t tile_n = min(TILE, a.n - base);
    const uint32_t item0 = warp * (32 * IPT) + lane;   // item k at item0 + 32k (warp-contiguous runs)
    uint32_t gen = 0;

    const uint32_t *src_k = a.keys_in;
    const uint32_t *src_v = a.vals_in;
    for (int p = 0; p < a.passes; ++p) {
        uint32_t *dst_k, *dst_v;
        if (a.alias) {
            dst_k = (p % 2 == 0) ? a.tmp_k : a.keys_out;
            dst_v = (p % 2 == 0) ? a.tmp_v : a.vals_out;
        } else {
            dst_k = ((a.passes - 1 - p) % 2 == 0) ? a.keys_out : a.tmp_k;
            dst_v = ((a.passes - 1 - p) % 2 == 0) ? a.vals_out : a.tmp_v;
        }
        const uint32_t shift = a.begin_bit + 8 * p;
        const uint32_t mask = (p == a.passes - 1) ? a.last_mask : 0xFFu;

        // ---- load (L2: the previous pass wrote these words from other CTAs)
        uint32_t key[IPT], val[PAIRS ? IPT : 1];
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            const uint32_t i = item0 + 32 * k;
            const bool ok = i < tile_n;
            key[k] = ok ? __ldcg(src_k + base + i) : 0u;
            if (MAPPED && p == 0) key[k] = order_in<uint32_t>(key[k], a.fmask, a.flip);
            if (PAIRS) val[k] = ok ? __ldcg(src_v + base + i) : 0u;
        }
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
        }
        // Pass 0 publishes its tile counts and waits for everyone's.  Later
        // passes find theirs complete: the previous pass's scatter added every
        // key to the count of the tile it landed in.
        if (p == 0) {
            if (tid < 256) {
                __stcg(count_buf(a, tiles, 0) + tile * 256 + tid, cnt);
                if (a.passes > 1) __stcg(count_buf(a, tiles, 1) + tile * 256 + tid, 0u);
            }
            if (!grid_barrier(a, gen, &s_misc[0])) return;
        }
        // this tile's row of the buffer that the next pass's scatter fills
        // (read by everyone two passes ago, before the last barrier)
        if (p + 2 < a.passes && tid < 256) __stcg(count_buf(a, tiles, p + 2) + tile * 256 + tid, 0u);

        // ---- bin starts and the prefix over earlier tiles, one digit per thread
        const uint32_t *counts = count_buf(a, tiles, p);
        if (tid < 256) {
            // 32 independent loads in flight per round (the loop is latency-bound)
            uint32_t before = 0, total = 0;
            for (uint32_t t0 = 0; t0 < tiles; t0 += 32) {
                uint32_t c[32];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    c[j] = (t0 + j < tiles) ? __ldcg(counts + (t0 + j) * 256 + tid) : 0u;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    before += (t0 + j < tile) ? c[j] : 0u;
                    total += c[j];
                }
            }
            const uint32_t it = warp_inclusive_scan(total, lane);
            const uint32_t ic = warp_inclusive_scan(cnt, lane);
            if (lane == 31) {
                s_misc[4 + warp] = it;
                s_misc[12 + warp] = ic;
            }
            s_goff[tid] = it - total + before;   // completed below with the other warps' sums
            s_tex[tid] = ic - cnt;
        }
        __syncthreads();
        if (tid < 256) {
            uint32_t bt = 0, bc = 0;
            for (uint32_t w = 0; w < warp; ++w) {
                bt += s_misc[4 + w];
                bc += s_misc[12 + w];
            }
            const uint32_t tex = s_tex[tid] + bc;
            s_goff[tid] += bt - tex;   // global index of tile slot i holding digit d: s_goff[d] + i
#pragma unroll
            for (int w = 0; w < WARPS; ++w) s_cnt[w * kRow + tid] += tex;
        }
        __syncthreads();

        // ---- warp multisplit: stable slot of each key in the tile-sorted order
        {
            uint32_t *wc = s_cnt + warp * kRow;
            const uint32_t ltm = lanemask_lt();
            const LaneConsts c = lane_consts(lane);
#pragma unroll
            for (int k = 0; k < IPT; ++k) {
                const bool valid = item0 + 32 * k < tile_n;
                const uint32_t d = valid ? digit_at<false>(key[k], shift, mask) : 0u;
                uint32_t peers = digit_peers<kMatchTable>(d, c) & __ballot_sync(kFullMask, valid);
                const uint32_t leader = highest_bit(peers);
                uint32_t b = 0;
                if (valid && lane == leader) b = atomicAdd(&wc[d], static_cast<uint32_t>(__popc(peers)));
                b = __shfl_sync(kFullMask, b, leader);
                if (valid) {
                    const uint32_t slot = b + __popc(peers & ltm);
                    s_keys[slot] = key[k];
                    if (PAIRS) s_vals[slot] = val[k];
                }
            }
        }
        __syncthreads();

        // ---- contiguous runs per digit out; each key also counts, for the
        // next pass, in the row of the tile it lands in
        const bool last = p == a.passes - 1;
        uint32_t *next_counts = last ? nullptr : count_buf(a, tiles, p + 1);
        const uint32_t next_shift = shift + 8;
        const uint32_t next_mask = (p + 1 == a.passes - 1) ? a.last_mask : 0xFFu;
        for (uint32_t i = tid; i < tile_n; i += T) {
            const uint32_t kk = s_keys[i];
            const uint32_t g = s_goff[digit_at<false>(kk, shift, mask)] + i;
            if (g < a.n) {
                __stcg(dst_k + g, (MAPPED && last) ? order_out<uint32_t>(kk, a.fmask, a.flip) : kk);
                if (PAIRS) __stcg(dst_v + g, s_vals[i]);
                if (!last) atomicAdd(next_counts + (g / TILE) * 256 + digit_at<false>(kk, next_shift, next_mask), 1u);
            }
        }
        if (!grid_barrier(a, gen, &s_misc[0])) return;
        src_k = dst_k;
        src_v = dst_v;
    }
    // in place with an odd pass count: the result is in tmp; copy this tile back
    if (src_k != a.keys_out) {
        for (uint32_t i = tid; i < tile_n; i += T) {
            a.keys_out[base + i] = __ldcg(src_k + base + i);
            if (PAIRS) a.vals_out[base + i] = __ldcg(src_v + base + i);
        }
    }
}

template <bool PAIRS, bool MAPPED>
bool try_launch(const SmallSortArgs &a, uint32_t tiles, int sm_count, cudaStream_t s, cudaError_t &err) {
    auto k = k_small_sort<PAIRS, MAPPED>;
    int per_sm = 0;
    if (blocks_per_sm(reinterpret_cast<const void *>(k), kSmallSortThreads, 0, &per_sm) != cudaSuccess ||
        static_cast<long long>(per_sm) * sm_count < tiles)
        return false;   // not every CTA could be resident: use the large-input path
    SmallSortArgs args = a;
    void *params[] = {&args};
    err = cudaLaunchCooperativeKernel(reinterpret_cast<void *>(k), dim3(tiles), dim3(kSmallSortThreads),
                                      params, 0, s);
    return true;
}

}  // namespace

bool small_sort_applies(uint32_t n, int key_bytes, int variant) {
    return key_bytes == 4 && variant == 0 && n > 0 && n <= kSmallSortMaxN;
}

uint32_t small_sort_tile() { return kSmallSortTile; }

// Returns GSORT_OK when the sort was launched, GSORT_ECUDA on a launch error,
// and 1 when the small-input kernel cannot run here (the caller falls back).
int launch_small_sort(const SmallSortLaunch &L) {
    SmallSortArgs a;
    a.keys_in = L.keys_in;
    a.keys_out = L.keys_out;
    a.vals_in = L.vals_in;
    a.vals_out = L.vals_out;
    a.tmp_k = L.tmp_k;
    a.tmp_v = L.tmp_v;
    a.n = L.n;
    a.passes = L.passes;
    a.begin_bit = static_cast<uint32_t>(L.begin_bit);
    a.last_mask = L.last_mask;
    a.fmask = L.fmask;
    a.flip = L.flip;
    a.alias = L.alias ? 1 : 0;
    a.counts = L.counts;
    a.bar_count = L.bar_count;
    a.status = L.status;
    a.abort_flag = L.abort_flag;
    a.spin_limit = L.spin_limit;
    a.stall_tile = L.stall_tile;
    const uint32_t tiles = (L.n + kSmallSortTile - 1) / kSmallSortTile;
    const bool pairs = L.vals_in != nullptr;
    const bool mapped = L.fmask != 0 || L.flip != 0;
    cudaError_t err = cudaSuccess;
    bool launched;
    if (pairs)
        launched = mapped ? try_launch<true, true>(a, tiles, L.sm_count, L.stream, err)
                          : try_launch<true, false>(a, tiles, L.sm_count, L.stream, err);
    else
        launched = mapped ? try_launch<false, true>(a, tiles, L.sm_count, L.stream, err)
                          : try_launch<false, false>(a, tiles, L.sm_count, L.stream, err);
    if (!launched) return 1;
    return err == cudaSuccess ? GSORT_OK : GSORT_ECUDA;
}

}  // namespace gsort

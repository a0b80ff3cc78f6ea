// radix.cu -- stable LSD radix sort with 8-bit digits for sm_103a.
//
// Steps (page tags as in include/gsort.h):
//   init       clear the workspace header (status, tile counters, histograms)
//   histogram  one read of the keys builds the 256-bin histogram of every
//              digit pass ([CUDA3] "processing several bits at once", kernel 1;
//              [PMPP10] 10.3 histogram step) and clears the first pass's
//              look-back words
//   P x pass   single-pass digit scatter ([CUDA3] kernel 3): each tile ranks
//              its keys stably per digit with a warp multisplit, publishes its
//              per-digit counts, looks back over earlier tiles' counts
//              (decoupled look-back), and writes every key to
//                bin start of its digit (exclusive scan of the pass histogram,
//                [CUDA3] kernel 2, done per tile from the 256 counts)
//              + count of the digit in earlier tiles
//              + stable rank of the key among the tile's keys of that digit,
//              after reordering the tile in shared memory so that global
//              writes go out as contiguous runs per digit ([PMPP10] 10.4 data
//              buffering).  Values move with their keys ([PMPP10] 10.6).
//
// Differences from the pages' kernels: the in-tile rank comes from a warp
// multisplit (peer mask of equal digits + popcount below the lane) instead of
// eight block-wide 1-bit splits; a tile counts its digits first (cheap shared
// atomics) and publishes the counts before ranking, so its look-back overlaps
// other warps' ranking, and the per-warp counters then hand out tile slots
// directly; look-back words are cleared one row per tile by the previous
// kernel instead of a memset per pass; every wait is bounded.
#include <algorithm>

#include "gsort_internal.cuh"

namespace gsort {
namespace {

// ------------------------------------------------------------------- init
__global__ void k_zero_words(uint32_t *p, uint32_t nwords) {
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < nwords;
         i += gridDim.x * blockDim.x)
        p[i] = 0;
}

// -------------------------------------------------------------- histogram
// Every lane owns a private column of counters: counter (pass, digit, lane)
// sits at word ((pass*256 + digit) * 32 + lane), i.e. always in bank `lane`,
// so the shared-memory atomics of a warp never conflict, whatever the keys
// (equal keys included).  One 1024-thread CTA per SM, 128 KiB of counters;
// the columns are summed once per CTA and added to the global histogram.
constexpr int kHistThreads = 1024;
constexpr int kHistUnroll = 4;    // 16-byte loads in flight per thread

__host__ __device__ constexpr size_t hist_smem_bytes(int passes) {
    return static_cast<size_t>(passes) * 256 * 32 * sizeof(uint32_t);
}

// Digit p of key k.  BYTE: the digits are whole bytes of the key (begin_bit a
// multiple of 8, full 8-bit masks) and are extracted with one byte permute.
template <bool BYTE>
__device__ __forceinline__ uint32_t digit_at(uint32_t k, uint32_t shift, uint32_t mask) {
    if constexpr (BYTE) return __byte_perm(k, 0u, 0x4440u | (shift >> 3));
    else return (k >> shift) & mask;
}

template <bool XF, bool BYTE>
__device__ __forceinline__ void hist_count(uint32_t *col, uint32_t k, uint32_t begin_bit,
                                           int passes, uint32_t last_mask) {
    if (XF) k = float_key_in(k);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        if (p < passes) {
            const uint32_t d = digit_at<BYTE>(k, begin_bit + 8 * p, p == passes - 1 ? last_mask : 0xFFu);
            atomicAdd(&col[(p * 256 + d) * 32], 1u);
        }
    }
}

template <bool XF, bool BYTE>
__global__ void __launch_bounds__(kHistThreads, 1)
k_digit_hist(const uint32_t *__restrict__ keys, uint32_t n, uint32_t begin_bit, int passes,
             uint32_t last_mask, uint32_t *__restrict__ hist, uint4 *__restrict__ clear,
             uint32_t clear_vec4) {
    extern __shared__ uint32_t s_h[];
    const uint32_t tid = threadIdx.x;
    const uint32_t words = static_cast<uint32_t>(passes) * 256 * 32;
    for (uint32_t i = tid; i < words; i += kHistThreads) s_h[i] = 0;
    const uint32_t gtid = blockIdx.x * kHistThreads + tid;
    const uint32_t gstride = gridDim.x * kHistThreads;
    for (uint32_t i = gtid; i < clear_vec4; i += gstride) clear[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();

    uint32_t *col = s_h + (tid & 31);
    // elements before the first 16-byte boundary, the vector body, the tail
    uint32_t head = static_cast<uint32_t>(((16 - (reinterpret_cast<uintptr_t>(keys) & 15)) & 15) >> 2);
    head = min(head, n);
    const uint32_t nvec = (n - head) >> 2;
    const uint4 *vec = reinterpret_cast<const uint4 *>(keys + head);
    for (uint32_t v = gtid; v < nvec; v += kHistUnroll * gstride) {
        uint4 q[kHistUnroll];
#pragma unroll
        for (int u = 0; u < kHistUnroll; ++u) {
            const uint32_t idx = v + u * gstride;
            if (idx < nvec) q[u] = __ldcs(vec + idx);
        }
#pragma unroll
        for (int u = 0; u < kHistUnroll; ++u) {
            if (v + u * gstride < nvec) {
                hist_count<XF, BYTE>(col, q[u].x, begin_bit, passes, last_mask);
                hist_count<XF, BYTE>(col, q[u].y, begin_bit, passes, last_mask);
                hist_count<XF, BYTE>(col, q[u].z, begin_bit, passes, last_mask);
                hist_count<XF, BYTE>(col, q[u].w, begin_bit, passes, last_mask);
            }
        }
    }
    const uint32_t tail0 = head + nvec * 4;
    if (gtid < head) hist_count<XF, BYTE>(col, keys[gtid], begin_bit, passes, last_mask);
    if (gtid < n - tail0) hist_count<XF, BYTE>(col, keys[tail0 + gtid], begin_bit, passes, last_mask);
    __syncthreads();

    // sum each (pass, digit) row over the 32 lane columns; the rotated start
    // keeps the 32 threads of a warp on 32 different banks
    for (uint32_t i = tid; i < static_cast<uint32_t>(passes) * 256; i += kHistThreads) {
        uint32_t s = 0;
#pragma unroll 8
        for (uint32_t j = 0; j < 32; ++j) s += s_h[i * 32 + ((j + i) & 31)];
        if (s) atomicAdd(&hist[i], s);
    }
}

// ----------------------------------------------------------- digit pass
struct PassArgs {
    const uint32_t *src_k;
    uint32_t *dst_k;
    const uint32_t *src_v;
    uint32_t *dst_v;
    uint32_t n;
    uint32_t shift;         // digit = (key >> shift) & mask
    uint32_t mask;
    const uint32_t *hist;   // the 256 counts of this pass
    uint32_t *look;         // [tiles][256] look-back words of this pass (cleared): flag | count
    uint32_t *look_clear;   // next pass's words: row `tile` is cleared here; may be null
    uint32_t *tile_counter;
    uint32_t *status;
    uint32_t *abort_flag;
    uint32_t spin_limit;
    uint32_t stall_tile;
};

// ------------------------------------------------------- warp multisplit
// Ranking methods for the mask of lanes whose digit equals this lane's:
//   kMatchTable  the eight ballots (bit planes of the warp's digits) are turned
//                into two lane-distributed tables: lane l holds the mask of
//                lanes whose low five digit bits equal l, and the mask of lanes
//                whose top three bits equal l & 7 (built with per-lane
//                constants, no per-key bit tests); a lane fetches its two
//                entries with two shuffles and ANDs them.
//   kMatchSelect each lane selects, per bit, the ballot or its complement.
//   kMatchAny    the hardware match.any instruction.
constexpr int kMatchTable = 0, kMatchSelect = 1, kMatchAny = 2;

struct LaneConsts {
    uint32_t inv[5];   // ~0 where bit b of the lane id is 0, else 0
};

__device__ __forceinline__ LaneConsts lane_consts(uint32_t lane) {
    LaneConsts c;
#pragma unroll
    for (int b = 0; b < 5; ++b) c.inv[b] = ((lane >> b) & 1u) ? 0u : kFullMask;
    return c;
}

// Ballot of (d & bit) != 0 over the warp.
__device__ __forceinline__ uint32_t ballot_bit(uint32_t d, uint32_t bit) {
    return __ballot_sync(kFullMask, (d & bit) != 0u);
}

// (a ^ b) & c in one three-input logic operation.
__device__ __forceinline__ uint32_t xor_and(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x28;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// Position of the highest set bit (x != 0).
__device__ __forceinline__ uint32_t highest_bit(uint32_t x) {
    uint32_t r;
    asm("bfind.u32 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}

template <int MATCH>
__device__ __forceinline__ uint32_t digit_peers(uint32_t d, const LaneConsts &c) {
    if constexpr (MATCH == kMatchAny) {
        return __match_any_sync(kFullMask, d);
    } else if constexpr (MATCH == kMatchSelect) {
        uint32_t peers = kFullMask;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const bool bit = (d >> b) & 1u;
            const uint32_t m = __ballot_sync(kFullMask, bit);
            peers &= bit ? m : ~m;
        }
        return peers;
    } else {
        uint32_t m[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) m[b] = ballot_bit(d, 1u << b);
        // lo: lanes whose digit bits 0..4 equal this lane's id; hi: lanes whose
        // digit bits 5..7 equal this lane's id bits 0..2
        uint32_t lo = m[0] ^ c.inv[0];
        lo = xor_and(m[1], c.inv[1], lo);
        lo = xor_and(m[2], c.inv[2], lo);
        lo = xor_and(m[3], c.inv[3], lo);
        lo = xor_and(m[4], c.inv[4], lo);
        uint32_t hi = m[5] ^ c.inv[0];
        hi = xor_and(m[6], c.inv[1], hi);
        hi = xor_and(m[7], c.inv[2], hi);
        // a shuffle reads its source lane from the low five bits of its lane operand
        return __shfl_sync(kFullMask, lo, d) & __shfl_sync(kFullMask, hi, d >> 5);
    }
}

constexpr int kRow = 256;   // per-warp digit counters

template <int WARPS, int IPT, bool PAIRS>
constexpr size_t pass_smem_words() {
    // keys [+ values] of the tile, per-warp counters, 256 digit offsets, 32 misc words
    return static_cast<size_t>(WARPS * 32 * IPT) * (PAIRS ? 2 : 1) + WARPS * kRow + 256 + 32;
}


// Exclusive prefix of digit d over all tiles before `tile`.  Each word holds a
// flag (AGG: the tile's count; PREFIX: the count over tiles 0..t) and a
// 30-bit count, so one round trip reads W predecessors at once; the
// nearest PREFIX word ends the walk and the AGG words before it are summed.
// Returns false if a wait gave up.
template <int W>
__device__ __forceinline__ bool look_back(const PassArgs &a, uint32_t tile, uint32_t d,
                                          uint32_t &excl) {
    excl = 0;
    int32_t t = static_cast<int32_t>(tile) - 1;
    uint32_t polls = 0, ns = 32;
    while (true) {
        uint32_t w[W];
#pragma unroll
        for (int i = 0; i < W; ++i)
            w[i] = (t - i >= 0) ? ld_relaxed(a.look + static_cast<uint32_t>(t - i) * 256 + d)
                                : kFlagPrefix;   // before tile 0: an empty prefix
        // sum words up to and including the nearest PREFIX; any empty word
        // before it means a predecessor has not published yet
        uint32_t sum = 0;
        bool done = false, pending = false;
#pragma unroll
        for (int i = 0; i < W; ++i) {
            if (!done) {
                pending |= (w[i] & ~kValueMask) == 0;
                sum += w[i] & kValueMask;
                done = (w[i] & kFlagPrefix) != 0;
            }
        }
        if (pending) {
            if (++polls >= a.spin_limit || ld_relaxed(a.abort_flag)) return false;
            backoff(ns);
            continue;
        }
        excl += sum;
        if (done) return true;
        t -= W;
    }
}

// One tile of a digit pass.  kin/vin point at the tile's first key/value (in
// global memory, or in a shared staging buffer); the tile-sorted keys/values
// go to s_keys/s_vals (which may be the staging buffers: every key is in
// registers before the first write).  tab = the shared tables: per-warp digit
// counters, digit offsets, misc words.  before_output() runs in every thread
// after the last block barrier, before the output phase.  Returns false when
// the tile stops (device error or the test stall), after that barrier.
struct NoHook {
    __device__ void operator()() const {}
};

template <int WARPS, int IPT, int MATCH, int LW, bool BYTE, bool PAIRS, bool XIN, bool XOUT, bool FULL,
          class Hook = NoHook>
__device__ __forceinline__ bool pass_tile(const PassArgs &a, uint32_t *tab, uint32_t tile,
                                          const uint32_t *kin, const uint32_t *vin,
                                          uint32_t *s_keys, uint32_t *s_vals,
                                          const Hook &before_output = Hook()) {
    constexpr int T = WARPS * 32;
    constexpr int TILE = T * IPT;
    uint32_t *s_cnt = tab;                      // [WARPS][256] counts, then next free slots
    uint32_t *s_goff = s_cnt + WARPS * kRow;    // [256] global index - tile slot
    uint32_t *s_misc = s_goff + 256;            // [32]

    const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t tile_base = tile * TILE;
    const uint32_t tile_n = FULL ? TILE : a.n - tile_base;
    // Item k of this thread sits at tile index item0 + 32k: each warp owns a
    // contiguous run of 32*IPT keys and walks it in order, which makes the
    // warp-local ranks stable.
    const uint32_t item0 = warp * (32 * IPT) + lane;

    uint32_t key[IPT];
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        const uint32_t i = item0 + k * 32;
        key[k] = (FULL || i < tile_n) ? kin[i] : 0u;
        if (XIN) key[k] = float_key_in(key[k]);
    }
    uint32_t val[PAIRS ? IPT : 1];
    if (PAIRS) {
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            const uint32_t i = item0 + k * 32;
            val[k] = (FULL || i < tile_n) ? vin[i] : 0u;
        }
    }

    // ---- early counts: this warp's keys per digit (order does not matter here)
    {
        uint32_t *wc = s_cnt + warp * kRow;
#pragma unroll
        for (int k = 0; k < IPT; ++k)
            if (FULL || item0 + k * 32 < tile_n) atomicAdd(&wc[digit_at<BYTE>(key[k], a.shift, a.mask)], 1u);
    }
    __syncthreads();

    // ---- tile counts per digit, published at once; scans over the 256 digits
    uint32_t cnt = 0, tile_excl = 0, bin_excl = 0;
    if (tid < 256) {
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            const uint32_t cw = s_cnt[w * kRow + tid];
            s_cnt[w * kRow + tid] = cnt;   // exclusive over warps
            cnt += cw;
        }
        if (tile != a.stall_tile)
            st_relaxed(a.look + tile * 256 + tid, (tile == 0 ? kFlagPrefix : kFlagAgg) | cnt);
        const uint32_t bin = a.hist[tid];
        const uint32_t ic = warp_inclusive_scan(cnt, lane);
        const uint32_t ib = warp_inclusive_scan(bin, lane);
        if (lane == 31) {
            s_misc[4 + warp] = ic;
            s_misc[12 + warp] = ib;
        }
        tile_excl = ic - cnt;
        bin_excl = ib - bin;
    }
    if (a.look_clear != nullptr)
        for (uint32_t i = tid; i < 256; i += T) a.look_clear[tile * 256 + i] = 0;
    __syncthreads();
    if (tid < 256) {
        for (uint32_t w = 0; w < warp; ++w) {
            tile_excl += s_misc[4 + w];
            bin_excl += s_misc[12 + w];
        }
        // s_cnt[w][d]: tile slot where warp w's first key of digit d goes
#pragma unroll
        for (int w = 0; w < WARPS; ++w) s_cnt[w * kRow + tid] += tile_excl;
    }
    __syncthreads();

    // ---- decoupled look-back, one digit per thread of the first 8 warps
    // (the other warps rank meanwhile); then publish this tile's prefixes
    if (tid < 256) {
        uint32_t excl = 0;
        bool ok = true;
        if (tile > 0 && tile != a.stall_tile) {
            ok = look_back<LW>(a, tile, tid, excl);
            if (ok) st_relaxed(a.look + tile * 256 + tid, kFlagPrefix | (excl + cnt));
        }
        if (!ok) {
            s_misc[2] = 1;
            record_error(a.status, a.abort_flag, GSORT_ETIMEOUT);
        }
        // global index of tile slot i holding digit d: s_goff[d] + i
        s_goff[tid] = bin_excl + excl - tile_excl;
    }

    // ---- warp multisplit: stable slot of each key in the tile-sorted order
    {
        uint32_t *wc = s_cnt + warp * kRow;
        const uint32_t ltm = lanemask_lt();
        const LaneConsts c = lane_consts(lane);
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            const bool valid = FULL || item0 + k * 32 < tile_n;
            const uint32_t d = valid ? digit_at<BYTE>(key[k], a.shift, a.mask) : 0u;
            uint32_t peers = digit_peers<MATCH>(d, c);
            if (!FULL) peers &= __ballot_sync(kFullMask, valid);
            const uint32_t leader = highest_bit(peers);   // peers is empty only for padding lanes
            uint32_t base = 0;
            if (valid && lane == leader)
                base = atomicAdd(&wc[d], static_cast<uint32_t>(__popc(peers)));
            base = __shfl_sync(kFullMask, base, leader);
            if (valid) {
                const uint32_t slot = base + __popc(peers & ltm);
                s_keys[slot] = key[k];
                if (PAIRS) s_vals[slot] = val[k];
            }
        }
    }
    __syncthreads();
    before_output();
    if (s_misc[2] || tile == a.stall_tile) return false;

    // ---- contiguous runs per digit out to global memory
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        const uint32_t i = k * T + tid;
        if (FULL || i < tile_n) {
            const uint32_t kk = s_keys[i];
            const uint32_t g = s_goff[digit_at<BYTE>(kk, a.shift, a.mask)] + i;
            if (g < a.n) {
                a.dst_k[g] = XOUT ? float_key_out(kk) : kk;
                if (PAIRS) a.dst_v[g] = s_vals[i];
            }
        }
    }
    return true;
}

template <int WARPS, int IPT, int MINB, int MATCH, int LW, bool BYTE, bool PAIRS, bool XIN, bool XOUT>
__global__ void __launch_bounds__(WARPS * 32, MINB) k_digit_pass(const PassArgs a) {
    constexpr int TILE = WARPS * 32 * IPT;
    extern __shared__ uint32_t smem[];
    uint32_t *s_misc = smem + pass_smem_words<WARPS, IPT, PAIRS>() - 32;
    const uint32_t tid = threadIdx.x;
    if (tid == 0) {
        s_misc[0] = atomicAdd(a.tile_counter, 1u);   // tiles in start order: look-back always progresses
        s_misc[1] = ld_relaxed(a.abort_flag);
        s_misc[2] = 0;
    }
    uint32_t *s_cnt = smem + TILE * (PAIRS ? 2 : 1);
    for (uint32_t i = tid; i < WARPS * kRow; i += WARPS * 32) s_cnt[i] = 0;
    __syncthreads();
    const uint32_t tile = s_misc[0];
    if (s_misc[1]) return;   // an earlier wait gave up; the result is void anyway
    uint32_t *s_keys = smem, *s_vals = smem + TILE;
    const uint32_t *kin = a.src_k + tile * TILE;
    const uint32_t *vin = PAIRS ? a.src_v + tile * TILE : nullptr;
    if (a.n - tile * TILE >= static_cast<uint32_t>(TILE))
        pass_tile<WARPS, IPT, MATCH, LW, BYTE, PAIRS, XIN, XOUT, true>(a, s_cnt, tile, kin, vin, s_keys, s_vals);
    else
        pass_tile<WARPS, IPT, MATCH, LW, BYTE, PAIRS, XIN, XOUT, false>(a, s_cnt, tile, kin, vin, s_keys, s_vals);
}

// ------------------------------------------------- persistent digit pass
// A grid of resident CTAs loops over tiles.  During the output phase of tile
// k a CTA claims its next tile and starts a TMA bulk copy of its keys into the
// other shared buffer, so the claim and the loads overlap the stores of tile
// k.  A claimed tile waits only for one output phase before its counts are
// published (claiming any earlier makes other tiles' look-backs wait), and
// tiles are claimed and processed in increasing order, so the smallest
// unfinished tile can always complete.
constexpr uint32_t kBulkWaitLimit = 1u << 20;   // polls of a load barrier before giving up

template <int WARPS, int IPT, bool PAIRS>
constexpr size_t persist_smem_words() {
    // 2 barriers (padded to 32 words), 2 key buffers [, 2 value buffers], tables
    return 32 + static_cast<size_t>(WARPS * 32 * IPT) * (PAIRS ? 4 : 2) + WARPS * kRow + 256 + 32;
}

template <int TILE, bool PAIRS>
struct Prefetch {
    const PassArgs *a;
    uint64_t *bar;
    uint32_t *kbuf, *vbuf;
    // thread 0: bulk copy of tile t into buffer b
    __device__ void operator()(uint32_t t, uint32_t b) const {
        const uint32_t n_t = min(static_cast<uint32_t>(TILE), a->n - t * TILE);
        const uint32_t bytes = (n_t & ~3u) * 4u;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bar[b], bytes * (PAIRS ? 2u : 1u));
        if (bytes > 0) {
            bulk_load(kbuf + b * TILE, a->src_k + t * TILE, bytes, &bar[b]);
            if (PAIRS) bulk_load(vbuf + b * TILE, a->src_v + t * TILE, bytes, &bar[b]);
        }
    }
};

template <int TILE, bool PAIRS>
struct ClaimNext {
    const Prefetch<TILE, PAIRS> *pf;
    uint32_t *counter, *slot;
    uint32_t tiles, buffer;
    __device__ void operator()() const {
        if (threadIdx.x == 0) {
            const uint32_t next = atomicAdd(counter, 1u);
            *slot = next;
            if (next < tiles) (*pf)(next, buffer);
        }
    }
};

template <int WARPS, int IPT, int MATCH, int LW, bool BYTE, bool PAIRS, bool XIN, bool XOUT>
__global__ void __launch_bounds__(WARPS * 32, 2) k_digit_pass_persistent(const PassArgs a,
                                                                        uint32_t tiles) {
    constexpr int T = WARPS * 32;
    constexpr int TILE = T * IPT;
    extern __shared__ __align__(128) uint32_t smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);          // [2]
    uint32_t *kbuf = smem + 32;                                   // [2][TILE]
    uint32_t *vbuf = kbuf + 2 * TILE;                             // [2][TILE] (pairs)
    uint32_t *tab = smem + 32 + static_cast<size_t>(TILE) * (PAIRS ? 4 : 2);
    uint32_t *s_misc = tab + WARPS * kRow + 256;
    const uint32_t tid = threadIdx.x;
    const Prefetch<TILE, PAIRS> prefetch{&a, bar, kbuf, vbuf};

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        const uint32_t t0 = atomicAdd(a.tile_counter, 1u);
        s_misc[24] = t0;
        if (t0 < tiles) prefetch(t0, 0);
    }
    __syncthreads();
    uint32_t tile = s_misc[24];   // its copy into buffer b is in flight if tile < tiles
    uint32_t b = 0;
    uint32_t phase[2] = {0u, 0u};
    while (tile < tiles) {
        if (tid == 0) s_misc[2] = 0;
        for (uint32_t i = tid; i < WARPS * kRow; i += T) tab[i] = 0;
        const bool arrived = mbar_wait_bounded(&bar[b], phase[b], kBulkWaitLimit);
        const uint32_t tile_n = min(static_cast<uint32_t>(TILE), a.n - tile * TILE);
        uint32_t *kb = kbuf + b * TILE;
        uint32_t *vb = vbuf + b * TILE;
        const uint32_t rest = tile_n & 3u;   // the last keys of a ragged tile come by plain loads
        if (arrived && tid < rest) {
            kb[tile_n - rest + tid] = a.src_k[tile * TILE + tile_n - rest + tid];
            if (PAIRS) vb[tile_n - rest + tid] = a.src_v[tile * TILE + tile_n - rest + tid];
        }
        if (__syncthreads_or(!arrived || (tid == 0 && ld_relaxed(a.abort_flag) != 0))) {
            // the result is void; leave only once no copy into this block is in flight
            if (tid == 0 && !arrived) record_error(a.status, a.abort_flag, GSORT_ETIMEOUT);
            if (!arrived) mbar_wait_bounded(&bar[b], phase[b], kBulkWaitLimit);
            return;
        }
        phase[b] ^= 1u;
        const ClaimNext<TILE, PAIRS> claim{&prefetch, a.tile_counter, &s_misc[24], tiles, b ^ 1u};
        bool ok;
        if (tile_n == static_cast<uint32_t>(TILE))
            ok = pass_tile<WARPS, IPT, MATCH, LW, BYTE, PAIRS, XIN, XOUT, true>(a, tab, tile, kb, vb, kb, vb, claim);
        else
            ok = pass_tile<WARPS, IPT, MATCH, LW, BYTE, PAIRS, XIN, XOUT, false>(a, tab, tile, kb, vb, kb, vb, claim);
        __syncthreads();   // buffer b is read out, and the next tile id is visible
        const uint32_t next = s_misc[24];
        if (!ok && tile != a.stall_tile) {   // a look-back gave up
            if (next < tiles) mbar_wait_bounded(&bar[b ^ 1u], phase[b ^ 1u], kBulkWaitLimit);
            return;
        }
        tile = next;
        b ^= 1u;
    }
}

// ------------------------------------------------------------ variants
template <int WARPS, int IPT, int MINB, int MATCH, int LW = 8>
struct PassConfig {
    static constexpr uint32_t kTile = WARPS * 32 * IPT;

    template <bool B, bool P, bool XI, bool XO>
    static cudaError_t launch_one(const PassArgs &a, uint32_t tiles, cudaStream_t s) {
        auto k = k_digit_pass<WARPS, IPT, MINB, MATCH, LW, B, P, XI, XO>;
        const size_t smem = pass_smem_words<WARPS, IPT, P>() * sizeof(uint32_t);
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        k<<<tiles, WARPS * 32, smem, s>>>(a);
        return cudaGetLastError();
    }

    template <bool B>
    static cudaError_t launch_b(const PassArgs &a, bool pairs, bool xin, bool xout, uint32_t tiles,
                                cudaStream_t s) {
        const int sel = (pairs ? 4 : 0) | (xin ? 2 : 0) | (xout ? 1 : 0);
        switch (sel) {
            case 0: return launch_one<B, false, false, false>(a, tiles, s);
            case 1: return launch_one<B, false, false, true>(a, tiles, s);
            case 2: return launch_one<B, false, true, false>(a, tiles, s);
            case 3: return launch_one<B, false, true, true>(a, tiles, s);
            case 4: return launch_one<B, true, false, false>(a, tiles, s);
            case 5: return launch_one<B, true, false, true>(a, tiles, s);
            case 6: return launch_one<B, true, true, false>(a, tiles, s);
            default: return launch_one<B, true, true, true>(a, tiles, s);
        }
    }

    static cudaError_t launch(const PassArgs &a, bool pairs, bool xin, bool xout, uint32_t tiles,
                              cudaStream_t s) {
        const bool byte = (a.shift % 8) == 0 && a.mask == 0xFFu;
        return byte ? launch_b<true>(a, pairs, xin, xout, tiles, s)
                    : launch_b<false>(a, pairs, xin, xout, tiles, s);
    }
};

// Persistent configuration: grid = 2 CTAs per SM (at most one per tile).
// Sources that are not 16-byte aligned take the one-tile-per-CTA kernel with
// the same tile shape.
template <int WARPS, int IPT, int MATCH, int LW = 8>
struct PersistentConfig {
    static constexpr uint32_t kTile = WARPS * 32 * IPT;

    template <bool B, bool P, bool XI, bool XO>
    static cudaError_t launch_one(const PassArgs &a, uint32_t tiles, cudaStream_t s) {
        auto k = k_digit_pass_persistent<WARPS, IPT, MATCH, LW, B, P, XI, XO>;
        const size_t smem = persist_smem_words<WARPS, IPT, P>() * sizeof(uint32_t);
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, WARPS * 32, smem);
        if (e != cudaSuccess) return e;
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cudaErrorUnknown;
        const uint32_t grid = std::max(1u, std::min(tiles, static_cast<uint32_t>(std::max(per_sm, 1) * sms)));
        k<<<grid, WARPS * 32, smem, s>>>(a, tiles);
        return cudaGetLastError();
    }

    template <bool B>
    static cudaError_t launch_b(const PassArgs &a, bool pairs, bool xin, bool xout, uint32_t tiles,
                                cudaStream_t s) {
        const int sel = (pairs ? 4 : 0) | (xin ? 2 : 0) | (xout ? 1 : 0);
        switch (sel) {
            case 0: return launch_one<B, false, false, false>(a, tiles, s);
            case 1: return launch_one<B, false, false, true>(a, tiles, s);
            case 2: return launch_one<B, false, true, false>(a, tiles, s);
            case 3: return launch_one<B, false, true, true>(a, tiles, s);
            case 4: return launch_one<B, true, false, false>(a, tiles, s);
            case 5: return launch_one<B, true, false, true>(a, tiles, s);
            case 6: return launch_one<B, true, true, false>(a, tiles, s);
            default: return launch_one<B, true, true, true>(a, tiles, s);
        }
    }

    static cudaError_t launch(const PassArgs &a, bool pairs, bool xin, bool xout, uint32_t tiles,
                              cudaStream_t s) {
        const bool aligned16 = (reinterpret_cast<uintptr_t>(a.src_k) & 15) == 0 &&
                               (!pairs || (reinterpret_cast<uintptr_t>(a.src_v) & 15) == 0);
        if (!aligned16)
            return PassConfig<WARPS, IPT, 2, MATCH, LW>::launch(a, pairs, xin, xout, tiles, s);
        const bool byte = (a.shift % 8) == 0 && a.mask == 0xFFu;
        return byte ? launch_b<true>(a, pairs, xin, xout, tiles, s)
                    : launch_b<false>(a, pairs, xin, xout, tiles, s);
    }
};

struct Variant {
    const char *name;
    uint32_t tile;
    cudaError_t (*launch)(const PassArgs &, bool, bool, bool, uint32_t, cudaStream_t);
};

const Variant kVariants[] = {
    {"one tile per CTA, 16 warps x 16 items", PassConfig<16, 16, 2, kMatchTable>::kTile,
     &PassConfig<16, 16, 2, kMatchTable>::launch},
    {"persistent, 16 warps x 16 items, TMA prefetch", PersistentConfig<16, 16, kMatchTable>::kTile,
     &PersistentConfig<16, 16, kMatchTable>::launch},
    {"one tile per CTA, 8 warps x 16 items", PassConfig<8, 16, 3, kMatchTable>::kTile,
     &PassConfig<8, 16, 3, kMatchTable>::launch},
};
constexpr int kNumVariants = sizeof(kVariants) / sizeof(kVariants[0]);

cudaError_t launch_hist(const uint32_t *keys, uint32_t n, int kind, int begin_bit, int passes,
                        uint32_t last_mask, uint32_t *hist, uint32_t *clear, uint32_t clear_words,
                        cudaStream_t s, int sm_count) {
    // one CTA per SM (fewer for small inputs: about 16 keys per thread at least)
    const uint32_t want = (n + kHistThreads * 16 - 1) / (kHistThreads * 16);
    const uint32_t grid = std::max(1u, std::min(want, static_cast<uint32_t>(sm_count)));
    uint4 *cl = reinterpret_cast<uint4 *>(clear);
    const bool byte = (begin_bit % 8) == 0 && last_mask == 0xFFu;
    auto k = (kind == GSORT_KEY_F32) ? (byte ? k_digit_hist<true, true> : k_digit_hist<true, false>)
                                     : (byte ? k_digit_hist<false, true> : k_digit_hist<false, false>);
    const size_t smem = hist_smem_bytes(passes);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(hist_smem_bytes(4)));
    if (e != cudaSuccess) return e;
    k<<<grid, kHistThreads, smem, s>>>(keys, n, begin_bit, passes, last_mask, hist, cl,
                                       clear_words / 4);
    return cudaGetLastError();
}

void record(cudaEvent_t *ev, int num, int idx, cudaStream_t s) {
    if (ev != nullptr && idx < num && ev[idx] != nullptr) cudaEventRecord(ev[idx], s);
}

}  // namespace

int radix_num_variants() { return kNumVariants; }

const char *radix_variant_name(int v) {
    return (v >= 0 && v < kNumVariants) ? kVariants[v].name : nullptr;
}

uint32_t radix_variant_tile(int v) { return kVariants[v].tile; }

RadixLayout radix_layout(uint32_t n, bool with_values) {
    RadixLayout L{};
    L.tiles_max = (n + kMinRadixTile - 1) / kMinRadixTile;
    size_t off = kHdrBytes;
    const size_t region = align_up(static_cast<size_t>(L.tiles_max) * 256 * sizeof(uint32_t), kWsAlign);
    L.look_a = off;   // [tiles_max][256] look-back words, passes 0, 2
    off += region;
    L.look_b = off;   // passes 1, 3
    off += region;
    L.tmp_keys = off;
    off += align_up(static_cast<size_t>(n) * sizeof(uint32_t), kWsAlign);
    L.tmp_vals = off;
    if (with_values) off += align_up(static_cast<size_t>(n) * sizeof(uint32_t), kWsAlign);
    L.total = off;
    return L;
}

int launch_radix(const RadixLaunch &L) {
    const int passes = (L.end_bit - L.begin_bit + 7) / 8;
    const bool pairs = L.vals_in != nullptr;
    const RadixLayout lay = radix_layout(L.n, pairs);
    const Variant &V = kVariants[L.variant];
    const uint32_t tiles = (L.n + V.tile - 1) / V.tile;
    cudaStream_t s = L.stream;

    uint32_t *hdr = reinterpret_cast<uint32_t *>(L.ws);
    uint32_t *status = reinterpret_cast<uint32_t *>(L.ws + kHdrStatus);
    uint32_t *abort_flag = reinterpret_cast<uint32_t *>(L.ws + kHdrAbort);
    uint32_t *hist = reinterpret_cast<uint32_t *>(L.ws + kHdrHist);
    uint32_t *look[2] = {reinterpret_cast<uint32_t *>(L.ws + lay.look_a),
                         reinterpret_cast<uint32_t *>(L.ws + lay.look_b)};
    uint32_t *tmp_k = reinterpret_cast<uint32_t *>(L.ws + lay.tmp_keys);
    uint32_t *tmp_v = pairs ? reinterpret_cast<uint32_t *>(L.ws + lay.tmp_vals) : nullptr;

    record(L.events, L.num_events, 0, s);
    k_zero_words<<<1, 256, 0, s>>>(hdr, static_cast<uint32_t>(kHdrBytes / sizeof(uint32_t)));
    if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
    record(L.events, L.num_events, 1, s);

    const uint32_t last_width = static_cast<uint32_t>(L.end_bit - L.begin_bit - 8 * (passes - 1));
    const uint32_t last_mask = (1u << last_width) - 1u;
    // the histogram kernel also clears the first pass's look-back words
    if (launch_hist(L.keys_in, L.n, L.kind, L.begin_bit, passes, last_mask, hist, look[0],
                    tiles * 256, s, L.sm_count) != cudaSuccess)
        return GSORT_ECUDA;
    record(L.events, L.num_events, 2, s);

    // In place (either array): in -> tmp -> out -> tmp ...; an odd pass count
    // ends in tmp and is copied back.  Otherwise the sequence is arranged so
    // that the last pass writes to out.
    const bool alias = (L.keys_in == L.keys_out) || (pairs && L.vals_in == L.vals_out);
    const uint32_t *src_k = L.keys_in;
    const uint32_t *src_v = L.vals_in;
    uint32_t *dst_k = nullptr, *dst_v = nullptr;
    for (int p = 0; p < passes; ++p) {
        const bool to_out = alias ? (p % 2 == 1) : ((passes - 1 - p) % 2 == 0);
        dst_k = to_out ? L.keys_out : tmp_k;
        dst_v = pairs ? (to_out ? L.vals_out : tmp_v) : nullptr;
        PassArgs a;
        a.src_k = src_k;
        a.dst_k = dst_k;
        a.src_v = src_v;
        a.dst_v = dst_v;
        a.n = L.n;
        a.shift = static_cast<uint32_t>(L.begin_bit + 8 * p);
        a.mask = (p == passes - 1) ? last_mask : 0xFFu;
        a.hist = hist + p * 256;
        a.look = look[p & 1];
        a.look_clear = (p + 1 < passes) ? look[(p + 1) & 1] : nullptr;
        a.tile_counter = reinterpret_cast<uint32_t *>(L.ws + kHdrCounters + 128 * p);
        a.status = status;
        a.abort_flag = abort_flag;
        a.spin_limit = L.spin_limit;
        a.stall_tile = L.stall_tile;
        const bool xin = (L.kind == GSORT_KEY_F32) && p == 0;
        const bool xout = (L.kind == GSORT_KEY_F32) && p == passes - 1;
        if (V.launch(a, pairs, xin, xout, tiles, s) != cudaSuccess) return GSORT_ECUDA;
        record(L.events, L.num_events, 3 + p, s);
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

int launch_digit_histograms(const uint32_t *keys, uint32_t n, int kind, int begin_bit, int end_bit,
                            uint32_t *hist_out, cudaStream_t stream, int sm_count) {
    const int passes = (end_bit - begin_bit + 7) / 8;
    if (passes == 0) return GSORT_OK;
    k_zero_words<<<1, 256, 0, stream>>>(hist_out, static_cast<uint32_t>(passes * 256));
    if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
    if (n == 0) return GSORT_OK;
    const uint32_t last_width = static_cast<uint32_t>(end_bit - begin_bit - 8 * (passes - 1));
    const uint32_t last_mask = (1u << last_width) - 1u;
    if (launch_hist(keys, n, kind, begin_bit, passes, last_mask, hist_out, nullptr, 0, stream,
                    sm_count) != cudaSuccess)
        return GSORT_ECUDA;
    return GSORT_OK;
}

}  // namespace gsort

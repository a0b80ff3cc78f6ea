// radix_kernels.cuh -- device code of the LSD radix sort, generic in the key
// word (32- or 64-bit), shared by radix.cu (32-bit keys) and radix64.cu
// (64-bit keys).
//
// Steps (page tags as in include/gsort.h):
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
// Key kinds other than unsigned ascending are sorted through an order map
// applied when a pass first loads a key and inverted when the last pass
// stores it: floats ([PMPP10] section 8, exercise 7) map to unsigned integers
// in IEEE totalOrder, signed integers flip their sign bit (the same idea for
// two's complement), and descending order ([PMPP10] section 8, exercise 6)
// complements the mapped key, which keeps equal keys in input order.
// Intermediate passes move the mapped keys.  64-bit keys take 8 passes of
// radix 256 ([PMPP10] section 8, exercise 2).
//
// Differences from the pages' kernels: the in-tile rank comes from a warp
// multisplit (peer mask of equal digits + popcount below the lane) instead of
// eight block-wide 1-bit splits; a tile counts its digits first (cheap shared
// atomics) and publishes the counts before ranking, so its look-back overlaps
// other warps' ranking, and the per-warp counters then hand out tile slots
// directly; look-back words are cleared one row per tile by the previous
// kernel instead of a memset per pass; every wait is bounded.
//
// Keys-only sorts over every bit of the key need less than full stability:
// equal keys are identical, so a pass must keep the input order only between
// keys that differ in the bits below its digit (by which its input is already
// sorted).  Hence (both give the same output as the stable sort):
//   - the first pass (k_digit_pass_free) ranks by one shared atomic per key
//     and reserves each tile's places in the bins with atomic bin cursors, no
//     multisplit and no look-back;
//   - in later passes a warp whose keys agree below the digit (or take two
//     values there) ranks by shared atomics instead of the multisplit;
//   - where such runs are short (most warps stable), the multisplit's peer
//     masks come from shared OR-reductions into per-warp tables (kMatchRedOr)
//     instead of ballots: less integer work, more shared-memory traffic.
#pragma once

#include <algorithm>
#include <type_traits>

#include "gsort_internal.cuh"

namespace gsort {

// Arguments of one digit pass.  Key arrays hold 32- or 64-bit words (the
// kernel's key type); values are 32-bit.
struct PassArgs {
    const void *src_k;
    void *dst_k;
    const uint32_t *src_v;
    uint32_t *dst_v;
    uint32_t n;
    uint32_t shift;         // digit = (key >> shift) & mask
    uint32_t mask;
    uint64_t fmask;         // order map: all ones for float keys, else 0
    uint64_t flip;          // order map: bits flipped after the float map
    const uint32_t *hist;   // the 256 counts of this pass
    uint32_t *look;         // [tiles][256] look-back words of this pass (cleared): flag | count
    uint32_t *look_clear;   // next pass's words: row `tile` is cleared here; may be null
    uint32_t *tile_counter;
    uint32_t *status;
    uint32_t *abort_flag;
    uint32_t spin_limit;
    uint32_t stall_tile;
    uint32_t prefetch_dist;  // a CTA asks L2 for the keys of tile (its tile + this); 0: off
    // Keys-only sort over every bit of the key: a warp whose keys all agree
    // in the bits `free_low` (the bits below this pass's digit, by which the
    // input is already sorted) may rank them in any order, since such keys
    // with one digit agree in every bit sorted so far.
    uint32_t order_free = 0;
    uint64_t free_low = 0;
    // Non-zero: a warp whose keys take two values in `free_low` may rank in
    // two order-free rounds (worth testing only where runs are long).
    uint32_t two_runs_ok = 0;
    // Non-null (first pass of such a sort, where every warp is order-free):
    // any tile may take any place inside a digit's bin, so a tile reserves
    // its places with one atomic add per digit on these 256 bin cursors
    // (each set to its bin's start) instead of looking back, and takes its
    // tile by block index.
    uint32_t *cursor = nullptr;
    // Non-null: the bin starts of this pass (the exclusive scan of `hist`,
    // written by the histogram kernel), so that no tile scans the 256 counts again.
    const uint32_t *start = nullptr;
    // Non-null: the pass's most frequent digit if it holds more than 1/8 of
    // the keys, else 256 (written by the histogram kernel).
    const uint32_t *hot = nullptr;
};

// Launch of one digit pass over `tiles` tiles (one configuration of the kernel).
using PassLauncher = cudaError_t (*)(const PassArgs &, bool pairs, bool xin, bool xout,
                                     uint32_t tiles, cudaStream_t);

// Where the histogram kernel's last CTA writes what the passes need from the
// finished histogram (all null: nothing): the bin starts of every pass, the
// first pass's bin cursors set to its bin starts (null: none), each pass's
// skewed digit (256: none), and a zeroed counter of finished CTAs.
struct BinStartsOut {
    uint32_t *start = nullptr;
    uint32_t *cursor = nullptr;
    uint32_t *hot = nullptr;
    uint32_t *done = nullptr;
};

// 64-bit keys (radix64.cu): the digit pass, its tile size, and the histogram.
cudaError_t launch_pass_u64(const PassArgs &a, bool pairs, bool xin, bool xout, uint32_t tiles,
                            cudaStream_t s);
cudaError_t launch_pass_u64_free(const PassArgs &a, bool pairs, bool xin, bool xout, uint32_t tiles,
                                 cudaStream_t s);
uint32_t pass_tile_u64();
cudaError_t launch_hist_u64(const uint64_t *keys, uint32_t n, bool xf, uint64_t fmask, uint64_t flip,
                            int begin_bit, int passes, uint32_t last_mask, uint32_t *hist,
                            uint32_t *clear, uint32_t clear_words, cudaStream_t s, int sm_count,
                            const BinStartsOut &bs);

namespace {

// ------------------------------------------------------------- order map
// ordered = (float ? float_map(bits) : bits) ^ flip, where float_map flips
// every bit of a negative value and only the sign bit of a non-negative one.
template <class K>
__device__ __forceinline__ K order_in(K bits, K fmask, K flip) {
    using S = typename std::conditional<sizeof(K) == 8, int64_t, int32_t>::type;
    constexpr K sign = K(1) << (8 * sizeof(K) - 1);
    const K m = static_cast<K>(static_cast<S>(bits) >> (8 * sizeof(K) - 1)) | sign;
    return bits ^ (m & fmask) ^ flip;
}

// Inverse of order_in.
template <class K>
__device__ __forceinline__ K order_out(K u, K fmask, K flip) {
    using S = typename std::conditional<sizeof(K) == 8, int64_t, int32_t>::type;
    constexpr K sign = K(1) << (8 * sizeof(K) - 1);
    const K y = u ^ flip;
    const K m = static_cast<K>(static_cast<S>(~y) >> (8 * sizeof(K) - 1)) | sign;
    return y ^ (m & fmask);
}

// Digit of key k at bit `shift`.  BYTE: the digit is a whole byte of the key
// (shift a multiple of 8, full 8-bit mask), extracted with one byte permute.
template <bool BYTE>
__device__ __forceinline__ uint32_t digit_at(uint32_t k, uint32_t shift, uint32_t mask) {
    if constexpr (BYTE) return __byte_perm(k, 0u, 0x4440u | (shift >> 3));
    else return (k >> shift) & mask;
}

template <bool BYTE>
__device__ __forceinline__ uint32_t digit_at(uint64_t k, uint32_t shift, uint32_t mask) {
    if constexpr (BYTE) {
        const uint32_t w = (shift & 32u) ? static_cast<uint32_t>(k >> 32) : static_cast<uint32_t>(k);
        return __byte_perm(w, 0u, 0x4440u | ((shift & 31u) >> 3));
    } else {
        return static_cast<uint32_t>(k >> shift) & mask;
    }
}

// -------------------------------------------------------------- init
__global__ void k_zero_words(uint32_t *p, uint32_t nwords) {
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < nwords;
         i += gridDim.x * blockDim.x)
        p[i] = 0;
}

// -------------------------------------------------------------- histogram
// Every lane owns a private column of counters, so the shared-memory atomics
// of a warp never conflict, whatever the keys (equal keys included).  One
// 1024-thread CTA per SM; the columns are summed once per CTA and added to
// the global histogram.
//   32-bit keys: counter (pass, digit, lane) at word ((pass*256 + digit)*32 +
//                lane), up to 4 passes: 128 KiB.
//   64-bit keys: 16-bit counters, two digits per word: (pass, digit) in half
//                (digit & 1) of word ((pass*128 + digit/2)*32 + lane), up to 8
//                passes: 128 KiB.  A lane counts at most ceil(n / (grid *
//                1024)) keys, far below 2^16 for n <= 2^30 and the grid below.
constexpr int kHistThreads = 1024;
constexpr int kHistUnroll = 4;    // 16-byte loads in flight per thread
constexpr size_t kHistSmemBytes = 4 * 256 * 32 * sizeof(uint32_t);

template <bool XF, bool BYTE>
__device__ __forceinline__ void hist_count(uint32_t *col, uint32_t k, uint32_t begin_bit,
                                           int passes, uint32_t last_mask, uint32_t fmask,
                                           uint32_t flip) {
    if (XF) k = order_in<uint32_t>(k, fmask, flip);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        if (p < passes) {
            const uint32_t d = digit_at<BYTE>(k, begin_bit + 8 * p, p == passes - 1 ? last_mask : 0xFFu);
            atomicAdd(&col[(p * 256 + d) * 32], 1u);
        }
    }
}

template <bool XF, bool BYTE>
__device__ __forceinline__ void hist_count(uint32_t *col, uint64_t k, uint32_t begin_bit,
                                           int passes, uint32_t last_mask, uint64_t fmask,
                                           uint64_t flip) {
    if (XF) k = order_in<uint64_t>(k, fmask, flip);
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        if (p < passes) {
            const uint32_t d = digit_at<BYTE>(k, begin_bit + 8 * p, p == passes - 1 ? last_mask : 0xFFu);
            atomicAdd(&col[(p * 128 + (d >> 1)) * 32], 1u << ((d & 1u) * 16u));
        }
    }
}

// The finished histogram's bin starts ([CUDA3] kernel 2; [PMPP10] 10.3), the
// first pass's bin cursors and each pass's skewed digit, computed by the
// histogram kernel's last CTA (kHistThreads threads: four passes at a time,
// 256 threads per pass, one digit each).  `scratch` holds 64 words.
__device__ __forceinline__ void bin_starts_block(const uint32_t *hist, int passes, uint32_t n,
                                                 const BinStartsOut &bs, uint32_t *scratch) {
    const uint32_t tid = threadIdx.x, lane = tid & 31, g = tid >> 8, wg = (tid >> 5) & 7, d = tid & 255;
    uint32_t *s_sum = scratch;        // [4][8]
    uint32_t *s_top = scratch + 32;   // [4][8]: (count << 8 | 255 - digit) of each warp's largest bin
    for (int p0 = 0; p0 < passes; p0 += 4) {
        const int p = p0 + static_cast<int>(g);
        const uint32_t h = p < passes ? __ldcg(hist + p * 256 + d) : 0u;
        const uint32_t inc = warp_inclusive_scan(h, lane);
        // the largest count first (a bin may hold every key, so no digit fits
        // beside it in one word), then the lowest digit holding it
        uint32_t m = h;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(kFullMask, m, o));
        if (lane == 31) s_sum[g * 8 + wg] = inc;
        if (lane == 0) s_top[g * 8 + wg] = m;
        __syncthreads();
        uint32_t base = 0, top = 0;
        for (uint32_t w = 0; w < 8; ++w) {
            if (w < wg) base += s_sum[g * 8 + w];
            top = max(top, s_top[g * 8 + w]);
        }
        __syncthreads();
        if (p < passes) {
            const uint32_t st = base + inc - h;
            bs.start[p * 256 + d] = st;
            if (p == 0 && bs.cursor != nullptr) bs.cursor[d] = st;
            // skewed only when one digit holds more than 1/8 of the keys (32x its
            // share among 256 equally likely digits); the lowest such digit
            if (top > n / 8u) {
                const uint32_t firsts = __ballot_sync(kFullMask, h == top);
                if (lane == 0) s_top[g * 8 + wg] = firsts ? wg * 32 + __ffs(firsts) - 1 : 256u;
            } else if (lane == 0) {
                s_top[g * 8 + wg] = 256u;
            }
        }
        __syncthreads();
        if (p < passes && d == 0) {
            uint32_t hd = 256u;
            for (uint32_t w = 0; w < 8; ++w) hd = min(hd, s_top[g * 8 + w]);
            bs.hot[p] = hd;
        }
        __syncthreads();
    }
}

template <class K, bool XF, bool BYTE>
__global__ void __launch_bounds__(kHistThreads, 1)
k_digit_hist(const K *__restrict__ keys, uint32_t n, uint32_t begin_bit, int passes,
             uint32_t last_mask, K fmask, K flip, uint32_t *__restrict__ hist,
             uint4 *__restrict__ clear, uint32_t clear_vec4, const BinStartsOut bs) {
    constexpr bool kWide = sizeof(K) == 8;
    constexpr uint32_t kPerVec = 16 / sizeof(K);   // keys per 16-byte load
    extern __shared__ uint32_t s_h[];
    const uint32_t tid = threadIdx.x;
    const uint32_t words = static_cast<uint32_t>(passes) * (kWide ? 128 : 256) * 32;
    for (uint32_t i = tid; i < words; i += kHistThreads) s_h[i] = 0;
    const uint32_t gtid = blockIdx.x * kHistThreads + tid;
    const uint32_t gstride = gridDim.x * kHistThreads;
    for (uint32_t i = gtid; i < clear_vec4; i += gstride) clear[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();

    uint32_t *col = s_h + (tid & 31);
    // elements before the first 16-byte boundary, the vector body, the tail
    uint32_t head = static_cast<uint32_t>(((16 - (reinterpret_cast<uintptr_t>(keys) & 15)) & 15) / sizeof(K));
    head = min(head, n);
    const uint32_t nvec = (n - head) / kPerVec;
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
                if constexpr (kWide) {
                    const uint64_t a = (static_cast<uint64_t>(q[u].y) << 32) | q[u].x;
                    const uint64_t b = (static_cast<uint64_t>(q[u].w) << 32) | q[u].z;
                    hist_count<XF, BYTE>(col, a, begin_bit, passes, last_mask, fmask, flip);
                    hist_count<XF, BYTE>(col, b, begin_bit, passes, last_mask, fmask, flip);
                } else {
                    hist_count<XF, BYTE>(col, q[u].x, begin_bit, passes, last_mask, fmask, flip);
                    hist_count<XF, BYTE>(col, q[u].y, begin_bit, passes, last_mask, fmask, flip);
                    hist_count<XF, BYTE>(col, q[u].z, begin_bit, passes, last_mask, fmask, flip);
                    hist_count<XF, BYTE>(col, q[u].w, begin_bit, passes, last_mask, fmask, flip);
                }
            }
        }
    }
    const uint32_t tail0 = head + nvec * kPerVec;
    if (gtid < head) hist_count<XF, BYTE>(col, keys[gtid], begin_bit, passes, last_mask, fmask, flip);
    if (gtid < n - tail0)
        hist_count<XF, BYTE>(col, keys[tail0 + gtid], begin_bit, passes, last_mask, fmask, flip);
    __syncthreads();

    // sum each (pass, digit) row over the 32 lane columns; the rotated start
    // keeps the 32 threads of a warp on 32 different banks
    for (uint32_t i = tid; i < static_cast<uint32_t>(passes) * 256; i += kHistThreads) {
        uint32_t s = 0;
        if constexpr (kWide) {
            const uint32_t row = (i >> 8) * 128 + ((i & 255u) >> 1), half = (i & 1u) * 16u;
#pragma unroll 8
            for (uint32_t j = 0; j < 32; ++j) s += (s_h[row * 32 + ((j + row) & 31)] >> half) & 0xFFFFu;
        } else {
#pragma unroll 8
            for (uint32_t j = 0; j < 32; ++j) s += s_h[i * 32 + ((j + i) & 31)];
        }
        if (s) atomicAdd(&hist[i], s);
    }
    if (bs.done == nullptr) return;
    // the last CTA to finish finds the histogram complete: every CTA's adds
    // are ordered before its count of finished CTAs by the fence
    __threadfence();
    __syncthreads();
    if (tid == 0) s_h[0] = atomicAdd(bs.done, 1u) == gridDim.x - 1 ? 1u : 0u;
    __syncthreads();
    if (s_h[0] == 0u) return;
    __threadfence();
    __syncthreads();
    bin_starts_block(hist, passes, n, bs, s_h + 32);
}

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
constexpr int kMatchTable = 0, kMatchSelect = 1, kMatchAny = 2, kMatchRedOr = 3;
// kMatchRedOr: each lane ORs its lane bit into a per-warp shared table entry
// of its digit (a reduction, no value returned), reads the entry back after a
// warp barrier, and the group's leader clears it.

// Shared words of the per-warp peer tables of kMatchRedOr (after the misc words).
template <int WARPS, int MATCH>
__host__ __device__ constexpr size_t peer_table_words() {
    return MATCH == kMatchRedOr ? static_cast<size_t>(WARPS) * 256 : 0;
}

__device__ __forceinline__ void red_or_shared(uint32_t *p, uint32_t v) {
    asm volatile("red.shared.or.b32 [%0], %1;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(v)
                 : "memory");
}

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

// Next free slot of digit d for this lane's key, from counter table `tab`
// (order among the warp's keys of one digit is free).  `one_digit`: every lane
// of the warp holds digit d (runs of equal keys); one lane then reserves all
// 32 slots, because same-address shared atomics that return a value
// serialise across the lanes (reductions and distinct addresses do not).
__device__ __forceinline__ uint32_t take_slot(uint32_t *tab, uint32_t d, uint32_t lane, bool one_digit) {
    if (one_digit) {
        uint32_t base = 0;
        if (lane == 0) base = atomicAdd(&tab[d], 32u);
        return __shfl_sync(kFullMask, base, 0) + lane;
    }
    return atomicAdd(&tab[d], 1u);
}

// Next free slot of digit d for this lane's key (order free), where `hot` is
// the pass's most frequent digit: the lanes holding it take their slots with
// one atomic of the lowest such lane, since same-address atomics that return
// a value serialise across the lanes and skewed inputs can put a third of a
// warp's keys on one digit.  Lanes with valid == false take nothing (every
// lane of the warp must call this).
__device__ __forceinline__ uint32_t take_slot_hot(uint32_t *tab, uint32_t d, uint32_t hot, uint32_t lane,
                                                  bool valid) {
    const bool h = valid && d == hot;
    const uint32_t hm = __ballot_sync(kFullMask, h);
    uint32_t r = 0;
    if (hm != 0) {   // the same in every lane
        const uint32_t leader = __ffs(hm) - 1;
        uint32_t base = 0;
        if (lane == leader) base = atomicAdd(&tab[hot], static_cast<uint32_t>(__popc(hm)));
        r = __shfl_sync(kFullMask, base, leader) + __popc(hm & lanemask_lt());
    }
    if (valid && !h) r = atomicAdd(&tab[d], 1u);
    return r;
}

constexpr int kRow = 256;   // per-warp digit counters

template <class K, int WARPS, int IPT, bool PAIRS>
__host__ __device__ constexpr size_t pass_smem_words() {
    // keys [+ values] of the tile, per-warp counters, 256 digit offsets, 32 misc words
    return static_cast<size_t>(WARPS * 32 * IPT) * (sizeof(K) / 4 + (PAIRS ? 1 : 0)) + WARPS * kRow +
           256 + 32;
}

// Where one tile sits: its look-back row, the first row of its chain (the
// tiles first..row share one prefix: the whole input, or one segment), its
// keys, the 256 counts of the pass for its chain, and the output range.
struct TileDesc {
    uint32_t row;           // look-back row of this tile
    uint32_t first;         // look-back row of the chain's first tile
    uint32_t n;             // keys in this tile
    const uint32_t *hist;   // the chain's 256 digit counts of this pass
    uint32_t out_base;      // output index of the chain's first key
    uint32_t out_end;       // one past the chain's last output index
};

// Exclusive prefix of digit d over the tiles first .. row-1 of the chain.
// Each word holds a flag (AGG: the tile's count; PREFIX: the count over the
// chain's tiles up to this one) and a 30-bit count, so one round trip reads W
// predecessors at once; the nearest PREFIX word ends the walk and the AGG
// words before it are summed.  Returns false if a wait gave up.
template <int W>
__device__ __forceinline__ bool look_back(const PassArgs &a, const TileDesc &td, uint32_t d,
                                          uint32_t &excl) {
    excl = 0;
    int32_t t = static_cast<int32_t>(td.row) - 1;
    const int32_t first = static_cast<int32_t>(td.first);
    uint32_t polls = 0, ns = 32;
    while (true) {
        uint32_t w[W];
#pragma unroll
        for (int i = 0; i < W; ++i)
            w[i] = (t - i >= first) ? ld_relaxed(a.look + static_cast<uint32_t>(t - i) * 256 + d)
                                    : kFlagPrefix;   // before the chain: an empty prefix
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
// counters, digit offsets, misc words; the kernel sets misc word 2 to 0 and
// misc word 3 to the pass's skewed digit (256: none) before the call.  before_output() runs in every thread
// after the last block barrier, before the output phase.  Returns false when
// the tile stops (device error or the test stall), after that barrier.
struct NoHook {
    __device__ void operator()() const {}
};

template <class K, int WARPS, int IPT, int MATCH, int LW, bool BYTE, bool PAIRS, bool XIN, bool XOUT,
          bool FULL, class Hook = NoHook>
__device__ __forceinline__ bool pass_tile(const PassArgs &a, uint32_t *tab, const TileDesc &td,
                                          const K *kin, const uint32_t *vin,
                                          K *s_keys, uint32_t *s_vals,
                                          const Hook &before_output = Hook()) {
    constexpr int T = WARPS * 32;
    constexpr int TILE = T * IPT;
    uint32_t *s_cnt = tab;                      // [WARPS][256] counts, then next free slots
    uint32_t *s_goff = s_cnt + WARPS * kRow;    // [256] global index - tile slot
    uint32_t *s_misc = s_goff + 256;            // [32]

    const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t tile = td.row;
    const uint32_t tile_n = FULL ? TILE : td.n;
    // Item k of this thread sits at tile index item0 + 32k: each warp owns a
    // contiguous run of 32*IPT keys and walks it in order, which makes the
    // warp-local ranks stable.
    const uint32_t item0 = warp * (32 * IPT) + lane;
    K key[IPT];
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        const uint32_t i = item0 + k * 32;
        key[k] = (FULL || i < tile_n) ? kin[i] : K(0);
        if (XIN) key[k] = order_in<K>(key[k], static_cast<K>(a.fmask), static_cast<K>(a.flip));
    }
    uint32_t val[PAIRS ? IPT : 1];
    if (PAIRS) {
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            const uint32_t i = item0 + k * 32;
            val[k] = (FULL || i < tile_n) ? vin[i] : 0u;
        }
    }

    // ---- early counts: this warp's keys per digit (order does not matter
    // here); keys-only sorts also note whether all the warp's keys share a digit
    bool one_digit = false;
    {
        uint32_t *wc = s_cnt + warp * kRow;
        const uint32_t d0 = __shfl_sync(kFullMask, digit_at<BYTE>(key[0], a.shift, a.mask), 0);
        bool same = true;
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            if (FULL || item0 + k * 32 < tile_n) {
                const uint32_t d = digit_at<BYTE>(key[k], a.shift, a.mask);
                atomicAdd(&wc[d], 1u);
                same &= d == d0;
            }
        }
        if constexpr (!PAIRS && FULL) one_digit = __all_sync(kFullMask, same);
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
        if (tile != a.stall_tile && a.cursor == nullptr)
            st_relaxed(a.look + tile * 256 + tid, (tile == td.first ? kFlagPrefix : kFlagAgg) | cnt);
        const uint32_t ic = warp_inclusive_scan(cnt, lane);
        if (lane == 31) s_misc[4 + warp] = ic;
        tile_excl = ic - cnt;
        if (a.start != nullptr) {
            bin_excl = a.start[tid];
        } else {   // per-segment counts: scan them here
            const uint32_t bin = td.hist[tid];
            const uint32_t ib = warp_inclusive_scan(bin, lane);
            if (lane == 31) s_misc[12 + warp] = ib;
            bin_excl = ib - bin;
        }
    }
    if (a.look_clear != nullptr)
        for (uint32_t i = tid; i < 256; i += T) a.look_clear[tile * 256 + i] = 0;
    __syncthreads();
    if (tid < 256) {
        for (uint32_t w = 0; w < warp; ++w) {
            tile_excl += s_misc[4 + w];
            if (a.start == nullptr) bin_excl += s_misc[12 + w];
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
        if (a.cursor != nullptr) {
            if (cnt != 0 && tile != a.stall_tile) excl = atomicAdd(a.cursor + tid, cnt);
        } else if (tile > td.first && tile != a.stall_tile) {
            ok = look_back<LW>(a, td, tid, excl);
            if (ok) st_relaxed(a.look + tile * 256 + tid, kFlagPrefix | (excl + cnt));
        }
        if (!ok) {
            s_misc[2] = 1;
            record_error(a.status, a.abort_flag, GSORT_ETIMEOUT);
        }
        // global index of tile slot i holding digit d: s_goff[d] + i (a bin
        // cursor already holds its bin's start)
        s_goff[tid] = td.out_base + (a.cursor != nullptr ? 0u : bin_excl) + excl - tile_excl;
    }

    // ---- order-free warps: the warp's keys are sorted by the bits below this
    // digit (the earlier passes' order), so if its first and last keys agree
    // there, all of them do, and keys of one digit are interchangeable: each
    // takes the next free slot of its digit (one shared atomic, no ballots)
    // A warp whose keys take exactly two values in those bits (a run boundary
    // inside the warp) ranks in two rounds: every key of the first value,
    // then, after a warp barrier, every key of the second, so that the first
    // value's keys of each digit take the lower slots.
    bool order_free = false, two_runs = false;
    K low_first = 0;
    if constexpr (!PAIRS && FULL) {
        if (a.order_free) {
            const K fl = static_cast<K>(a.free_low);
            low_first = __shfl_sync(kFullMask, key[0], 0) & fl;
            const K low_last = __shfl_sync(kFullMask, key[IPT - 1], 31) & fl;
            order_free = low_first == low_last;
            if (!order_free && a.two_runs_ok) {
                bool two = true;
#pragma unroll
                for (int k = 0; k < IPT; ++k) {
                    const K lo = key[k] & fl;
                    two &= lo == low_first || lo == low_last;
                }
                order_free = two_runs = __all_sync(kFullMask, two);
            }
        }
    }
    if (order_free) {
        uint32_t *wc = s_cnt + warp * kRow;
        const uint32_t hot = s_misc[3];   // the pass's skewed digit (256: none), set by the kernel
        if (hot < 256u && !one_digit && !two_runs) {   // skewed digits (the same in every thread of the grid)
#pragma unroll
            for (int k = 0; k < IPT; ++k)
                s_keys[take_slot_hot(wc, digit_at<BYTE>(key[k], a.shift, a.mask), hot, lane, true)] = key[k];
        } else if (!two_runs) {
#pragma unroll
            for (int k = 0; k < IPT; ++k)   // order-free warps come from full tiles only
                s_keys[take_slot(wc, digit_at<BYTE>(key[k], a.shift, a.mask), lane, one_digit)] = key[k];
        } else {
            const K fl = static_cast<K>(a.free_low);
#pragma unroll
            for (int k = 0; k < IPT; ++k)
                if ((key[k] & fl) == low_first)
                    s_keys[atomicAdd(&wc[digit_at<BYTE>(key[k], a.shift, a.mask)], 1u)] = key[k];
            __syncwarp();   // the first run's slots are taken before the second run's
#pragma unroll
            for (int k = 0; k < IPT; ++k)
                if ((key[k] & fl) != low_first)
                    s_keys[atomicAdd(&wc[digit_at<BYTE>(key[k], a.shift, a.mask)], 1u)] = key[k];
        }
    } else
    // ---- warp multisplit: stable slot of each key in the tile-sorted order
    {
        uint32_t *wc = s_cnt + warp * kRow;
        const uint32_t ltm = lanemask_lt();
        const LaneConsts c = lane_consts(lane);
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            const bool valid = FULL || item0 + k * 32 < tile_n;
            const uint32_t d = valid ? digit_at<BYTE>(key[k], a.shift, a.mask) : 0u;
            uint32_t peers;
            if constexpr (MATCH == kMatchRedOr) {
                uint32_t *pt = s_misc + 32 + warp * 256;   // this warp's peer table (zero between items)
                if (valid) red_or_shared(&pt[d], 1u << lane);
                __syncwarp();
                peers = valid ? pt[d] : 0u;
                __syncwarp();   // every lane has read its entry before the leaders clear them
            } else {
                peers = digit_peers<MATCH>(d, c);
                if (!FULL) peers &= __ballot_sync(kFullMask, valid);
            }
            const uint32_t leader = highest_bit(peers);   // peers is empty only for padding lanes
            uint32_t base = 0;
            if (valid && lane == leader) {
                base = atomicAdd(&wc[d], static_cast<uint32_t>(__popc(peers)));
                if constexpr (MATCH == kMatchRedOr) s_misc[32 + warp * 256 + d] = 0u;
            }
            base = __shfl_sync(kFullMask, base, leader);
            if constexpr (MATCH == kMatchRedOr) __syncwarp();   // cleared before the next item's reductions
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
    K *dst_k = static_cast<K *>(a.dst_k);
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        const uint32_t i = k * T + tid;
        if (FULL || i < tile_n) {
            const K kk = s_keys[i];
            const uint32_t g = s_goff[digit_at<BYTE>(kk, a.shift, a.mask)] + i;
            if (g < td.out_end) {
                dst_k[g] = XOUT ? order_out<K>(kk, static_cast<K>(a.fmask), static_cast<K>(a.flip)) : kk;
                if (PAIRS) a.dst_v[g] = s_vals[i];
            }
        }
    }
    return true;
}

// The CTA that takes tile + prefetch_dist (about one CTA lifetime later)
// then finds its keys in L2 instead of waiting for HBM: one bulk L2 prefetch
// of that tile's keys (and values), issued by one thread.  Sources must be
// 16-byte aligned (prefetch_dist is 0 otherwise).
template <class K, int TILE, bool PAIRS>
__device__ __forceinline__ void prefetch_tile_l2(const PassArgs &a, uint32_t tile) {
    if (a.prefetch_dist == 0) return;
    const uint32_t pt = tile + a.prefetch_dist;
    if (pt >= (a.n + TILE - 1) / TILE) return;
    const uint32_t cnt = min(static_cast<uint32_t>(TILE), a.n - pt * TILE);
    const uint32_t kbytes = (cnt * static_cast<uint32_t>(sizeof(K))) & ~15u;
    if (kbytes)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                     ::"l"(static_cast<const K *>(a.src_k) + static_cast<size_t>(pt) * TILE), "r"(kbytes)
                     : "memory");
    const uint32_t vbytes = (cnt * 4u) & ~15u;
    if (PAIRS && vbytes)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                     ::"l"(a.src_v + static_cast<size_t>(pt) * TILE), "r"(vbytes) : "memory");
}

template <class K, int WARPS, int IPT, int MINB, int MATCH, int LW, bool BYTE, bool PAIRS, bool XIN,
          bool XOUT>
__global__ void __launch_bounds__(WARPS * 32, MINB) k_digit_pass(const PassArgs a) {
    constexpr int TILE = WARPS * 32 * IPT;
    extern __shared__ __align__(128) uint32_t smem[];
    uint32_t *s_misc = smem + pass_smem_words<K, WARPS, IPT, PAIRS>() - 32;
    const uint32_t tid = threadIdx.x;
    if (tid == 0) {
        // tiles in start order, so that a look-back always progresses; with
        // bin cursors no tile waits for another and the block index serves
        s_misc[0] = a.cursor != nullptr ? blockIdx.x : atomicAdd(a.tile_counter, 1u);
        s_misc[1] = ld_relaxed(a.abort_flag);
        s_misc[2] = 0;
        s_misc[3] = a.hot != nullptr ? *a.hot : 256u;
    }
    constexpr size_t kKeyWords = sizeof(K) / 4;
    uint32_t *s_cnt = smem + TILE * (kKeyWords + (PAIRS ? 1 : 0));
    for (uint32_t i = tid; i < WARPS * kRow; i += WARPS * 32) s_cnt[i] = 0;
    if constexpr (MATCH == kMatchRedOr)
        for (uint32_t i = tid; i < peer_table_words<WARPS, MATCH>(); i += WARPS * 32) s_misc[32 + i] = 0;
    __syncthreads();
    const uint32_t tile = s_misc[0];
    if (s_misc[1]) return;   // an earlier wait gave up; the result is void anyway
    if (tid == 0) prefetch_tile_l2<K, TILE, PAIRS>(a, tile);
    K *s_keys = reinterpret_cast<K *>(smem);
    uint32_t *s_vals = smem + TILE * kKeyWords;
    const K *kin = static_cast<const K *>(a.src_k) + tile * TILE;
    const uint32_t *vin = PAIRS ? a.src_v + tile * TILE : nullptr;
    const TileDesc td{tile, 0u, min(static_cast<uint32_t>(TILE), a.n - tile * TILE), a.hist, 0u, a.n};
    if (td.n == static_cast<uint32_t>(TILE))
        pass_tile<K, WARPS, IPT, MATCH, LW, BYTE, PAIRS, XIN, XOUT, true>(a, s_cnt, td, kin, vin, s_keys, s_vals);
    else
        pass_tile<K, WARPS, IPT, MATCH, LW, BYTE, PAIRS, XIN, XOUT, false>(a, s_cnt, td, kin, vin, s_keys, s_vals);
}

// One-tile-per-CTA launch configuration of the digit pass.
template <class K, int WARPS, int IPT, int MINB, int MATCH, int LW = 8>
struct PassConfig {
    static constexpr uint32_t kTile = WARPS * 32 * IPT;

    template <bool B, bool P, bool XI, bool XO>
    static cudaError_t launch_one(const PassArgs &a, uint32_t tiles, cudaStream_t s) {
        auto k = k_digit_pass<K, WARPS, IPT, MINB, MATCH, LW, B, P, XI, XO>;
        const size_t smem = (pass_smem_words<K, WARPS, IPT, P>() + peer_table_words<WARPS, MATCH>()) * sizeof(uint32_t);
        cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(k), smem);
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

    // Keys only (instantiates no pairs kernel).
    template <bool B>
    static cudaError_t launch_kb(const PassArgs &a, bool xin, bool xout, uint32_t tiles, cudaStream_t s) {
        if (xin) return xout ? launch_one<B, false, true, true>(a, tiles, s) : launch_one<B, false, true, false>(a, tiles, s);
        return xout ? launch_one<B, false, false, true>(a, tiles, s) : launch_one<B, false, false, false>(a, tiles, s);
    }

    static cudaError_t launch_keys(const PassArgs &a, bool pairs, bool xin, bool xout, uint32_t tiles,
                                   cudaStream_t s) {
        if (pairs) return cudaErrorInvalidValue;
        const bool byte = (a.shift % 8) == 0 && a.mask == 0xFFu;
        return byte ? launch_kb<true>(a, xin, xout, tiles, s) : launch_kb<false>(a, xin, xout, tiles, s);
    }
};

// ------------------------------------------- order-free first digit pass
// First pass of a keys-only sort over every bit of the key.  Equal keys are
// indistinguishable and no earlier pass fixed an order, so the keys of one
// digit may land in any order, within a tile and across tiles:
//   - one shared counter per digit for the whole tile; the atomic add that
//     counts a key also returns its rank among the tile's keys of its digit
//     (no per-warp tables, no warp-order scans, no multisplit);
//   - the tile reserves its places inside each digit's bin with one atomic
//     add per digit on 256 bin cursors (no look-back, no wait on any other
//     tile), and takes its tile by block index;
//   - the tile is reordered in shared memory and written as per-digit runs,
//     as in the stable pass;
//   - since the order inside the tile does not matter, a full, 16-byte
//     aligned tile comes in 16-byte loads ([CUDA3] vector access), and each
//     CTA asks L2 for the keys of the tile one CTA lifetime ahead.
// Shared memory: keys of the tile, 256 counts/tile offsets, 256 global
// offsets, 32 misc words.
template <class K, int WARPS, int IPT>
__host__ __device__ constexpr size_t free_pass_smem_words() {
    return static_cast<size_t>(WARPS * 32 * IPT) * (sizeof(K) / 4) + 256 + 256 + 32;
}

template <class K, int WARPS, int IPT, int MINB, bool BYTE, bool XIN, bool XOUT, bool VEC = true>
__global__ void __launch_bounds__(WARPS * 32, MINB) k_digit_pass_free(const PassArgs a) {
    static_assert(WARPS * 32 >= 256, "one thread per digit");
    static_assert(IPT % 2 == 0, "ranks are packed two per register");
    constexpr int T = WARPS * 32;
    constexpr int TILE = T * IPT;
    extern __shared__ __align__(128) uint32_t smem[];
    K *s_keys = reinterpret_cast<K *>(smem);
    uint32_t *s_cnt = smem + TILE * (sizeof(K) / 4);   // [256] counts, then tile offsets
    uint32_t *s_goff = s_cnt + 256;                    // [256] global index - tile slot
    uint32_t *s_misc = s_goff + 256;                   // [32]
    const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t tile = blockIdx.x;
    const uint32_t tile_n = min(static_cast<uint32_t>(TILE), a.n - tile * TILE);
    const K *kin = static_cast<const K *>(a.src_k) + static_cast<size_t>(tile) * TILE;

    const uint32_t hot = a.hot != nullptr ? *a.hot : 256u;   // the pass's skewed digit; 256: none
    // keys first (their latency overlaps the table set-up); the order of the
    // keys inside the tile does not matter here, so a full tile of 16-byte
    // aligned keys comes in 16-byte loads
    K key[IPT];
    constexpr int kPerVec = 16 / sizeof(K);
    if (VEC && tile_n == static_cast<uint32_t>(TILE) && (reinterpret_cast<uintptr_t>(kin) & 15) == 0) {
        const uint4 *kv = reinterpret_cast<const uint4 *>(kin);
#pragma unroll
        for (int j = 0; j < IPT / kPerVec; ++j) {
            const uint4 q = __ldcs(kv + j * T + tid);
            if constexpr (sizeof(K) == 4) {
                key[4 * j] = q.x;
                key[4 * j + 1] = q.y;
                key[4 * j + 2] = q.z;
                key[4 * j + 3] = q.w;
            } else {
                key[2 * j] = (static_cast<uint64_t>(q.y) << 32) | q.x;
                key[2 * j + 1] = (static_cast<uint64_t>(q.w) << 32) | q.z;
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            const uint32_t i = k * T + tid;
            key[k] = i < tile_n ? kin[i] : K(0);
        }
    }
    if (XIN) {
#pragma unroll
        for (int k = 0; k < IPT; ++k) key[k] = order_in<K>(key[k], static_cast<K>(a.fmask), static_cast<K>(a.flip));
    }
    if (tid < 256) s_cnt[tid] = 0;
    if (tid == 0) {
        s_misc[0] = ld_relaxed(a.abort_flag);
        prefetch_tile_l2<K, TILE, false>(a, tile);
    }
    __syncthreads();
    if (s_misc[0]) return;   // an earlier wait gave up; the result is void anyway

    // count and rank in one shared atomic per key (one per item when all the
    // warp's keys share a digit: presorted or constant input)
    bool one_digit = false;
    if (tile_n == static_cast<uint32_t>(TILE)) {   // tile-uniform
        const uint32_t d0 = __shfl_sync(kFullMask, digit_at<BYTE>(key[0], a.shift, a.mask), 0);
        bool same = true;
#pragma unroll
        for (int k = 0; k < IPT; ++k) same &= digit_at<BYTE>(key[k], a.shift, a.mask) == d0;
        one_digit = __all_sync(kFullMask, same);
    }
    uint32_t rk[IPT / 2];
    uint32_t hot_base = 0;
    if (hot < 256u && !one_digit) {   // the same in every thread of the grid
        // keys of the hot digit rank by this warp's running count of them, and
        // the warp reserves their slots with one atomic after the loop (their
        // order is free); bit 15 marks such a rank until then
        const uint32_t ltm = lanemask_lt();
        uint32_t run = 0;
#pragma unroll
        for (int k = 0; k < IPT; k += 2) {
            uint32_t r[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const bool valid = (k + u) * T + tid < tile_n;
                const uint32_t d = digit_at<BYTE>(key[k + u], a.shift, a.mask);
                const bool h = valid && d == hot;
                const uint32_t hm = __ballot_sync(kFullMask, h);
                r[u] = h ? (0x8000u | (run + __popc(hm & ltm))) : (valid ? atomicAdd(&s_cnt[d], 1u) : 0u);
                run += __popc(hm);
            }
            rk[k / 2] = r[0] | (r[1] << 16);
        }
        if (lane == 0 && run != 0) hot_base = atomicAdd(&s_cnt[hot], run);
        hot_base = __shfl_sync(kFullMask, hot_base, 0);
    } else {
#pragma unroll
        for (int k = 0; k < IPT; k += 2) {
            uint32_t r0 = 0, r1 = 0;
            if (one_digit) {
                r0 = take_slot(s_cnt, digit_at<BYTE>(key[k], a.shift, a.mask), lane, true);
                r1 = take_slot(s_cnt, digit_at<BYTE>(key[k + 1], a.shift, a.mask), lane, true);
            } else {
                if (k * T + tid < tile_n) r0 = atomicAdd(&s_cnt[digit_at<BYTE>(key[k], a.shift, a.mask)], 1u);
                if ((k + 1) * T + tid < tile_n)
                    r1 = atomicAdd(&s_cnt[digit_at<BYTE>(key[k + 1], a.shift, a.mask)], 1u);
            }
            rk[k / 2] = r0 | (r1 << 16);
        }
    }
    __syncthreads();

    // scan over the 256 digits: tile offsets (the bin starts are in the cursors)
    uint32_t cnt = 0, tile_excl = 0;
    if (tid < 256) {
        cnt = s_cnt[tid];
        const uint32_t ic = warp_inclusive_scan(cnt, lane);
        if (lane == 31) s_misc[4 + warp] = ic;
        tile_excl = ic - cnt;
    }
    __syncthreads();
    if (tid < 256) {
        for (uint32_t w = 0; w < warp; ++w) tile_excl += s_misc[4 + w];
        s_cnt[tid] = tile_excl;
    }
    __syncthreads();

    // reserve the tile's places in the bins (in flight during the reorder)
    uint32_t excl = 0;
    if (tid < 256 && cnt != 0 && tile != a.stall_tile) excl = atomicAdd(a.cursor + tid, cnt);
    if (a.look_clear != nullptr)
        for (uint32_t i = tid; i < 256; i += T) a.look_clear[tile * 256 + i] = 0;
    if (hot < 256u && !one_digit) {
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            if (k * T + tid < tile_n) {
                uint32_t r = (rk[k / 2] >> ((k & 1) * 16)) & 0xFFFFu;
                if (r & 0x8000u) r = hot_base + (r & 0x7FFFu);
                s_keys[s_cnt[digit_at<BYTE>(key[k], a.shift, a.mask)] + r] = key[k];
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            if (k * T + tid < tile_n) {
                const uint32_t r = (rk[k / 2] >> ((k & 1) * 16)) & 0xFFFFu;
                s_keys[s_cnt[digit_at<BYTE>(key[k], a.shift, a.mask)] + r] = key[k];
            }
        }
    }
    if (tid < 256) s_goff[tid] = excl - tile_excl;   // the cursor started at the bin's start
    __syncthreads();
    if (tile == a.stall_tile) return;

    // contiguous runs per digit out to global memory
    K *dst_k = static_cast<K *>(a.dst_k);
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        const uint32_t i = k * T + tid;
        if (i < tile_n) {
            const K kk = s_keys[i];
            const uint32_t g = s_goff[digit_at<BYTE>(kk, a.shift, a.mask)] + i;
            if (g < a.n) dst_k[g] = XOUT ? order_out<K>(kk, static_cast<K>(a.fmask), static_cast<K>(a.flip)) : kk;
        }
    }
}

// Launch configuration of the order-free first pass (k_digit_pass_free).
// Its tile must not exceed the next pass's, so that clearing row `tile` of
// the next pass's look-back words covers every row that pass uses.
template <class K, int WARPS, int IPT, int MINB>
struct FreePassConfig {
    static constexpr uint32_t kTile = WARPS * 32 * IPT;

    template <bool B, bool XI, bool XO>
    static cudaError_t launch_one(const PassArgs &a, uint32_t tiles, cudaStream_t s) {
        auto k = k_digit_pass_free<K, WARPS, IPT, MINB, B, XI, XO>;
        const size_t smem = free_pass_smem_words<K, WARPS, IPT>() * sizeof(uint32_t);
        cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(k), smem);
        if (e != cudaSuccess) return e;
        k<<<tiles, WARPS * 32, smem, s>>>(a);
        return cudaGetLastError();
    }

    template <bool B>
    static cudaError_t launch_b(const PassArgs &a, bool xin, bool xout, uint32_t tiles, cudaStream_t s) {
        if (xin) return xout ? launch_one<B, true, true>(a, tiles, s) : launch_one<B, true, false>(a, tiles, s);
        return xout ? launch_one<B, false, true>(a, tiles, s) : launch_one<B, false, false>(a, tiles, s);
    }

    // `tiles` counts tiles of kTile keys.
    static cudaError_t launch(const PassArgs &a, bool pairs, bool xin, bool xout, uint32_t tiles,
                              cudaStream_t s) {
        if (pairs || a.cursor == nullptr) return cudaErrorInvalidValue;
        const bool byte = (a.shift % 8) == 0 && a.mask == 0xFFu;
        return byte ? launch_b<true>(a, xin, xout, tiles, s) : launch_b<false>(a, xin, xout, tiles, s);
    }
};

// Histogram launch: one CTA per SM (fewer for small inputs: about 16 keys per
// thread at least).
template <class K>
cudaError_t launch_hist_kernel(const K *keys, uint32_t n, bool xf, K fmask, K flip, int begin_bit,
                               int passes, uint32_t last_mask, uint32_t *hist, uint32_t *clear,
                               uint32_t clear_words, cudaStream_t s, int sm_count,
                               const BinStartsOut &bs = BinStartsOut()) {
    const uint32_t want = (n + kHistThreads * 16 - 1) / (kHistThreads * 16);
    const uint32_t grid = std::max(1u, std::min(want, static_cast<uint32_t>(sm_count)));
    uint4 *cl = reinterpret_cast<uint4 *>(clear);
    const bool byte = (begin_bit % 8) == 0 && last_mask == 0xFFu;
    auto k = xf ? (byte ? k_digit_hist<K, true, true> : k_digit_hist<K, true, false>)
                : (byte ? k_digit_hist<K, false, true> : k_digit_hist<K, false, false>);
    const size_t smem = static_cast<size_t>(passes) * (sizeof(K) == 8 ? 128 : 256) * 32 * sizeof(uint32_t);
    cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(k), kHistSmemBytes);
    if (e != cudaSuccess) return e;
    k<<<grid, kHistThreads, smem, s>>>(keys, n, begin_bit, passes, last_mask, fmask, flip, hist, cl,
                                       clear_words / 4, bs);
    return cudaGetLastError();
}

}  // namespace
}  // namespace gsort

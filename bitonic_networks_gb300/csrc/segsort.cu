// segsort.cu -- stable sort of variable-length segments (an offsets array),
// the hybrid strategy of [PMPP10] 10.5 (strategy 2: radix sort for the
// coarse order, bitonic networks for small pieces) and of [GPUSORT]
// (partitioned sort whose pieces of <= 1024 keys go to a bitonic sort):
//
//   classify   one pass over the segments: checks the offsets, lists the
//              segments of 2..1024 keys ("small") and of more than 1024 keys
//              ("large"), copies segments of one key when the output is
//              another buffer
//   scan       exclusive scan of the tile counts of the large segments: the
//              tiles of segment j are rows tile_base[j] .. tile_base[j+1]-1
//   tilemap    one descriptor per tile (its segment, keys, look-back chain);
//              clears each large segment's counts
//   histogram  the 4 x 256 digit counts of every large segment, and the
//              first pass's look-back rows cleared
//   4 x pass   the single-pass digit scatter of radix_kernels.cuh on tiles
//              that never straddle a segment: bin starts come from the
//              segment's own histogram, and the decoupled look-back of a tile
//              stops at its segment's first tile (a chain per segment); the
//              first pass of keys only reserves places on per-segment bin
//              cursors instead
//   small      one warp per small segment: the register bitonic network of
//              bitonic_network.cuh; with values, the network sorts (key,
//              position) composites, which makes the result stable.  These
//              kernels run on side streams, beside the large segments' ones
//
// Every segment is sorted by the whole mapped key (the order map of the key
// kind and direction, as in the radix sort), equal keys keeping their input
// order, so the result is unique with or without values.
#include <mutex>

#include "bitonic_network.cuh"
#include "radix_kernels.cuh"

namespace gsort {
namespace {

constexpr uint32_t kSmallMax = 1024;                  // longest segment the warp network takes
constexpr int kSegPassWarps = 16, kSegPassIpt = 16;
constexpr uint32_t kSegTile = kSegPassWarps * 32 * kSegPassIpt;   // 8192 keys
constexpr int kSmallWarps = 4;

// Header words (after the tile counters): list lengths and the tile total.
constexpr size_t kHdrSegCounts = kHdrHist;   // u32 [0] small, [1] large, [2] tiles

// Descriptor of one tile of a large segment (32 bytes: two 16-byte loads).
struct SegTile {
    uint32_t seg;        // index into the large-segment arrays
    uint32_t base;       // index of the tile's first key
    uint32_t n;          // keys in the tile
    uint32_t first;      // look-back row of the segment's first tile
    uint32_t out_base;   // the segment's first index
    uint32_t out_end;    // one past the segment's last index
    uint32_t pad[2];
};

// ---------------------------------------------------------------- classify
__global__ void k_seg_classify(const uint32_t *__restrict__ offsets, uint32_t num_segments,
                               uint32_t n, uint32_t *small_list, uint32_t small_max,
                               uint32_t *large_start, uint32_t *large_len, uint32_t large_max,
                               const uint32_t *keys_in, uint32_t *keys_out,
                               const uint32_t *vals_in, uint32_t *vals_out, uint32_t *counts,
                               uint32_t *status, uint32_t *abort_flag) {
    for (uint32_t s = blockIdx.x * blockDim.x + threadIdx.x; s < num_segments;
         s += gridDim.x * blockDim.x) {
        const uint32_t a = offsets[s], b = offsets[s + 1];
        const bool bad = b < a || b > n || (s == 0 && a != 0) || (s == num_segments - 1 && b != n);
        if (bad) {
            record_error(status, abort_flag, GSORT_EINVAL);
            continue;
        }
        const uint32_t len = b - a;
        if (len > kSmallMax) {
            const uint32_t j = atomicAdd(&counts[1], 1u);
            if (j >= large_max) {   // only reachable with overlapping (invalid) segments
                record_error(status, abort_flag, GSORT_EINVAL);
                continue;
            }
            large_start[j] = a;
            large_len[j] = len;
        } else if (len >= 2) {
            const uint32_t j = atomicAdd(&counts[0], 1u);
            if (j >= small_max) {
                record_error(status, abort_flag, GSORT_EINVAL);
                continue;
            }
            small_list[j] = s;
        } else if (len == 1 && keys_out != keys_in) {
            keys_out[a] = keys_in[a];
            if (vals_out != nullptr) vals_out[a] = vals_in[a];
        } else if (len == 1 && vals_out != nullptr && vals_out != vals_in) {
            vals_out[a] = vals_in[a];
        }
    }
}

// -------------------------------------------------------------------- scan
// One CTA: exclusive scan of ceil(len / tile) over the large segments; each
// thread scans a contiguous chunk, the chunk totals are scanned across the CTA.
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads)
k_seg_scan(const uint32_t *large_len, uint32_t large_max, uint32_t tiles_max, uint32_t *tile_base,
           uint32_t *counts, uint32_t *status, uint32_t *abort_flag) {
    __shared__ uint32_t s_warp[32];
    __shared__ uint32_t s_total;
    const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool aborted = ld_relaxed(abort_flag) != 0;
    const uint32_t L = aborted ? 0u : min(counts[1], large_max);
    const uint32_t chunk = (L + kScanThreads - 1) / kScanThreads;
    const uint32_t lo = min(L, tid * chunk), hi = min(L, lo + chunk);
    uint32_t sum = 0;
    for (uint32_t j = lo; j < hi; ++j) sum += (large_len[j] + kSegTile - 1) / kSegTile;
    const uint32_t inc = warp_inclusive_scan(sum, lane);
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const uint32_t w = s_warp[lane];
        const uint32_t wi = warp_inclusive_scan(w, lane);
        s_warp[lane] = wi - w;
        if (lane == 31) s_total = wi;
    }
    __syncthreads();
    uint32_t run = s_warp[warp] + inc - sum;
    for (uint32_t j = lo; j < hi; ++j) {
        tile_base[j] = run;
        run += (large_len[j] + kSegTile - 1) / kSegTile;
    }
    if (tid == 0) {
        uint32_t total = s_total;
        if (total > tiles_max) {   // only reachable with overlapping (invalid) segments
            record_error(status, abort_flag, GSORT_EINVAL);
            total = 0;
        }
        tile_base[L] = total;
        counts[2] = total;
    }
}

// ----------------------------------------------------------------- tilemap
// One warp per large segment writes the descriptors of its tiles and
// clears the segment's 4 x 256 digit counts.
__global__ void k_seg_tilemap(const uint32_t *large_start, const uint32_t *large_len,
                              const uint32_t *tile_base, const uint32_t *counts, uint32_t large_max,
                              SegTile *tiles, uint4 *hist, const uint32_t *abort_flag) {
    if (ld_relaxed(abort_flag)) return;
    const uint32_t L = min(counts[1], large_max);
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t warps = gridDim.x * (blockDim.x >> 5);
    for (uint32_t j = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); j < L; j += warps) {
        const uint32_t a = large_start[j], len = large_len[j], first = tile_base[j];
        const uint32_t nt = (len + kSegTile - 1) / kSegTile;
        for (uint32_t k = lane; k < nt; k += 32) {
            SegTile t;
            t.seg = j;
            t.base = a + k * kSegTile;
            t.n = min(kSegTile, len - k * kSegTile);
            t.first = first;
            t.out_base = a;
            t.out_end = a + len;
            t.pad[0] = t.pad[1] = 0;
            tiles[first + k] = t;
        }
        for (uint32_t i = lane; i < 256; i += 32) hist[j * 256 + i] = make_uint4(0, 0, 0, 0);
    }
}

// --------------------------------------------------------------- histogram
// Each CTA takes a contiguous run of tiles (the same number for every CTA).
// The tiles of one segment are consecutive rows over consecutive keys, so the
// run splits into pieces, one per segment it touches, each a contiguous key
// range.  A piece's keys are counted in shared memory, four digits each, one
// column of counters per lane (conflict-free adds), the aligned body in
// 16-byte loads; after the piece, the columns are summed into the segment's
// histogram (one global add per non-zero count).  The next pieces' keys, and
// a long piece's keys two rounds ahead, are asked into L2 meanwhile.  The
// CTA also clears the look-back rows of its tiles for the first pass.
constexpr int kSegHistThreads = 1024, kSegHistUnroll = 4;   // 16-byte loads in flight per thread
constexpr uint32_t kSegHistAhead = 8;                           // tiles prefetched past a piece
constexpr size_t kSegHistSmem = 1024 * 32 * sizeof(uint32_t);  // [p * 256 + d][32 lanes]

template <bool XF>
__device__ __forceinline__ void seg_hist_count(uint32_t *col, uint32_t k, uint32_t fmask, uint32_t flip) {
    const uint32_t kk = XF ? order_in<uint32_t>(k, fmask, flip) : k;
#pragma unroll
    for (int p = 0; p < 4; ++p) atomicAdd(&col[(p * 256 + ((kk >> (8 * p)) & 0xFFu)) * 32], 1u);
}

// Counter c (digit word p * 256 + d) of thread c summed over its 32 lane
// columns (eight 16-byte words, read in an order rotated by the thread so
// that each quarter-warp's reads fall in distinct banks) and cleared.
__device__ __forceinline__ void seg_hist_flush(uint32_t *s_h, uint32_t *h, uint32_t tid) {
    uint4 *row = reinterpret_cast<uint4 *>(s_h + tid * 32);
    uint32_t c = 0;
#pragma unroll
    for (uint32_t j = 0; j < 8; ++j) {
        const uint32_t q = (j + tid) & 7u;
        const uint4 v = row[q];
        c += v.x + v.y + v.z + v.w;
        row[q] = make_uint4(0, 0, 0, 0);
    }
    if (c != 0) atomicAdd(h + tid, c);
}

// L2 prefetch of bytes [lo, hi) of the keys, rounded inwards to 16 bytes
// (keys 16-byte aligned), in pieces of at most 32 KiB.
__device__ __forceinline__ void seg_hist_prefetch(const uint32_t *keys, uint64_t lo, uint64_t hi) {
    lo = (lo + 15u) & ~15ull;
    hi &= ~15ull;
    for (; lo < hi; lo += 32768u) {
        const uint32_t bytes = static_cast<uint32_t>(min(hi - lo, static_cast<uint64_t>(32768u)));
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                     ::"l"(reinterpret_cast<const char *>(keys) + lo), "r"(bytes) : "memory");
    }
}

template <bool XF>
__global__ void __launch_bounds__(kSegHistThreads, 1)
k_seg_hist(const uint32_t *__restrict__ keys, const SegTile *tiles, const uint32_t *counts,
           uint32_t fmask, uint32_t flip, uint32_t *hist, uint32_t *look_clear,
           const uint32_t *abort_flag) {
    static_assert(kSegHistThreads == 1024, "one thread per digit word in the flush");
    constexpr uint32_t T = kSegHistThreads;
    extern __shared__ __align__(16) uint32_t s_h[];
    if (ld_relaxed(abort_flag)) return;
    const uint32_t total = counts[2];
    const uint32_t per = (total + gridDim.x - 1) / gridDim.x;
    const uint32_t t0 = min(total, blockIdx.x * per), t1 = min(total, t0 + per);
    if (t0 >= t1) return;   // uniform
    const uint32_t tid = threadIdx.x;
    for (uint32_t i = tid; i < 1024 * 32 / 4; i += T) reinterpret_cast<uint4 *>(s_h)[i] = make_uint4(0, 0, 0, 0);
    {
        uint4 *lc = reinterpret_cast<uint4 *>(look_clear + static_cast<size_t>(t0) * 256);
        for (uint32_t i = tid; i < (t1 - t0) * 64; i += T) lc[i] = make_uint4(0, 0, 0, 0);
    }
    uint32_t *col = s_h + (tid & 31u);
    const bool vec = (reinterpret_cast<uintptr_t>(keys) & 15u) == 0;
    // the piece starting at tile t: tiles t .. te-1, all of one segment, keys
    // [a, b), the 16-byte aligned body [a4, a4 + 4 nv)
    struct Piece {
        uint32_t seg, te, a, b, a4, nv;
    };
    auto piece_at = [&](uint32_t t) {
        const SegTile d = tiles[t];
        const uint32_t seg_tiles = (d.out_end - d.out_base + kSegTile - 1) / kSegTile;
        Piece P;
        P.seg = d.seg;
        P.te = min(t1, d.first + seg_tiles);
        P.a = d.base;
        P.b = min(d.out_end, d.base + (P.te - t) * kSegTile);
        P.a4 = P.a;
        uint32_t b4 = P.a;
        if (vec) {
            P.a4 = min(P.b, (P.a + 3u) & ~3u);
            b4 = max(P.a4, P.b & ~3u);
        }
        P.nv = (b4 - P.a4) / 4;
        return P;
    };
    // the first round of a piece's body, loaded ahead (during the previous
    // piece's flush)
    uint4 q[kSegHistUnroll];
    auto load_round = [&](const Piece &P, uint32_t v) {
        const uint4 *kv = reinterpret_cast<const uint4 *>(keys + P.a4);
#pragma unroll
        for (int u = 0; u < kSegHistUnroll; ++u)
            if (v + u * T < P.nv) q[u] = __ldcs(kv + v + u * T);
    };
    Piece P = piece_at(t0);
    load_round(P, tid);
    __syncthreads();
    while (true) {
        // the next pieces' first tiles go to L2 while this piece is counted
        // (one descriptor and one bulk prefetch per lane of the last warp)
        if (vec && tid >= T - kSegHistAhead && P.te + (tid - (T - kSegHistAhead)) < t1) {
            const SegTile dn = tiles[P.te + (tid - (T - kSegHistAhead))];
            seg_hist_prefetch(keys, static_cast<uint64_t>(dn.base) * 4u, static_cast<uint64_t>(dn.base + dn.n) * 4u);
        }
        const uint32_t b4 = P.a4 + 4 * P.nv;
        if (tid < P.a4 - P.a) seg_hist_count<XF>(col, keys[P.a + tid], fmask, flip);
        for (uint32_t i = b4 + tid; i < P.b; i += T) seg_hist_count<XF>(col, keys[i], fmask, flip);
        for (uint32_t v = tid; v < P.nv; v += T * kSegHistUnroll) {
            if (v != tid) load_round(P, v);   // the first round is in registers already
            if (tid == 0) {   // a long piece: its body two rounds ahead
                const uint32_t ahead = v + 2u * T * kSegHistUnroll;   // uint4 index in the body
                if (ahead < P.nv) {
                    const uint32_t end = min(P.nv, ahead + T * kSegHistUnroll);
                    seg_hist_prefetch(keys, (static_cast<uint64_t>(P.a4) + ahead * 4ull) * 4u,
                                      (static_cast<uint64_t>(P.a4) + end * 4ull) * 4u);
                }
            }
#pragma unroll
            for (int u = 0; u < kSegHistUnroll; ++u) {
                if (v + u * T < P.nv) {
                    seg_hist_count<XF>(col, q[u].x, fmask, flip);
                    seg_hist_count<XF>(col, q[u].y, fmask, flip);
                    seg_hist_count<XF>(col, q[u].z, fmask, flip);
                    seg_hist_count<XF>(col, q[u].w, fmask, flip);
                }
            }
        }
        const bool more = P.te < t1;   // uniform
        Piece N{};
        if (more) {   // the next piece's descriptor and first round, in flight during the flush
            N = piece_at(P.te);
            load_round(N, tid);
        }
        __syncthreads();   // every count of the piece is in
        seg_hist_flush(s_h, hist + P.seg * 1024, tid);
        if (!more) break;
        __syncthreads();
        P = N;
    }
}

// -------------------------------------------------------------------- pass
// Persistent CTAs claim tiles in increasing order (a CTA finishes one tile
// before it claims the next), so the smallest unfinished tile can always
// complete its look-back, whose chain ends at its segment's first tile.
// MATCH: kMatchTable (ballot tables), or kMatchRedOr (peer masks from shared
// reductions, keys-only passes whose runs of equal low bits are short: cheaper
// on spread digits; its per-warp tables follow the misc words and stay zero
// between items).
template <bool BYTE, bool PAIRS, bool XIN, bool XOUT, int MATCH>
__global__ void __launch_bounds__(kSegPassWarps * 32, PAIRS ? 2 : 3)
k_seg_pass(const PassArgs a, const SegTile *tiles, const uint32_t *counts, const uint32_t *hist) {
    constexpr int T = kSegPassWarps * 32;
    constexpr int TILE = kSegTile;
    extern __shared__ __align__(128) uint32_t smem[];
    uint32_t *s_keys = smem;
    uint32_t *s_vals = smem + TILE;
    uint32_t *s_cnt = smem + TILE * (PAIRS ? 2 : 1);
    uint32_t *s_misc = s_cnt + kSegPassWarps * kRow + 256;
    const uint32_t tid = threadIdx.x;
    const uint32_t total = counts[2];
    if constexpr (MATCH == kMatchRedOr)
        for (uint32_t i = tid; i < peer_table_words<kSegPassWarps, MATCH>(); i += T) s_misc[32 + i] = 0;
    while (true) {
        if (tid == 0) {
            s_misc[0] = atomicAdd(a.tile_counter, 1u);
            s_misc[1] = ld_relaxed(a.abort_flag);
            s_misc[2] = 0;
            s_misc[3] = 256u;   // no skewed digit
        }
        for (uint32_t i = tid; i < kSegPassWarps * kRow; i += T) s_cnt[i] = 0;
        __syncthreads();
        const uint32_t t = s_misc[0];
        if (s_misc[1] || t >= total) return;   // uniform: every thread read the same words
        const SegTile d = tiles[t];
        const TileDesc td{t, d.first, d.n, hist + d.seg * 1024 + (a.shift / 8) * 256, d.out_base,
                          d.out_end};
        const uint32_t *kin = static_cast<const uint32_t *>(a.src_k) + d.base;
        const uint32_t *vin = PAIRS ? a.src_v + d.base : nullptr;
        bool ok;
        if (d.n == static_cast<uint32_t>(TILE))
            ok = pass_tile<uint32_t, kSegPassWarps, kSegPassIpt, MATCH, 8, BYTE, PAIRS, XIN, XOUT, true>(
                a, s_cnt, td, kin, vin, s_keys, s_vals);
        else
            ok = pass_tile<uint32_t, kSegPassWarps, kSegPassIpt, MATCH, 8, BYTE, PAIRS, XIN, XOUT, false>(
                a, s_cnt, td, kin, vin, s_keys, s_vals);
        if (!ok) return;   // a look-back gave up (the abort flag is raised)
        __syncthreads();   // the tile buffers are read out before the next tile reuses them
    }
}

// First pass of a keys-only sort of the large segments, where every order
// of the keys of one digit is right (no lower bits to keep in order): the
// order-free digit pass of the radix sort on one tile of one segment.  A key
// takes its slot in the tile with one shared atomic add (warp-aggregated for
// the segment's most frequent digit when it holds over 1/8 of the segment's
// keys, and for warps whose keys share one digit); the tile reserves its
// places in the segment's bins on the segment's 256 cursors, which count
// from 0 inside each bin, the bin starts coming from a scan of the segment's
// counts; no look-back.  One tile per CTA; CTAs past the tile count return.
// Shared memory: the tile's keys, 256 counts/tile offsets, 256 global
// offsets, 32 misc words.
template <bool XIN>
__global__ void __launch_bounds__(kSegPassWarps * 32, 3)
k_seg_pass_free(const PassArgs a, const SegTile *tiles, const uint32_t *counts, const uint32_t *hist) {
    constexpr int T = kSegPassWarps * 32, IPT = kSegPassIpt, TILE = kSegTile;
    static_assert(T >= 256 && IPT % 4 == 0, "one thread per digit; 16-byte loads");
    extern __shared__ __align__(128) uint32_t smem[];
    uint32_t *s_keys = smem;           // [TILE]
    uint32_t *s_cnt = smem + TILE;     // [256] counts, then tile offsets
    uint32_t *s_goff = s_cnt + 256;    // [256] global index - tile slot
    uint32_t *s_misc = s_goff + 256;   // [32]
    const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t t = blockIdx.x;
    if (t >= counts[2]) return;   // uniform
    const SegTile d = tiles[t];
    const uint32_t tile_n = d.n;
    const uint32_t *kin = static_cast<const uint32_t *>(a.src_k) + d.base;

    // keys first; their order inside the tile does not matter, so a full,
    // 16-byte aligned tile comes in 16-byte loads
    uint32_t key[IPT];
    if (tile_n == static_cast<uint32_t>(TILE) && (reinterpret_cast<uintptr_t>(kin) & 15) == 0) {
        const uint4 *kv = reinterpret_cast<const uint4 *>(kin);
#pragma unroll
        for (int j = 0; j < IPT / 4; ++j) {
            const uint4 q = __ldcs(kv + j * T + tid);
            key[4 * j] = q.x;
            key[4 * j + 1] = q.y;
            key[4 * j + 2] = q.z;
            key[4 * j + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            const uint32_t i = k * T + tid;
            key[k] = i < tile_n ? kin[i] : 0u;
        }
    }
    if (XIN) {
#pragma unroll
        for (int k = 0; k < IPT; ++k) key[k] = order_in<uint32_t>(key[k], a.fmask, a.flip);
    }
    // the segment's counts of this digit; each warp of the first 8 notes its
    // largest count and that count's digit
    uint32_t bin = 0;
    if (tid < 256) {
        s_cnt[tid] = 0;
        bin = hist[d.seg * 1024 + tid];
        const uint32_t wmax = __reduce_max_sync(kFullMask, bin);
        const uint32_t at = __ffs(__ballot_sync(kFullMask, bin == wmax)) - 1;
        if (lane == 0) {
            s_misc[16 + warp] = wmax;
            s_misc[24 + warp] = warp * 32 + at;
        }
    }
    if (tid == 0) s_misc[0] = ld_relaxed(a.abort_flag);
    __syncthreads();
    if (s_misc[0]) return;   // an earlier wait gave up; the result is void anyway
    uint32_t hot = 256u, hmax = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t m = s_misc[16 + w];
        if (m > hmax) {
            hmax = m;
            hot = s_misc[24 + w];
        }
    }
    if (hmax <= (d.out_end - d.out_base) / 8) hot = 256u;   // no digit holds over 1/8 of the segment

    bool one_digit = false;
    if (tile_n == static_cast<uint32_t>(TILE)) {   // tile-uniform
        const uint32_t d0 = __shfl_sync(kFullMask, key[0] & 0xFFu, 0);
        bool same = true;
#pragma unroll
        for (int k = 0; k < IPT; ++k) same &= (key[k] & 0xFFu) == d0;
        one_digit = __all_sync(kFullMask, same);
    }
    uint32_t rk[IPT / 2];
    uint32_t hot_base = 0;
    if (hot < 256u && !one_digit) {   // CTA-uniform
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
                const uint32_t dg = key[k + u] & 0xFFu;
                const bool h = valid && dg == hot;
                const uint32_t hm = __ballot_sync(kFullMask, h);
                r[u] = h ? (0x8000u | (run + __popc(hm & ltm))) : (valid ? atomicAdd(&s_cnt[dg], 1u) : 0u);
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
                r0 = take_slot(s_cnt, key[k] & 0xFFu, lane, true);
                r1 = take_slot(s_cnt, key[k + 1] & 0xFFu, lane, true);
            } else {
                if (k * T + tid < tile_n) r0 = atomicAdd(&s_cnt[key[k] & 0xFFu], 1u);
                if ((k + 1) * T + tid < tile_n) r1 = atomicAdd(&s_cnt[key[k + 1] & 0xFFu], 1u);
            }
            rk[k / 2] = r0 | (r1 << 16);
        }
    }
    __syncthreads();

    // scans over the 256 digits: tile offsets and the segment's bin starts
    uint32_t cnt = 0, tile_excl = 0, bin_excl = 0;
    if (tid < 256) {
        cnt = s_cnt[tid];
        const uint32_t ic = warp_inclusive_scan(cnt, lane);
        const uint32_t ib = warp_inclusive_scan(bin, lane);
        if (lane == 31) {
            s_misc[4 + warp] = ic;
            s_misc[16 + warp] = ib;
        }
        tile_excl = ic - cnt;
        bin_excl = ib - bin;
    }
    __syncthreads();
    if (tid < 256) {
        for (uint32_t w = 0; w < warp; ++w) {
            tile_excl += s_misc[4 + w];
            bin_excl += s_misc[16 + w];
        }
        s_cnt[tid] = tile_excl;
    }
    __syncthreads();

    // reserve the tile's places in the segment's bins (in flight during the reorder)
    uint32_t excl = 0;
    if (tid < 256 && cnt != 0) excl = atomicAdd(a.cursor + d.seg * 256 + tid, cnt);
    if (a.look_clear != nullptr && tid < 256) a.look_clear[t * 256 + tid] = 0;
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        if (k * T + tid < tile_n) {
            uint32_t r = (rk[k / 2] >> ((k & 1) * 16)) & 0xFFFFu;
            if (r & 0x8000u) r = hot_base + (r & 0x7FFFu);
            s_keys[s_cnt[key[k] & 0xFFu] + r] = key[k];
        }
    }
    if (tid < 256) s_goff[tid] = d.out_base + bin_excl + excl - tile_excl;
    __syncthreads();

    // contiguous runs per digit out to global memory
    uint32_t *dst_k = static_cast<uint32_t *>(a.dst_k);
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        const uint32_t i = k * T + tid;
        if (i < tile_n) {
            const uint32_t kk = s_keys[i];
            const uint32_t g = s_goff[kk & 0xFFu] + i;
            if (g < d.out_end) dst_k[g] = kk;
        }
    }
}

template <bool PAIRS, int MATCH = kMatchTable>
struct SegPassLaunch {
    template <bool XI, bool XO>
    static cudaError_t one(const PassArgs &a, const SegTile *tiles, const uint32_t *counts,
                           const uint32_t *hist, uint32_t grid, cudaStream_t s) {
        auto k = k_seg_pass<true, PAIRS, XI, XO, MATCH>;
        const size_t smem = (static_cast<size_t>(kSegTile) * (PAIRS ? 2 : 1) + kSegPassWarps * kRow +
                             256 + 32 + peer_table_words<kSegPassWarps, MATCH>()) * sizeof(uint32_t);
        cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(k), smem);
        if (e != cudaSuccess) return e;
        k<<<grid, kSegPassWarps * 32, smem, s>>>(a, tiles, counts, hist);
        return cudaGetLastError();
    }
    static cudaError_t launch(const PassArgs &a, bool xin, bool xout, const SegTile *tiles,
                              const uint32_t *counts, const uint32_t *hist, uint32_t grid,
                              cudaStream_t s) {
        if (xin) return xout ? one<true, true>(a, tiles, counts, hist, grid, s)
                             : one<true, false>(a, tiles, counts, hist, grid, s);
        return xout ? one<false, true>(a, tiles, counts, hist, grid, s)
                    : one<false, false>(a, tiles, counts, hist, grid, s);
    }
};

// ------------------------------------------------------------------- small
// One warp per small segment (grid-stride over the list), padded to the next
// power of two >= 32.
// Keys only: the network sorts the mapped keys (padding 0xFFFFFFFF ties with
// real maximum keys, which is harmless: equal keys are identical).  With
// values: it sorts (mapped key << 32 | position) composites (padding all
// ones sorts after every real composite), and the values are gathered from a
// shared-memory copy of the segment by the position.
template <int LOG_R, bool PAIRS, bool XF>
__device__ __forceinline__ void sort_small(const uint32_t *keys_in, uint32_t *keys_out,
                                           const uint32_t *vals_in, uint32_t *vals_out,
                                           uint32_t a, uint32_t len, uint32_t lane,
                                           uint32_t fmask, uint32_t flip,
                                           typename std::conditional<PAIRS, uint64_t, uint32_t>::type *sw,
                                           uint32_t *sv) {
    using E = typename std::conditional<PAIRS, uint64_t, uint32_t>::type;
    constexpr int R = 1 << LOG_R;
#pragma unroll
    for (int c = 0; c < R; ++c) {
        const uint32_t e = c * 32 + lane;
        E x = ~E(0);
        if (e < len) {
            uint32_t k = keys_in[a + e];
            if (XF) k = order_in<uint32_t>(k, fmask, flip);
            if constexpr (PAIRS) {
                x = (static_cast<uint64_t>(k) << 32) | e;
                sv[e] = vals_in[a + e];
            } else {
                x = k;
            }
        }
        sw[e + (e >> 5)] = x;
    }
    __syncwarp();
    E x[R];
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
        if (e < len) {
            const E y = sw[e + (e >> 5)];
            uint32_t k;
            if constexpr (PAIRS) {
                k = static_cast<uint32_t>(y >> 32);
                vals_out[a + e] = sv[static_cast<uint32_t>(y) & 0x3FFu];
            } else {
                k = y;
            }
            keys_out[a + e] = XF ? order_out<uint32_t>(k, fmask, flip) : k;
        }
    }
    __syncwarp();   // the warp's staging buffers are free for its next segment
}

// One kernel per padded length 2^(5+LOG_R): every kernel walks the whole list
// and takes the segments of its length class, so that each network gets the
// registers it needs (one kernel holding all six would be sized by the largest).
template <int LOG_R, bool PAIRS, bool XF>
__global__ void __launch_bounds__(kSmallWarps * 32)
k_seg_small(const uint32_t *offsets, const uint32_t *small_list, const uint32_t *counts,
            uint32_t small_max, const uint32_t *keys_in, uint32_t *keys_out, const uint32_t *vals_in,
            uint32_t *vals_out, uint32_t fmask, uint32_t flip, const uint32_t *abort_flag) {
    using E = typename std::conditional<PAIRS, uint64_t, uint32_t>::type;
    constexpr uint32_t kLp = 32u << LOG_R;
    constexpr uint32_t kPadded = kLp + kLp / 32;
    extern __shared__ __align__(16) unsigned char s_raw[];
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    E *sw = reinterpret_cast<E *>(s_raw) + warp * kPadded;
    uint32_t *sv = reinterpret_cast<uint32_t *>(reinterpret_cast<E *>(s_raw) + kSmallWarps * kPadded) +
                   warp * kLp;
    if (ld_relaxed(abort_flag)) return;
    const uint32_t count = min(counts[0], small_max);
    const uint32_t warps = gridDim.x * kSmallWarps;
    for (uint32_t i = blockIdx.x * kSmallWarps + warp; i < count; i += warps) {
        const uint32_t s = small_list[i];
        const uint32_t a = offsets[s];
        const uint32_t len = offsets[s + 1] - a;   // 2 .. 1024, checked by the classifier
        const uint32_t log_lp = 32 - __clz(max(len, 32u) - 1);   // padded length 2^log_lp
        if (log_lp != 5 + LOG_R) continue;          // warp-uniform
        sort_small<LOG_R, PAIRS, XF>(keys_in, keys_out, vals_in, vals_out, a, len, lane, fmask, flip,
                                     sw, sv);
    }
}

template <int LOG_R, bool PAIRS, bool XF>
cudaError_t launch_small_class(const uint32_t *offsets, const uint32_t *small_list,
                               const uint32_t *counts, uint32_t small_max, const uint32_t *keys_in,
                               uint32_t *keys_out, const uint32_t *vals_in, uint32_t *vals_out,
                               uint32_t fmask, uint32_t flip, const uint32_t *abort_flag,
                               uint32_t grid, cudaStream_t s) {
    using E = typename std::conditional<PAIRS, uint64_t, uint32_t>::type;
    constexpr uint32_t kLp = 32u << LOG_R;
    constexpr uint32_t kPadded = kLp + kLp / 32;
    const size_t smem = kSmallWarps * (kPadded * sizeof(E) + (PAIRS ? kLp * sizeof(uint32_t) : 0));
    auto k = k_seg_small<LOG_R, PAIRS, XF>;
    cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(k), smem);
    if (e != cudaSuccess) return e;
    k<<<grid, kSmallWarps * 32, smem, s>>>(offsets, small_list, counts, small_max, keys_in, keys_out,
                                           vals_in, vals_out, fmask, flip, abort_flag);
    return cudaGetLastError();
}

constexpr int kSmallClasses = 6;   // padded lengths 32 .. 1024

template <bool PAIRS, bool XF>
cudaError_t launch_small(int cls, const uint32_t *offsets, const uint32_t *small_list, const uint32_t *counts,
                         uint32_t small_max, const uint32_t *keys_in, uint32_t *keys_out,
                         const uint32_t *vals_in, uint32_t *vals_out, uint32_t fmask, uint32_t flip,
                         const uint32_t *abort_flag, uint32_t grid, cudaStream_t s) {
    switch (cls) {
#define GSORT_SMALL_CLASS(R)                                                                            \
        case R:                                                                                         \
            return launch_small_class<R, PAIRS, XF>(offsets, small_list, counts, small_max, keys_in,   \
                                                    keys_out, vals_in, vals_out, fmask, flip,           \
                                                    abort_flag, grid, s);
        GSORT_SMALL_CLASS(0)
        GSORT_SMALL_CLASS(1)
        GSORT_SMALL_CLASS(2)
        GSORT_SMALL_CLASS(3)
        GSORT_SMALL_CLASS(4)
        GSORT_SMALL_CLASS(5)
#undef GSORT_SMALL_CLASS
        default:
            return cudaErrorInvalidValue;
    }
}

// Streams beside the caller's, one per small-segment length class, made once
// per device.  A call forks them from its stream with an event after the
// classification and makes its stream wait for all of them before it
// returns, so every kernel of the call stays ordered on the caller's stream
// while the networks overlap one another and the large segments' kernels.
// One call at a time enqueues on them (the fork and join events are shared).
constexpr int kMaxSideDevices = 64;

struct SideStreams {
    cudaStream_t st[kSmallClasses];
    cudaEvent_t join[kSmallClasses];
    cudaEvent_t fork;
};

std::mutex g_side_mutex;
SideStreams *g_side[kMaxSideDevices] = {};

// The current device's side streams (made on first use), or null if they
// cannot be made: the networks then run one after another on the caller's
// stream.  Called with g_side_mutex held.
SideStreams *side_streams() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxSideDevices) return nullptr;
    if (g_side[dev] != nullptr) return g_side[dev];
    SideStreams *S = new SideStreams();   // value-initialised: null handles
    bool ok = cudaEventCreateWithFlags(&S->fork, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < kSmallClasses; ++i)
        ok = cudaStreamCreateWithFlags(&S->st[i], cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&S->join[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        for (int i = 0; i < kSmallClasses; ++i) {
            if (S->st[i] != nullptr) cudaStreamDestroy(S->st[i]);
            if (S->join[i] != nullptr) cudaEventDestroy(S->join[i]);
        }
        if (S->fork != nullptr) cudaEventDestroy(S->fork);
        delete S;
        cudaGetLastError();   // the failed creation is not this call's error
        return nullptr;
    }
    g_side[dev] = S;
    return S;
}

void record(cudaEvent_t *ev, int num, int idx, cudaStream_t s) {
    if (ev != nullptr && idx < num && ev[idx] != nullptr) cudaEventRecord(ev[idx], s);
}

}  // namespace

SegLayout seg_layout(uint32_t n, uint32_t num_segments, bool with_values) {
    SegLayout L{};
    L.small_max = std::min<uint32_t>(num_segments, n / 2);
    L.large_max = std::min<uint32_t>(num_segments, n / (kSmallMax + 1));
    L.tiles_max = (n + kSegTile - 1) / kSegTile + L.large_max;
    size_t off = kHdrBytes;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += align_up(std::max<size_t>(bytes, 1), kWsAlign);
        return at;
    };
    L.small_list = take(static_cast<size_t>(L.small_max) * 4);
    L.large_start = take(static_cast<size_t>(L.large_max) * 4);
    L.large_len = take(static_cast<size_t>(L.large_max) * 4);
    L.tile_base = take((static_cast<size_t>(L.large_max) + 1) * 4);
    L.tiles = take(static_cast<size_t>(L.tiles_max) * sizeof(SegTile));
    L.hist = take(static_cast<size_t>(L.large_max) * 1024 * 4);
    L.look_a = take(static_cast<size_t>(L.tiles_max) * 256 * 4);
    L.look_b = take(static_cast<size_t>(L.tiles_max) * 256 * 4);
    L.tmp_keys = take(static_cast<size_t>(n) * 4);
    L.tmp_vals = with_values ? take(static_cast<size_t>(n) * 4) : off;
    L.total = off;
    return L;
}

namespace {

// The large segments' kernels, on the caller's stream: tile counts, tile
// descriptors, histograms, four digit passes.
int launch_large_segments(const SegLaunch &L, const SegLayout &lay, bool pairs, bool mapped,
                          const KeyOrder &order, cudaStream_t s) {
    const uint32_t fmask = static_cast<uint32_t>(order.fmask), flip = static_cast<uint32_t>(order.flip);
    unsigned char *ws = L.ws;
    uint32_t *status = reinterpret_cast<uint32_t *>(ws + kHdrStatus);
    uint32_t *abort_flag = reinterpret_cast<uint32_t *>(ws + kHdrAbort);
    uint32_t *counts = reinterpret_cast<uint32_t *>(ws + kHdrSegCounts);
    uint32_t *large_start = reinterpret_cast<uint32_t *>(ws + lay.large_start);
    uint32_t *large_len = reinterpret_cast<uint32_t *>(ws + lay.large_len);
    uint32_t *tile_base = reinterpret_cast<uint32_t *>(ws + lay.tile_base);
    SegTile *tiles = reinterpret_cast<SegTile *>(ws + lay.tiles);
    uint32_t *hist = reinterpret_cast<uint32_t *>(ws + lay.hist);
    uint32_t *look[2] = {reinterpret_cast<uint32_t *>(ws + lay.look_a),
                         reinterpret_cast<uint32_t *>(ws + lay.look_b)};
    uint32_t *tmp_k = reinterpret_cast<uint32_t *>(ws + lay.tmp_keys);
    uint32_t *tmp_v = pairs ? reinterpret_cast<uint32_t *>(ws + lay.tmp_vals) : nullptr;
    const uint32_t sms = static_cast<uint32_t>(L.sm_count);
    cudaError_t e;
    if (lay.large_max == 0) {
        for (int i = 3; i < 8; ++i) record(L.events, L.num_events, i, s);
        return GSORT_OK;
    }

    k_seg_scan<<<1, kScanThreads, 0, s>>>(large_len, lay.large_max, lay.tiles_max, tile_base, counts,
                                          status, abort_flag);
    if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
    const uint32_t mgrid = std::max(1u, std::min((lay.large_max + 7) / 8, sms * 8));
    k_seg_tilemap<<<mgrid, 256, 0, s>>>(large_start, large_len, tile_base, counts, lay.large_max, tiles,
                                        reinterpret_cast<uint4 *>(hist), abort_flag);
    if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
    const uint32_t hgrid = std::max(1u, std::min(lay.tiles_max, sms));
    {
        auto hk = mapped ? k_seg_hist<true> : k_seg_hist<false>;
        if (set_smem_limit(reinterpret_cast<const void *>(hk), kSegHistSmem) != cudaSuccess) return GSORT_ECUDA;
        hk<<<hgrid, kSegHistThreads, kSegHistSmem, s>>>(L.keys_in, tiles, counts, fmask, flip, hist, look[0],
                                                        abort_flag);
    }
    if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
    record(L.events, L.num_events, 3, s);

    // in -> tmp -> out -> tmp -> out (also when in == out: each pass reads
    // what the previous one wrote)
    // keys-only passes fit three CTAs per SM (40 registers), pairs two
    const uint32_t pgrid = std::max(1u, std::min(lay.tiles_max, sms * (pairs ? 2u : 3u)));
    const uint32_t *src_k = L.keys_in;
    const uint32_t *src_v = L.vals_in;
    for (int p = 0; p < 4; ++p) {
        uint32_t *dst_k = (p % 2 == 0) ? tmp_k : L.keys_out;
        uint32_t *dst_v = pairs ? ((p % 2 == 0) ? tmp_v : L.vals_out) : nullptr;
        PassArgs a;
        a.src_k = src_k;
        a.dst_k = dst_k;
        a.src_v = src_v;
        a.dst_v = dst_v;
        a.n = L.n;
        a.shift = static_cast<uint32_t>(8 * p);
        a.mask = 0xFFu;
        a.fmask = order.fmask;
        a.flip = order.flip;
        a.hist = nullptr;   // per segment, from the tile descriptor
        a.look = look[p & 1];
        a.look_clear = (p + 1 < 4) ? look[(p + 1) & 1] : nullptr;
        a.tile_counter = reinterpret_cast<uint32_t *>(ws + kHdrCounters + 128 * p);
        a.status = status;
        a.abort_flag = abort_flag;
        a.spin_limit = L.spin_limit;
        a.stall_tile = kNoStall;
        a.prefetch_dist = 0;   // tiles map to segments; no prefetch
        // keys only: equal keys are indistinguishable (tiles never cross a segment)
        a.order_free = pairs ? 0u : 1u;
        a.free_low = (1ull << a.shift) - 1ull;
        a.two_runs_ok = p <= 1 ? 1u : 0u;   // later passes see short runs in any segment
        // keys only, first pass: any order inside a digit is right, so a tile
        // reserves its places in its segment's bins on 256 cursors of its own
        // segment (no look-back); the cursors are the first pass's look-back
        // rows, which the histogram kernel cleared and this pass does not use
        a.cursor = (!pairs && p == 0) ? look[0] : nullptr;
        const bool xin = mapped && p == 0, xout = mapped && p == 3;
        if (a.cursor != nullptr) {   // keys only, first pass
            auto k = xin ? k_seg_pass_free<true> : k_seg_pass_free<false>;
            const size_t smem = (static_cast<size_t>(kSegTile) + 256 + 256 + 32) * sizeof(uint32_t);
            if (set_smem_limit(reinterpret_cast<const void *>(k), smem) != cudaSuccess) return GSORT_ECUDA;
            k<<<std::max(1u, lay.tiles_max), kSegPassWarps * 32, smem, s>>>(a, tiles, counts, hist);
            if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
            record(L.events, L.num_events, 4 + p, s);
            src_k = dst_k;
            src_v = dst_v;
            continue;
        }
        // keys only: peer masks from shared reductions (inside segments runs of
        // equal low bits are short from the second pass on)
        e = pairs ? SegPassLaunch<true>::launch(a, xin, xout, tiles, counts, hist, pgrid, s)
                  : SegPassLaunch<false, kMatchRedOr>::launch(a, xin, xout, tiles, counts, hist, pgrid, s);
        if (e != cudaSuccess) return GSORT_ECUDA;
        record(L.events, L.num_events, 4 + p, s);
        src_k = dst_k;
        src_v = dst_v;
    }
    return GSORT_OK;
}

}  // namespace

int launch_segmented_sort(const SegLaunch &L) {
    const bool pairs = L.vals_in != nullptr;
    const SegLayout lay = seg_layout(L.n, L.num_segments, pairs);
    const KeyOrder order = key_order(L.kind, L.flags);
    const bool mapped = order.fmask != 0 || order.flip != 0;
    const uint32_t fmask = static_cast<uint32_t>(order.fmask), flip = static_cast<uint32_t>(order.flip);
    cudaStream_t s = L.stream;
    unsigned char *ws = L.ws;
    uint32_t *status = reinterpret_cast<uint32_t *>(ws + kHdrStatus);
    uint32_t *abort_flag = reinterpret_cast<uint32_t *>(ws + kHdrAbort);
    uint32_t *counts = reinterpret_cast<uint32_t *>(ws + kHdrSegCounts);
    uint32_t *small_list = reinterpret_cast<uint32_t *>(ws + lay.small_list);
    uint32_t *large_start = reinterpret_cast<uint32_t *>(ws + lay.large_start);
    uint32_t *large_len = reinterpret_cast<uint32_t *>(ws + lay.large_len);
    const uint32_t sms = static_cast<uint32_t>(L.sm_count);

    record(L.events, L.num_events, 0, s);
    k_zero_words<<<1, 256, 0, s>>>(reinterpret_cast<uint32_t *>(ws), static_cast<uint32_t>(kHdrBytes / 4));
    if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
    const uint32_t cgrid = std::max(1u, std::min((L.num_segments + 255) / 256, sms * 8));
    k_seg_classify<<<cgrid, 256, 0, s>>>(L.offsets, L.num_segments, L.n, small_list, lay.small_max,
                                         large_start, large_len, lay.large_max, L.keys_in, L.keys_out,
                                         L.vals_in, L.vals_out, counts, status, abort_flag);
    if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
    record(L.events, L.num_events, 1, s);

    // small segments: one network kernel per length class, independent of
    // the large-segment kernels (disjoint key ranges), each on a side stream
    std::lock_guard<std::mutex> lock(g_side_mutex);
    SideStreams *side = side_streams();
    if (side != nullptr && cudaEventRecord(side->fork, s) != cudaSuccess) return GSORT_ECUDA;
    const uint32_t sgrid = std::max(1u, std::min((lay.small_max + kSmallWarps - 1) / kSmallWarps, sms * 16));
    int rc = GSORT_OK, forked = 0;   // side streams whose work the caller's stream must wait for
    for (int c = 0; c < kSmallClasses && rc == GSORT_OK; ++c) {
        cudaStream_t ss = side != nullptr ? side->st[c] : s;
        if (side != nullptr && cudaStreamWaitEvent(ss, side->fork, 0) != cudaSuccess) {
            rc = GSORT_ECUDA;
            break;
        }
        cudaError_t e;
        if (pairs)
            e = mapped ? launch_small<true, true>(c, L.offsets, small_list, counts, lay.small_max, L.keys_in,
                                                  L.keys_out, L.vals_in, L.vals_out, fmask, flip, abort_flag,
                                                  sgrid, ss)
                       : launch_small<true, false>(c, L.offsets, small_list, counts, lay.small_max, L.keys_in,
                                                   L.keys_out, L.vals_in, L.vals_out, fmask, flip, abort_flag,
                                                   sgrid, ss);
        else
            e = mapped ? launch_small<false, true>(c, L.offsets, small_list, counts, lay.small_max, L.keys_in,
                                                   L.keys_out, nullptr, nullptr, fmask, flip, abort_flag, sgrid, ss)
                       : launch_small<false, false>(c, L.offsets, small_list, counts, lay.small_max, L.keys_in,
                                                    L.keys_out, nullptr, nullptr, fmask, flip, abort_flag, sgrid,
                                                    ss);
        if (side != nullptr) {
            // joined even after a failed launch: whatever reached the side stream is waited for
            if (cudaEventRecord(side->join[c], ss) == cudaSuccess) ++forked;
            else rc = GSORT_ECUDA;
        }
        if (e != cudaSuccess) rc = GSORT_ECUDA;
    }
    if (rc == GSORT_OK) rc = launch_large_segments(L, lay, pairs, mapped, order, s);
    for (int c = 0; c < forked; ++c)
        if (cudaStreamWaitEvent(s, side->join[c], 0) != cudaSuccess) rc = GSORT_ECUDA;
    record(L.events, L.num_events, 2, s);
    return rc;
}

}  // namespace gsort

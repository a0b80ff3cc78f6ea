// radix.cu -- stable LSD radix sort with 8-bit digits for sm_103a.
//
// Steps (page tags as in include/gsort.h):
//   init       clear the workspace header (status, tile counters, histograms)
//   histogram  one read of the keys builds the 256-bin histogram of every
//              digit pass ([CUDA3] "processing several bits at once", kernel 1;
//              [PMPP10] 10.3 histogram step) and clears the first pass's
//              look-back region
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
// multisplit (peer mask of equal digits + popcount below the lane, one
// shared counter per warp and digit) instead of eight block-wide 1-bit splits;
// look-back regions are cleared one row per tile by the previous kernel
// instead of a memset per pass; every wait is bounded.
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
constexpr int kHistThreads = 256;
constexpr int kHistParts = 4;     // sub-histograms by lane, spreading same-digit atomics
constexpr int kHistUnroll = 4;    // 16-byte loads in flight per thread

template <bool XF>
__device__ __forceinline__ void hist_count(uint32_t *s_h, uint32_t k, uint32_t begin_bit,
                                           int passes, uint32_t last_mask, uint32_t part) {
    if (XF) k = float_key_in(k);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        if (p < passes) {
            const uint32_t d = (k >> (begin_bit + 8 * p)) & (p == passes - 1 ? last_mask : 0xFFu);
            atomicAdd(&s_h[(p * 256 + d) * kHistParts + part], 1u);
        }
    }
}

template <bool XF>
__global__ void __launch_bounds__(kHistThreads)
k_digit_hist(const uint32_t *__restrict__ keys, uint32_t n, uint32_t begin_bit, int passes,
             uint32_t last_mask, uint32_t *__restrict__ hist, uint4 *__restrict__ clear,
             uint32_t clear_vec4) {
    __shared__ uint32_t s_h[4 * 256 * kHistParts];
    const uint32_t tid = threadIdx.x;
    for (uint32_t i = tid; i < 4 * 256 * kHistParts; i += kHistThreads) s_h[i] = 0;
    const uint32_t gtid = blockIdx.x * kHistThreads + tid;
    const uint32_t gstride = gridDim.x * kHistThreads;
    for (uint32_t i = gtid; i < clear_vec4; i += gstride) clear[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();

    const uint32_t part = tid & (kHistParts - 1);
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
                hist_count<XF>(s_h, q[u].x, begin_bit, passes, last_mask, part);
                hist_count<XF>(s_h, q[u].y, begin_bit, passes, last_mask, part);
                hist_count<XF>(s_h, q[u].z, begin_bit, passes, last_mask, part);
                hist_count<XF>(s_h, q[u].w, begin_bit, passes, last_mask, part);
            }
        }
    }
    const uint32_t tail0 = head + nvec * 4;
    if (gtid < head) hist_count<XF>(s_h, keys[gtid], begin_bit, passes, last_mask, part);
    if (gtid < n - tail0) hist_count<XF>(s_h, keys[tail0 + gtid], begin_bit, passes, last_mask, part);
    __syncthreads();

    for (uint32_t i = tid; i < static_cast<uint32_t>(passes) * 256; i += kHistThreads) {
        uint32_t s = 0;
#pragma unroll
        for (int q = 0; q < kHistParts; ++q) s += s_h[i * kHistParts + q];
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
    uint32_t *look;         // [tiles][256] look-back words of this pass (cleared)
    uint32_t *look_clear;   // next pass's region: row `tile` is cleared here; may be null
    uint32_t *tile_counter;
    uint32_t *status;
    uint32_t *abort_flag;
    uint32_t spin_limit;
    uint32_t stall_tile;
};

// Mask of the lanes whose digit equals this lane's digit.  BITS = digit
// width considered (8, or 9 when padding items carry the pseudo-digit 256).
template <int BITS, bool HW>
__device__ __forceinline__ uint32_t match_digit(uint32_t d) {
    if constexpr (HW) {
        return __match_any_sync(kFullMask, d);
    } else {
        uint32_t peers = kFullMask;
#pragma unroll
        for (int b = 0; b < BITS; ++b) {
            const bool bit = (d >> b) & 1u;
            const uint32_t m = __ballot_sync(kFullMask, bit);
            peers &= bit ? m : ~m;
        }
        return peers;
    }
}

constexpr int kRow = 257;   // per-warp digit counters, slot 256 = padding items

template <int WARPS, int IPT, bool PAIRS>
constexpr size_t pass_smem_words() {
    return static_cast<size_t>(WARPS * 32 * IPT) * (PAIRS ? 2 : 1) + WARPS * kRow + 256 + 32;
}

template <int WARPS, int IPT, bool HWM, bool PAIRS, bool XIN, bool XOUT, bool FULL>
__device__ __forceinline__ void pass_tile(const PassArgs &a, uint32_t *smem, uint32_t tile) {
    constexpr int T = WARPS * 32;
    constexpr int TILE = T * IPT;
    uint32_t *s_keys = smem;
    uint32_t *s_vals = smem + TILE;
    uint32_t *s_cnt = smem + TILE * (PAIRS ? 2 : 1);
    uint32_t *s_goff = s_cnt + WARPS * kRow;
    uint32_t *s_misc = s_goff + 256;

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
        key[k] = (FULL || i < tile_n) ? a.src_k[tile_base + i] : 0u;
        if (XIN) key[k] = float_key_in(key[k]);
    }

    // ---- warp multisplit: stable rank among this warp's keys of each digit
    uint32_t pos[IPT];
    {
        uint32_t *wc = s_cnt + warp * kRow;
        const uint32_t ltm = lanemask_lt();
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            uint32_t d = (key[k] >> a.shift) & a.mask;
            uint32_t peers;
            if (FULL) {
                peers = match_digit<8, HWM>(d);
            } else {
                if (item0 + k * 32 >= tile_n) d = 256;
                peers = match_digit<9, HWM>(d);
            }
            const int leader = 31 - __clz(peers);
            uint32_t base = 0;
            if (lane == static_cast<uint32_t>(leader)) base = atomicAdd(&wc[d], static_cast<uint32_t>(__popc(peers)));
            base = __shfl_sync(kFullMask, base, leader);
            pos[k] = base + __popc(peers & ltm);
        }
    }

    uint32_t val[PAIRS ? IPT : 1];
    if (PAIRS) {
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            const uint32_t i = item0 + k * 32;
            val[k] = (FULL || i < tile_n) ? a.src_v[tile_base + i] : 0u;
        }
    }
    __syncthreads();

    // ---- tile counts per digit; publish them; scans over the 256 digits
    uint32_t cnt = 0, bin = 0, tile_excl = 0, bin_excl = 0;
    if (tid < 256) {
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            const uint32_t c = s_cnt[w * kRow + tid];
            s_cnt[w * kRow + tid] = cnt;   // exclusive over warps
            cnt += c;
        }
        if (tile != a.stall_tile)
            st_relaxed(a.look + tile * 256 + tid, (tile == 0 ? kFlagPrefix : kFlagAgg) | cnt);
        bin = a.hist[tid];
        const uint32_t ic = warp_inclusive_scan(cnt, lane);
        const uint32_t ib = warp_inclusive_scan(bin, lane);
        if (lane == 31) {
            s_misc[4 + warp] = ic;
            s_misc[12 + warp] = ib;
        }
        tile_excl = ic - cnt;
        bin_excl = ib - bin;
    }
    __syncthreads();

    // ---- decoupled look-back, one digit per thread
    if (tid < 256) {
        for (uint32_t w = 0; w < warp; ++w) {
            tile_excl += s_misc[4 + w];
            bin_excl += s_misc[12 + w];
        }
        uint32_t excl = 0;
        bool ok = true;
        if (tile > 0 && tile != a.stall_tile) {
            int32_t t = static_cast<int32_t>(tile) - 1;
            uint32_t polls = 0, ns = 32;
            while (true) {
                if (t < 0) { ok = false; break; }   // tile 0 always publishes a prefix
                const uint32_t s = ld_relaxed(a.look + static_cast<uint32_t>(t) * 256 + tid);
                if ((s & ~kValueMask) == 0) {
                    if (++polls >= a.spin_limit || ld_relaxed(a.abort_flag)) { ok = false; break; }
                    backoff(ns);
                    continue;
                }
                excl += s & kValueMask;
                if (s & kFlagPrefix) break;
                --t;
            }
            if (ok) st_relaxed(a.look + tile * 256 + tid, kFlagPrefix | (excl + cnt));
        }
        if (!ok) {
            s_misc[2] = 1;
            record_error(a.status, a.abort_flag, GSORT_ETIMEOUT);
        }
        // global index = bin start + earlier tiles + (tile-local slot - tile start of digit)
        s_goff[tid] = bin_excl + excl - tile_excl;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) s_cnt[w * kRow + tid] += tile_excl;
    }
    __syncthreads();
    if (s_misc[2] || tile == a.stall_tile) return;

    // ---- reorder the tile by digit in shared memory
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        if (FULL || item0 + k * 32 < tile_n) {
            const uint32_t d = (key[k] >> a.shift) & a.mask;
            const uint32_t p = pos[k] + s_cnt[warp * kRow + d];
            s_keys[p] = key[k];
            if (PAIRS) s_vals[p] = val[k];
        }
    }
    __syncthreads();

    // ---- contiguous runs per digit out to global memory
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
        const uint32_t i = k * T + tid;
        if (FULL || i < tile_n) {
            const uint32_t kk = s_keys[i];
            const uint32_t g = s_goff[(kk >> a.shift) & a.mask] + i;
            if (g < a.n) {
                a.dst_k[g] = XOUT ? float_key_out(kk) : kk;
                if (PAIRS) a.dst_v[g] = s_vals[i];
            }
        }
    }
}

template <int WARPS, int IPT, int MINB, bool HWM, bool PAIRS, bool XIN, bool XOUT>
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
    if (a.look_clear != nullptr)
        for (uint32_t i = tid; i < 256; i += WARPS * 32) a.look_clear[tile * 256 + i] = 0;
    if (a.n - tile * TILE >= static_cast<uint32_t>(TILE))
        pass_tile<WARPS, IPT, HWM, PAIRS, XIN, XOUT, true>(a, smem, tile);
    else
        pass_tile<WARPS, IPT, HWM, PAIRS, XIN, XOUT, false>(a, smem, tile);
}

// ------------------------------------------------------------ variants
template <int WARPS, int IPT, int MINB, bool HWM>
struct PassConfig {
    static constexpr uint32_t kTile = WARPS * 32 * IPT;

    template <bool P, bool XI, bool XO>
    static cudaError_t launch_one(const PassArgs &a, uint32_t tiles, cudaStream_t s) {
        auto k = k_digit_pass<WARPS, IPT, MINB, HWM, P, XI, XO>;
        const size_t smem = pass_smem_words<WARPS, IPT, P>() * sizeof(uint32_t);
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        k<<<tiles, WARPS * 32, smem, s>>>(a);
        return cudaGetLastError();
    }

    static cudaError_t launch(const PassArgs &a, bool pairs, bool xin, bool xout, uint32_t tiles,
                              cudaStream_t s) {
        const int sel = (pairs ? 4 : 0) | (xin ? 2 : 0) | (xout ? 1 : 0);
        switch (sel) {
            case 0: return launch_one<false, false, false>(a, tiles, s);
            case 1: return launch_one<false, false, true>(a, tiles, s);
            case 2: return launch_one<false, true, false>(a, tiles, s);
            case 3: return launch_one<false, true, true>(a, tiles, s);
            case 4: return launch_one<true, false, false>(a, tiles, s);
            case 5: return launch_one<true, false, true>(a, tiles, s);
            case 6: return launch_one<true, true, false>(a, tiles, s);
            default: return launch_one<true, true, true>(a, tiles, s);
        }
    }
};

struct Variant {
    const char *name;
    uint32_t tile;
    cudaError_t (*launch)(const PassArgs &, bool, bool, bool, uint32_t, cudaStream_t);
};

const Variant kVariants[] = {
    {"16 warps x 16 items, ballot multisplit", PassConfig<16, 16, 2, false>::kTile,
     &PassConfig<16, 16, 2, false>::launch},
    {"16 warps x 16 items, match.any multisplit", PassConfig<16, 16, 2, true>::kTile,
     &PassConfig<16, 16, 2, true>::launch},
    {"8 warps x 16 items, ballot multisplit", PassConfig<8, 16, 3, false>::kTile,
     &PassConfig<8, 16, 3, false>::launch},
    {"8 warps x 16 items, match.any multisplit", PassConfig<8, 16, 3, true>::kTile,
     &PassConfig<8, 16, 3, true>::launch},
};
constexpr int kNumVariants = sizeof(kVariants) / sizeof(kVariants[0]);

uint32_t hist_grid(uint32_t n, int sm_count) {
    const uint32_t vec = (n >> 2) + 1;
    const uint32_t want = (vec + kHistThreads * kHistUnroll - 1) / (kHistThreads * kHistUnroll);
    return std::max(1u, std::min(want, static_cast<uint32_t>(sm_count) * 8u));
}

cudaError_t launch_hist(const uint32_t *keys, uint32_t n, int kind, int begin_bit, int passes,
                        uint32_t last_mask, uint32_t *hist, uint32_t *clear, uint32_t clear_words,
                        cudaStream_t s, int sm_count) {
    const uint32_t grid = std::max(hist_grid(n, sm_count),
                                   std::min<uint32_t>(clear_words / 4 / kHistThreads + 1,
                                                      static_cast<uint32_t>(sm_count) * 8u));
    uint4 *cl = reinterpret_cast<uint4 *>(clear);
    if (kind == GSORT_KEY_F32)
        k_digit_hist<true><<<grid, kHistThreads, 0, s>>>(keys, n, begin_bit, passes, last_mask,
                                                         hist, cl, clear_words / 4);
    else
        k_digit_hist<false><<<grid, kHistThreads, 0, s>>>(keys, n, begin_bit, passes, last_mask,
                                                          hist, cl, clear_words / 4);
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
    L.look_a = off;
    off += region;
    L.look_b = off;
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
    const uint32_t last_mask = (last_width >= 32) ? 0xFFFFFFFFu : ((1u << last_width) - 1u);
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

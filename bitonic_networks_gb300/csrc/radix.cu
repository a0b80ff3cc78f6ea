// radix.cu -- stable LSD radix sort with 8-bit digits for sm_103a: the
// 32-bit key configurations of the digit pass, the workspace layout and the
// host sequence (init, histogram, P digit passes) for every key kind.  The
// device code and the algorithm notes are in radix_kernels.cuh; 64-bit keys
// are instantiated in radix64.cu.
#include "radix_kernels.cuh"

namespace gsort {
namespace {

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
            bulk_load(kbuf + b * TILE, static_cast<const uint32_t *>(a->src_k) + t * TILE, bytes, &bar[b]);
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
        if (tid == 0) {
            s_misc[2] = 0;
            s_misc[3] = a.hot != nullptr ? *a.hot : 256u;
        }
        for (uint32_t i = tid; i < WARPS * kRow; i += T) tab[i] = 0;
        const bool arrived = mbar_wait_bounded(&bar[b], phase[b], kBulkWaitLimit);
        const uint32_t tile_n = min(static_cast<uint32_t>(TILE), a.n - tile * TILE);
        uint32_t *kb = kbuf + b * TILE;
        uint32_t *vb = vbuf + b * TILE;
        const uint32_t rest = tile_n & 3u;   // the last keys of a ragged tile come by plain loads
        if (arrived && tid < rest) {
            kb[tile_n - rest + tid] = static_cast<const uint32_t *>(a.src_k)[tile * TILE + tile_n - rest + tid];
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
        const TileDesc td{tile, 0u, tile_n, a.hist, 0u, a.n};
        bool ok;
        if (tile_n == static_cast<uint32_t>(TILE))
            ok = pass_tile<uint32_t, WARPS, IPT, MATCH, LW, BYTE, PAIRS, XIN, XOUT, true>(a, tab, td, kb, vb, kb, vb, claim);
        else
            ok = pass_tile<uint32_t, WARPS, IPT, MATCH, LW, BYTE, PAIRS, XIN, XOUT, false>(a, tab, td, kb, vb, kb, vb, claim);
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
        cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(k), smem);
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = blocks_per_sm(reinterpret_cast<const void *>(k), WARPS * 32, smem, &per_sm);
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
            return PassConfig<uint32_t, WARPS, IPT, 2, MATCH, LW>::launch(a, pairs, xin, xout, tiles, s);
        const bool byte = (a.shift % 8) == 0 && a.mask == 0xFFu;
        return byte ? launch_b<true>(a, pairs, xin, xout, tiles, s)
                    : launch_b<false>(a, pairs, xin, xout, tiles, s);
    }
};


// Keys and pairs in one variant with different occupancy: keys-only passes
// fit 40 registers without spilling, so three CTAs share an SM; pairs hold
// twice the registers per item and keep two.  Keys-only passes whose runs of
// equal low bits are expected to be short (under 256 keys for uniform input,
// so most warps take the stable path: the last pass of a large sort) build
// their peer masks with shared reductions (ShortRunsCfg), which costs less
// integer work than the ballots on spread digits; elsewhere the ballot
// tables, which do not serialise on repeated digits.
template <class KeysCfg, class ShortRunsCfg, class PairsCfg>
struct KeysPairsConfig {
    static_assert(KeysCfg::kTile == PairsCfg::kTile && ShortRunsCfg::kTile == KeysCfg::kTile,
                  "one tile size per variant");
    static constexpr uint32_t kTile = KeysCfg::kTile;
    static cudaError_t launch(const PassArgs &a, bool pairs, bool xin, bool xout, uint32_t tiles,
                              cudaStream_t s) {
        if (pairs) return PairsCfg::launch(a, pairs, xin, xout, tiles, s);
        return a.two_runs_ok ? KeysCfg::launch_keys(a, pairs, xin, xout, tiles, s)
                             : ShortRunsCfg::launch_keys(a, pairs, xin, xout, tiles, s);
    }
};
using Variant0 = KeysPairsConfig<PassConfig<uint32_t, 16, 16, 3, kMatchTable>,
                                 PassConfig<uint32_t, 16, 16, 3, kMatchRedOr>,
                                 PassConfig<uint32_t, 16, 16, 2, kMatchTable>>;

// `free_launch`: the first pass of a keys-only sort over every bit, where
// every warp is order-free (same tile; null: the variant's own kernel, in its
// bin-cursor mode).
struct Variant {
    const char *name;
    uint32_t tile;
    PassLauncher launch;
    PassLauncher free_launch;
};

const Variant kVariants[] = {
    {"one tile per CTA, 16 warps x 16 items", Variant0::kTile, &Variant0::launch,
     &FreePassConfig<uint32_t, 16, 16, 3>::launch},
    {"persistent, 16 warps x 16 items, TMA prefetch", PersistentConfig<16, 16, kMatchTable>::kTile,
     &PersistentConfig<16, 16, kMatchTable>::launch, nullptr},
    {"one tile per CTA, 8 warps x 16 items", PassConfig<uint32_t, 8, 16, 3, kMatchTable>::kTile,
     &PassConfig<uint32_t, 8, 16, 3, kMatchTable>::launch, &FreePassConfig<uint32_t, 8, 16, 4>::launch},
};
static_assert(FreePassConfig<uint32_t, 16, 16, 3>::kTile == Variant0::kTile &&
                  FreePassConfig<uint32_t, 8, 16, 4>::kTile == PassConfig<uint32_t, 8, 16, 3, kMatchTable>::kTile,
              "an order-free first pass keeps its variant's tile");
constexpr int kNumVariants = sizeof(kVariants) / sizeof(kVariants[0]);

void record(cudaEvent_t *ev, int num, int idx, cudaStream_t s) {
    if (ev != nullptr && idx < num && ev[idx] != nullptr) cudaEventRecord(ev[idx], s);
}

}  // namespace

int radix_num_variants() { return kNumVariants; }

const char *radix_variant_name(int v) {
    return (v >= 0 && v < kNumVariants) ? kVariants[v].name : nullptr;
}

uint32_t radix_variant_tile(int v) { return kVariants[v].tile; }

KeyOrder key_order(int kind, int flags) {
    KeyOrder o{};
    o.key_bytes = key_kind_bytes(kind);
    const uint64_t all = o.key_bytes == 8 ? ~0ull : 0xFFFFFFFFull;
    const uint64_t sign = o.key_bytes == 8 ? (1ull << 63) : (1ull << 31);
    o.fmask = (kind == GSORT_KEY_F32 || kind == GSORT_KEY_F64) ? all : 0;
    o.flip = (kind == GSORT_KEY_I32 || kind == GSORT_KEY_I64) ? sign : 0;
    if (flags & GSORT_DESCENDING) o.flip ^= all;
    return o;
}

RadixLayout radix_layout(uint32_t n, bool with_values, int key_bytes) {
    RadixLayout L{};
    L.tiles_max = (n + kMinRadixTile - 1) / kMinRadixTile;
    size_t off = kHdrBytes;
    L.starts = off;   // bin starts of up to 8 passes
    off += align_up(8 * 256 * sizeof(uint32_t), kWsAlign);
    // 32-bit keys keep their 4 x 256 histogram counts in the header; 64-bit
    // keys have 8 passes and take a region of their own
    L.hist = key_bytes == 8 ? off : kHdrHist;
    if (key_bytes == 8) off += align_up(8 * 256 * sizeof(uint32_t), kWsAlign);
    const size_t region = align_up(static_cast<size_t>(L.tiles_max) * 256 * sizeof(uint32_t), kWsAlign);
    L.look_a = off;   // [tiles_max][256] look-back words, even passes
    off += region;
    L.look_b = off;   // odd passes
    off += region;
    L.tmp_keys = off;
    off += align_up(static_cast<size_t>(n) * key_bytes, kWsAlign);
    L.tmp_vals = off;
    if (with_values) off += align_up(static_cast<size_t>(n) * sizeof(uint32_t), kWsAlign);
    // the one-launch sort of small inputs: three rotating [tiles][256] count buffers
    L.small_counts = off;
    if (small_sort_applies(n, key_bytes, 0))
        off += align_up(3 * static_cast<size_t>((n + small_sort_tile() - 1) / small_sort_tile()) * 256 *
                            sizeof(uint32_t), kWsAlign);
    L.total = off;
    return L;
}

namespace {

cudaError_t launch_hist_any(const void *keys, uint32_t n, const KeyOrder &o, int begin_bit,
                            int passes, uint32_t last_mask, uint32_t *hist, uint32_t *clear,
                            uint32_t clear_words, cudaStream_t s, int sm_count,
                            const BinStartsOut &bs = BinStartsOut()) {
    const bool xf = o.fmask != 0 || o.flip != 0;
    if (o.key_bytes == 8)
        return launch_hist_u64(static_cast<const uint64_t *>(keys), n, xf, o.fmask, o.flip, begin_bit,
                               passes, last_mask, hist, clear, clear_words, s, sm_count, bs);
    return launch_hist_kernel<uint32_t>(static_cast<const uint32_t *>(keys), n, xf,
                                        static_cast<uint32_t>(o.fmask), static_cast<uint32_t>(o.flip),
                                        begin_bit, passes, last_mask, hist, clear, clear_words, s,
                                        sm_count, bs);
}

}  // namespace

int launch_radix(const RadixLaunch &L) {
    const KeyOrder order = key_order(L.kind, L.flags);
    const size_t kb = static_cast<size_t>(order.key_bytes);
    const int passes = (L.end_bit - L.begin_bit + 7) / 8;
    const bool pairs = L.vals_in != nullptr;
    const bool mapped = order.fmask != 0 || order.flip != 0;
    const RadixLayout lay = radix_layout(L.n, pairs, order.key_bytes);
    // 64-bit keys have one configuration; 32-bit keys take the chosen variant
    const uint32_t tile = kb == 8 ? pass_tile_u64() : kVariants[L.variant].tile;
    const PassLauncher launch = kb == 8 ? &launch_pass_u64 : kVariants[L.variant].launch;
    const PassLauncher free_launch = kb == 8 ? &launch_pass_u64_free : kVariants[L.variant].free_launch;
    const uint32_t tiles = (L.n + tile - 1) / tile;
    cudaStream_t s = L.stream;

    uint32_t *hdr = reinterpret_cast<uint32_t *>(L.ws);
    uint32_t *status = reinterpret_cast<uint32_t *>(L.ws + kHdrStatus);
    uint32_t *abort_flag = reinterpret_cast<uint32_t *>(L.ws + kHdrAbort);
    uint32_t *hist = reinterpret_cast<uint32_t *>(L.ws + lay.hist);
    uint32_t *starts = reinterpret_cast<uint32_t *>(L.ws + lay.starts);
    uint32_t *cursor = reinterpret_cast<uint32_t *>(L.ws + kHdrCursor);
    uint32_t *look[2] = {reinterpret_cast<uint32_t *>(L.ws + lay.look_a),
                         reinterpret_cast<uint32_t *>(L.ws + lay.look_b)};
    void *tmp_k = L.ws + lay.tmp_keys;
    uint32_t *tmp_v = pairs ? reinterpret_cast<uint32_t *>(L.ws + lay.tmp_vals) : nullptr;

    const uint32_t last_width = static_cast<uint32_t>(L.end_bit - L.begin_bit - 8 * (passes - 1));
    const uint32_t last_mask = (1u << last_width) - 1u;
    const bool alias = (L.keys_in == L.keys_out) || (pairs && L.vals_in == L.vals_out);

    record(L.events, L.num_events, 0, s);
    if (cluster_sort_applies(L.n, order.key_bytes, L.variant, L.stall_tile, passes)) {
        // one launch, no header clear (the kernel clears the status words)
        SmallSortLaunch S{};
        S.keys_in = static_cast<const uint32_t *>(L.keys_in);
        S.keys_out = static_cast<uint32_t *>(L.keys_out);
        S.vals_in = L.vals_in;
        S.vals_out = L.vals_out;
        S.n = L.n;
        S.passes = passes;
        S.begin_bit = L.begin_bit;
        S.last_mask = last_mask;
        S.fmask = static_cast<uint32_t>(order.fmask);
        S.flip = static_cast<uint32_t>(order.flip);
        S.alias = alias;
        S.status = status;
        S.abort_flag = abort_flag;
        S.stream = s;
        S.sm_count = L.sm_count;
        record(L.events, L.num_events, 1, s);
        const int rc = launch_cluster_sort(S);
        if (rc != 1) {
            for (int i = 2; i < 3 + passes; ++i) record(L.events, L.num_events, i, s);
            return rc;
        }
    }
    k_zero_words<<<1, 256, 0, s>>>(hdr, static_cast<uint32_t>(kHdrBytes / sizeof(uint32_t)));
    if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
    if (kb == 8) {
        k_zero_words<<<1, 256, 0, s>>>(hist, 8 * 256);
        if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
    }
    record(L.events, L.num_events, 1, s);

    if (small_sort_applies(L.n, order.key_bytes, L.variant)) {
        SmallSortLaunch S;
        S.keys_in = static_cast<const uint32_t *>(L.keys_in);
        S.keys_out = static_cast<uint32_t *>(L.keys_out);
        S.vals_in = L.vals_in;
        S.vals_out = L.vals_out;
        S.tmp_k = static_cast<uint32_t *>(tmp_k);
        S.tmp_v = tmp_v;
        S.n = L.n;
        S.passes = passes;
        S.begin_bit = L.begin_bit;
        S.last_mask = last_mask;
        S.fmask = static_cast<uint32_t>(order.fmask);
        S.flip = static_cast<uint32_t>(order.flip);
        S.alias = alias;
        S.counts = reinterpret_cast<uint32_t *>(L.ws + lay.small_counts);
        S.bar_count = reinterpret_cast<uint32_t *>(L.ws + kHdrCounters + 128 * 6);
        S.status = status;
        S.abort_flag = abort_flag;
        S.spin_limit = L.spin_limit;
        S.stall_tile = L.stall_tile;
        S.stream = s;
        S.sm_count = L.sm_count;
        const int rc = launch_small_sort(S);
        if (rc != 1) {
            for (int i = 2; i < 3 + passes; ++i) record(L.events, L.num_events, i, s);
            return rc;
        }
    }

    // keys only, every bit: equal keys are indistinguishable, so a warp needs
    // stable ranks only where its keys differ below the current digit
    const bool order_free = !pairs && L.begin_bit == 0 && L.end_bit == static_cast<int>(8 * kb);
    uint32_t *hot = reinterpret_cast<uint32_t *>(L.ws + kHdrHot);
    // the histogram kernel also clears the first pass's look-back words, and
    // its last CTA writes the bin starts, the first pass's cursors and the
    // skewed digits
    BinStartsOut bs;
    bs.start = starts;
    bs.cursor = order_free ? cursor : nullptr;
    bs.hot = hot;
    bs.done = reinterpret_cast<uint32_t *>(L.ws + kHdrHistDone);
    if (launch_hist_any(L.keys_in, L.n, order, L.begin_bit, passes, last_mask, hist, look[0],
                        tiles * 256, s, L.sm_count, bs) != cudaSuccess)
        return GSORT_ECUDA;
    record(L.events, L.num_events, 2, s);

    // In place (either array): in -> tmp -> out -> tmp ...; an odd pass count
    // ends in tmp and is copied back.  Otherwise the sequence is arranged so
    // that the last pass writes to out.
    const void *src_k = L.keys_in;
    const uint32_t *src_v = L.vals_in;
    void *dst_k = nullptr;
    uint32_t *dst_v = nullptr;
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
        a.fmask = order.fmask;
        a.flip = order.flip;
        a.hist = hist + p * 256;
        a.look = look[p & 1];
        a.look_clear = (p + 1 < passes) ? look[(p + 1) & 1] : nullptr;
        a.tile_counter = reinterpret_cast<uint32_t *>(L.ws + kHdrCounters + 128 * p);
        a.status = status;
        a.abort_flag = abort_flag;
        a.spin_limit = L.spin_limit;
        a.stall_tile = L.stall_tile;
        // bulk prefetches need 16-byte aligned sources; about two CTAs per SM are resident
        const bool src16 = (reinterpret_cast<uintptr_t>(src_k) & 15) == 0 &&
                           (!pairs || (reinterpret_cast<uintptr_t>(src_v) & 15) == 0);
        a.prefetch_dist = src16 ? 2u * static_cast<uint32_t>(L.sm_count) : 0u;
        a.order_free = order_free ? 1u : 0u;
        a.free_low = a.shift >= 64 ? ~0ull : ((1ull << a.shift) - 1ull);
        // runs of equal low bits hold about n / 2^shift keys of uniform input;
        // below half a warp's keys (512), two-value warps are rare
        a.two_runs_ok = (a.shift < 32 && (static_cast<uint64_t>(L.n) >> a.shift) >= 256) ? 1u : 0u;
        a.cursor = (a.order_free && p == 0) ? cursor : nullptr;
        a.start = starts + p * 256;
        a.hot = hot + p;
        const bool xin = mapped && p == 0;
        const bool xout = mapped && p == passes - 1;
        const PassLauncher use = a.cursor != nullptr && free_launch != nullptr ? free_launch : launch;
        if (use(a, pairs, xin, xout, tiles, s) != cudaSuccess) return GSORT_ECUDA;
        record(L.events, L.num_events, 3 + p, s);
        src_k = dst_k;
        src_v = dst_v;
    }
    if (dst_k != L.keys_out) {
        if (cudaMemcpyAsync(L.keys_out, dst_k, static_cast<size_t>(L.n) * kb, cudaMemcpyDeviceToDevice, s) !=
            cudaSuccess)
            return GSORT_ECUDA;
        if (pairs && cudaMemcpyAsync(L.vals_out, dst_v, static_cast<size_t>(L.n) * 4,
                                     cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return GSORT_ECUDA;
    }
    return GSORT_OK;
}

int launch_digit_histograms(const void *keys, uint32_t n, int kind, int flags, int begin_bit,
                            int end_bit, uint32_t *hist_out, cudaStream_t stream, int sm_count) {
    const int passes = (end_bit - begin_bit + 7) / 8;
    if (passes == 0) return GSORT_OK;
    k_zero_words<<<1, 256, 0, stream>>>(hist_out, static_cast<uint32_t>(passes * 256));
    if (cudaGetLastError() != cudaSuccess) return GSORT_ECUDA;
    if (n == 0) return GSORT_OK;
    const uint32_t last_width = static_cast<uint32_t>(end_bit - begin_bit - 8 * (passes - 1));
    const uint32_t last_mask = (1u << last_width) - 1u;
    if (launch_hist_any(keys, n, key_order(kind, flags), begin_bit, passes, last_mask, hist_out,
                        nullptr, 0, stream, sm_count) != cudaSuccess)
        return GSORT_ECUDA;
    return GSORT_OK;
}

}  // namespace gsort

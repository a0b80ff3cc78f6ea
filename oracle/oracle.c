/*
 * oracle.c -- plain, slow, obviously-correct CPU restatement of the sorting
 * path.  TEST INFRASTRUCTURE ONLY: nothing in the product library links,
 * includes or calls this file.  Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline leg of bench.py use it.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * Every function cites the passage of the reference pages it follows, by page
 * title and section:
 *   [PMPP10]   "Parallel Patterns: Sorting on the GPU" (textbook chapter 10):
 *              section 10.3 "Radix Sort", 10.6 "Key-Value sorting",
 *              10.7 "stable vs unstable", exercises (section 8).
 *   [CUDA3]    "CUDA 算子笔记 3" (CUDA operator notes 3): sections
 *              "Stream Compaction" and "Radix Sort" (CPU LSD example,
 *              "processing several bits at once").
 *   [WGPU41]   "WebGPU Unleashed 4.1 Radix Sort": three-pass 2-bit sort.
 *   [GPUSORT]  "gpu排序" (GPU sort): bitonic sort of <=1024 keys, padded
 *              with 0xFFFFFFFF.
 *
 * Readings taken where the pages are silent:
 *   - float keys: the pages pose the IEEE-754 preprocessing only as an
 *     exercise ([PMPP10] exercise 7).  The oracle uses the sign-dependent bit
 *     flip, which orders non-NaN values as IEEE totalOrder (-0 before +0).
 *   - begin_bit/end_bit: the key is sorted by bits [begin_bit, end_bit);
 *     other bits are carried unchanged.  Digits are 8 bits wide, the last
 *     digit narrowed to the remaining bits.
 *   - compaction keeps x > 0 under IEEE comparison (NaN, +0 and -0 are
 *     dropped, positive subnormals are kept) and zero-fills the tail with
 *     +0.0, as in the [CUDA3] "Stream Compaction" worked example.
 *
 * Pins: tests/test_oracle_pins.py checks every function here against things
 * other than itself (worked examples printed on the pages, Python's stable
 * sorted(), numpy, brute force over all tiny inputs, invariants).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)

/* ---------------------------------------------------------------------------
 * a0: order-preserving map between IEEE-754 binary32 bit patterns and
 * unsigned 32-bit integers ([PMPP10] exercise 7, reading above).
 * Non-negative floats: set the sign bit (they then rank above all negatives,
 * in the same order as their bits).  Negative floats: complement every bit
 * (a larger magnitude then gives a smaller integer).
 * ------------------------------------------------------------------------- */
uint32_t oracle_f32_bits_to_ordered(uint32_t bits)
{
    if (bits & 0x80000000u)
        return ~bits;
    return bits | 0x80000000u;
}

uint32_t oracle_ordered_to_f32_bits(uint32_t u)
{
    if (u & 0x80000000u)        /* came from a non-negative float */
        return u & 0x7FFFFFFFu;
    return ~u;                  /* came from a negative float */
}

/* The same map applied to an array (used by the exhaustive pin over all 2^32
 * bit patterns, which would be too slow one call at a time). */
void oracle_f32_bits_to_ordered_array(const uint32_t *in, uint32_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_bits_to_ordered(in[i]);
}

void oracle_ordered_to_f32_bits_array(const uint32_t *in, uint32_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_ordered_to_f32_bits(in[i]);
}

/* Number of 8-bit digit passes for the bit range [begin_bit, end_bit):
 * ceil((end_bit - begin_bit) / 8)  ([PMPP10] 10.3, radix 256 needs 4 passes for 32-bit keys). */
int oracle_num_passes(int begin_bit, int end_bit)
{
    if (begin_bit < 0 || end_bit > 32 || begin_bit > end_bit)
        return -1;
    return (end_bit - begin_bit + 7) / 8;
}

/* The p-th digit of key k: bits [begin_bit + 8p, min(begin_bit + 8p + 8, end_bit)). */
static uint32_t digit_of(uint32_t k, int begin_bit, int end_bit, int p)
{
    int lo = begin_bit + 8 * p;
    int width = end_bit - lo;
    if (width > 8)
        width = 8;
    return (uint32_t)(((uint64_t)k >> lo) & ((1u << width) - 1u));
}

/* ---------------------------------------------------------------------------
 * a1: the digit histograms of every pass, from one read of the keys
 * ([CUDA3] "processing several bits at once", kernel 1; [PMPP10] 10.3 step
 * "histogram").  hist has passes*256 entries; hist[p*256 + d] counts the keys
 * whose p-th digit equals d.  kind 1 = float keys (a0 applied first).
 * ------------------------------------------------------------------------- */
int oracle_digit_histograms(const uint32_t *keys, int64_t n, int kind,
                            int begin_bit, int end_bit, uint32_t *hist)
{
    int passes = oracle_num_passes(begin_bit, end_bit);
    if (passes < 0 || n < 0)
        return ORACLE_EINVAL;
    memset(hist, 0, sizeof(uint32_t) * 256 * (size_t)(passes > 0 ? passes : 1));
    for (int64_t i = 0; i < n; ++i) {
        uint32_t k = kind ? oracle_f32_bits_to_ordered(keys[i]) : keys[i];
        for (int p = 0; p < passes; ++p)
            hist[p * 256 + digit_of(k, begin_bit, end_bit, p)] += 1;
    }
    return ORACLE_OK;
}

/* a2: exclusive prefix sum of each pass's 256 bins: base[d] = sum over d' < d
 * of hist[d'] ([PMPP10] 10.3 step "exclusive scan"; [CUDA3] kernel 2). */
void oracle_exclusive_scan_bins(const uint32_t *hist, int passes, uint32_t *base)
{
    for (int p = 0; p < passes; ++p) {
        uint32_t running = 0;
        for (int d = 0; d < 256; ++d) {
            base[p * 256 + d] = running;
            running += hist[p * 256 + d];
        }
    }
}

/* ---------------------------------------------------------------------------
 * a3: stable LSD radix sort of (key, value) pairs by the key bits
 * [begin_bit, end_bit).  One counting-sort pass per 8-bit digit, least
 * significant first: count the digit, exclusive-scan the counts into bucket
 * starts, then move every element, in input order, to the next free slot of
 * its bucket.  Moving in input order is what makes each pass stable, and the
 * stability of every pass is what makes the LSD order correct
 * ([CUDA3] "Radix Sort", CPU version; [PMPP10] 10.3 and 10.7;
 * [WGPU41]: every per-digit reordering has to be stable).  Values move with their
 * keys ([PMPP10] 10.6).  vals_in/vals_out may be NULL (keys only).
 * kind 1 = float keys: a0 before the first pass, its inverse after the last.
 * ------------------------------------------------------------------------- */
int oracle_radix_sort_pairs(const uint32_t *keys_in, const uint32_t *vals_in,
                            uint32_t *keys_out, uint32_t *vals_out, int64_t n,
                            int kind, int begin_bit, int end_bit)
{
    int passes = oracle_num_passes(begin_bit, end_bit);
    if (passes < 0 || n < 0)
        return ORACLE_EINVAL;
    if (n == 0)
        return ORACLE_OK;
    int with_vals = (vals_in != NULL && vals_out != NULL);

    uint32_t *x = malloc(sizeof(uint32_t) * (size_t)n);
    uint32_t *y = malloc(sizeof(uint32_t) * (size_t)n);
    uint32_t *vx = with_vals ? malloc(sizeof(uint32_t) * (size_t)n) : NULL;
    uint32_t *vy = with_vals ? malloc(sizeof(uint32_t) * (size_t)n) : NULL;
    if (!x || !y || (with_vals && (!vx || !vy))) {
        free(x); free(y); free(vx); free(vy);
        return ORACLE_ENOMEM;
    }
    for (int64_t i = 0; i < n; ++i) {
        x[i] = kind ? oracle_f32_bits_to_ordered(keys_in[i]) : keys_in[i];
        if (with_vals)
            vx[i] = vals_in[i];
    }

    for (int p = 0; p < passes; ++p) {
        uint32_t count[256];
        uint32_t next[256];
        memset(count, 0, sizeof(count));
        for (int64_t i = 0; i < n; ++i)
            count[digit_of(x[i], begin_bit, end_bit, p)] += 1;
        uint32_t running = 0;
        for (int d = 0; d < 256; ++d) {
            next[d] = running;
            running += count[d];
        }
        for (int64_t i = 0; i < n; ++i) {
            uint32_t d = digit_of(x[i], begin_bit, end_bit, p);
            uint32_t slot = next[d]++;
            y[slot] = x[i];
            if (with_vals)
                vy[slot] = vx[i];
        }
        uint32_t *t = x; x = y; y = t;
        if (with_vals) { t = vx; vx = vy; vy = t; }
    }

    for (int64_t i = 0; i < n; ++i) {
        keys_out[i] = kind ? oracle_ordered_to_f32_bits(x[i]) : x[i];
        if (with_vals)
            vals_out[i] = vx[i];
    }
    free(x); free(y); free(vx); free(vy);
    return ORACLE_OK;
}

/* Keys only, all 32 bits. */
int oracle_radix_sort_keys(const uint32_t *keys_in, uint32_t *keys_out,
                           int64_t n, int kind)
{
    return oracle_radix_sort_pairs(keys_in, NULL, keys_out, NULL, n, kind, 0, 32);
}

/* ---------------------------------------------------------------------------
 * NEXT (f1): every key kind, ascending or descending.
 *   kinds: 0 u32, 1 f32, 2 i32, 3 u64, 4 f64, 5 i64 (4- or 8-byte words).
 * The key is replaced by an unsigned "ordered" value of its own width whose
 * unsigned order is the wanted order, sorted by the same stable LSD counting
 * passes as above ([CUDA3] "Radix Sort", CPU version), and mapped back.
 *   - signed: value + 2^(w-1), i.e. the signed range shifted onto the
 *     unsigned one (the pages do not cover signed keys; this is the plain
 *     reading of "sort the signed values");
 *   - float: the IEEE totalOrder map of a0, at 32 or 64 bits ([PMPP10]
 *     exercise 7);
 *   - descending: (2^w - 1) - ordered, which reverses the order of distinct
 *     values and leaves equal values equal, so the stable passes keep equal
 *     keys in input order ([PMPP10] exercise 6);
 *   - 64-bit keys take (end_bit - begin_bit)/8 = 8 passes for the whole key
 *     ([PMPP10] exercise 2: radix 256 on 64-bit integers).
 * ------------------------------------------------------------------------- */
int oracle_kind_bytes(int kind)
{
    switch (kind) {
    case 0: case 1: case 2: return 4;
    case 3: case 4: case 5: return 8;
    default: return 0;
    }
}

uint64_t oracle_key_to_ordered(uint64_t bits, int kind, int descending)
{
    uint64_t u;
    int w = oracle_kind_bytes(kind) * 8;
    switch (kind) {
    case 0: u = bits & 0xFFFFFFFFull; break;
    case 1: u = oracle_f32_bits_to_ordered((uint32_t)bits); break;
    case 2: u = (uint64_t)((int64_t)(int32_t)(uint32_t)bits + 2147483648LL); break;
    case 3: u = bits; break;
    case 4:
        if (bits >> 63)
            u = ~bits;
        else
            u = bits | 0x8000000000000000ull;
        break;
    case 5: u = bits + 0x8000000000000000ull; break;   /* value + 2^63, modulo 2^64 */
    default: return 0;
    }
    if (descending)
        u = (w == 64 ? 0xFFFFFFFFFFFFFFFFull : 0xFFFFFFFFull) - u;
    return u;
}

uint64_t oracle_ordered_to_key(uint64_t u, int kind, int descending)
{
    int w = oracle_kind_bytes(kind) * 8;
    if (descending)
        u = (w == 64 ? 0xFFFFFFFFFFFFFFFFull : 0xFFFFFFFFull) - u;
    switch (kind) {
    case 0: return u & 0xFFFFFFFFull;
    case 1: return oracle_ordered_to_f32_bits((uint32_t)u);
    case 2: return (uint64_t)(uint32_t)(int32_t)((int64_t)u - 2147483648LL);
    case 3: return u;
    case 4:
        if (u >> 63)
            return u & 0x7FFFFFFFFFFFFFFFull;
        return ~u;
    case 5: return u - 0x8000000000000000ull;
    default: return 0;
    }
}

static uint64_t load_key(const void *keys, int64_t i, int kb)
{
    if (kb == 4)
        return ((const uint32_t *)keys)[i];
    return ((const uint64_t *)keys)[i];
}

static void store_key(void *keys, int64_t i, int kb, uint64_t v)
{
    if (kb == 4)
        ((uint32_t *)keys)[i] = (uint32_t)v;
    else
        ((uint64_t *)keys)[i] = v;
}

/* The p-th digit of a 64-bit ordered value: bits [begin_bit + 8p, min(+8, end_bit)). */
static uint32_t digit_of64(uint64_t k, int begin_bit, int end_bit, int p)
{
    int lo = begin_bit + 8 * p;
    int width = end_bit - lo;
    if (width > 8)
        width = 8;
    return (uint32_t)((k >> lo) & ((1ull << width) - 1ull));
}

int oracle_digit_histograms_general(const void *keys, int64_t n, int kind, int flags,
                                    int begin_bit, int end_bit, uint32_t *hist)
{
    int kb = oracle_kind_bytes(kind);
    if (kb == 0 || n < 0 || begin_bit < 0 || end_bit > 8 * kb || begin_bit > end_bit)
        return ORACLE_EINVAL;
    int passes = (end_bit - begin_bit + 7) / 8;
    memset(hist, 0, sizeof(uint32_t) * 256 * (size_t)(passes > 0 ? passes : 1));
    for (int64_t i = 0; i < n; ++i) {
        uint64_t k = oracle_key_to_ordered(load_key(keys, i, kb), kind, flags & 1);
        for (int p = 0; p < passes; ++p)
            hist[p * 256 + digit_of64(k, begin_bit, end_bit, p)] += 1;
    }
    return ORACLE_OK;
}

int oracle_radix_sort_general(const void *keys_in, const uint32_t *vals_in,
                              void *keys_out, uint32_t *vals_out, int64_t n,
                              int kind, int flags, int begin_bit, int end_bit)
{
    int kb = oracle_kind_bytes(kind);
    if (kb == 0 || n < 0 || (flags & ~1) != 0 || begin_bit < 0 || end_bit > 8 * kb ||
        begin_bit > end_bit)
        return ORACLE_EINVAL;
    if (n == 0)
        return ORACLE_OK;
    int passes = (end_bit - begin_bit + 7) / 8;
    int with_vals = (vals_in != NULL && vals_out != NULL);
    uint64_t *x = malloc(sizeof(uint64_t) * (size_t)n);
    uint64_t *y = malloc(sizeof(uint64_t) * (size_t)n);
    uint32_t *vx = with_vals ? malloc(sizeof(uint32_t) * (size_t)n) : NULL;
    uint32_t *vy = with_vals ? malloc(sizeof(uint32_t) * (size_t)n) : NULL;
    if (!x || !y || (with_vals && (!vx || !vy))) {
        free(x); free(y); free(vx); free(vy);
        return ORACLE_ENOMEM;
    }
    for (int64_t i = 0; i < n; ++i) {
        x[i] = oracle_key_to_ordered(load_key(keys_in, i, kb), kind, flags & 1);
        if (with_vals)
            vx[i] = vals_in[i];
    }
    for (int p = 0; p < passes; ++p) {
        uint32_t count[256];
        uint32_t next[256];
        memset(count, 0, sizeof(count));
        for (int64_t i = 0; i < n; ++i)
            count[digit_of64(x[i], begin_bit, end_bit, p)] += 1;
        uint32_t running = 0;
        for (int d = 0; d < 256; ++d) {
            next[d] = running;
            running += count[d];
        }
        for (int64_t i = 0; i < n; ++i) {
            uint32_t slot = next[digit_of64(x[i], begin_bit, end_bit, p)]++;
            y[slot] = x[i];
            if (with_vals)
                vy[slot] = vx[i];
        }
        uint64_t *t = x; x = y; y = t;
        if (with_vals) { uint32_t *tv = vx; vx = vy; vy = tv; }
    }
    for (int64_t i = 0; i < n; ++i) {
        store_key(keys_out, i, kb, oracle_ordered_to_key(x[i], kind, flags & 1));
        if (with_vals)
            vals_out[i] = vx[i];
    }
    free(x); free(y); free(vx); free(vy);
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * NEXT (f2): variable-length segments.  Segment s is [offsets[s],
 * offsets[s+1]); the offsets must start at 0, never decrease and end at n.
 * Each segment is sorted on its own by the stable sort above (every 32-bit
 * kind, either direction), which is the definition of a stable segmented
 * sort ([PMPP10] 10.5 names the hybrid strategy; the result it must reach is
 * each piece sorted).  Returns ORACLE_EINVAL for offsets that break the rules.
 * ------------------------------------------------------------------------- */
int oracle_segmented_sort_general(const uint32_t *keys_in, const uint32_t *vals_in,
                                  uint32_t *keys_out, uint32_t *vals_out, int64_t n,
                                  const uint32_t *offsets, int64_t num_segments,
                                  int kind, int flags)
{
    if (oracle_kind_bytes(kind) != 4 || n < 0 || num_segments < 0)
        return ORACLE_EINVAL;
    if (n == 0)
        return ORACLE_OK;
    if (num_segments == 0 || offsets[0] != 0 || offsets[num_segments] != (uint32_t)n)
        return ORACLE_EINVAL;
    for (int64_t s = 0; s < num_segments; ++s)
        if (offsets[s + 1] < offsets[s])
            return ORACLE_EINVAL;
    int with_vals = (vals_in != NULL && vals_out != NULL);
    for (int64_t s = 0; s < num_segments; ++s) {
        uint32_t a = offsets[s];
        int64_t len = (int64_t)offsets[s + 1] - a;
        int rc = oracle_radix_sort_general(keys_in + a, with_vals ? vals_in + a : NULL,
                                           keys_out + a, with_vals ? vals_out + a : NULL,
                                           len, kind, flags, 0, 32);
        if (rc != ORACLE_OK)
            return rc;
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * NEXT (f3): stable 2-way split and the 1-bit split sort ([CUDA3] "Radix
 * Sort": per bit a predicate, a scan and a scatter of the zeros before the
 * ones).  oracle_partition copies the elements whose predicate holds, in
 * input order, then the others, in input order, and returns their count.
 * Predicates (pred): 0 flags[i] != 0; 1 bit `param` set; 2 bit `param`
 * clear; 3 x before param in the sort order of `kind` (the ordered values of
 * f1 compared); 4 x > 0 as a float (C comparison).
 * ------------------------------------------------------------------------- */
static int pred_holds(uint32_t x, int64_t i, int pred, int kind, uint32_t param,
                      const uint8_t *flags)
{
    switch (pred) {
    case 0: return flags[i] != 0;
    case 1: return ((x >> param) & 1u) == 1u;
    case 2: return ((x >> param) & 1u) == 0u;
    case 3: return oracle_key_to_ordered(x, kind, 0) < oracle_key_to_ordered(param, kind, 0);
    default: {
        float f;
        memcpy(&f, &x, sizeof(f));
        return f > 0.0f;
    }
    }
}

int64_t oracle_partition(const uint32_t *in, const uint32_t *vals_in, uint32_t *out,
                         uint32_t *vals_out, int64_t n, int pred, int kind, uint32_t param,
                         const uint8_t *flags)
{
    int with_vals = (vals_in != NULL && vals_out != NULL);
    int64_t m = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (pred_holds(in[i], i, pred, kind, param, flags)) {
            out[m] = in[i];
            if (with_vals)
                vals_out[m] = vals_in[i];
            ++m;
        }
    }
    int64_t k = m;
    for (int64_t i = 0; i < n; ++i) {
        if (!pred_holds(in[i], i, pred, kind, param, flags)) {
            out[k] = in[i];
            if (with_vals)
                vals_out[k] = vals_in[i];
            ++k;
        }
    }
    return m;
}

/* One stable split per bit b in [begin_bit, end_bit), zeros first. */
int oracle_split_sort(const uint32_t *keys_in, const uint32_t *vals_in, uint32_t *keys_out,
                      uint32_t *vals_out, int64_t n, int begin_bit, int end_bit)
{
    if (n < 0 || begin_bit < 0 || end_bit > 32 || begin_bit > end_bit)
        return ORACLE_EINVAL;
    int with_vals = (vals_in != NULL && vals_out != NULL);
    uint32_t *x = malloc(sizeof(uint32_t) * (size_t)(n > 0 ? n : 1));
    uint32_t *y = malloc(sizeof(uint32_t) * (size_t)(n > 0 ? n : 1));
    uint32_t *vx = malloc(sizeof(uint32_t) * (size_t)(n > 0 ? n : 1));
    uint32_t *vy = malloc(sizeof(uint32_t) * (size_t)(n > 0 ? n : 1));
    if (!x || !y || !vx || !vy) {
        free(x); free(y); free(vx); free(vy);
        return ORACLE_ENOMEM;
    }
    for (int64_t i = 0; i < n; ++i) {
        x[i] = keys_in[i];
        vx[i] = with_vals ? vals_in[i] : 0u;
    }
    for (int b = begin_bit; b < end_bit; ++b) {
        oracle_partition(x, vx, y, vy, n, 2, 0, (uint32_t)b, NULL);
        uint32_t *t = x; x = y; y = t;
        t = vx; vx = vy; vy = t;
    }
    for (int64_t i = 0; i < n; ++i) {
        keys_out[i] = x[i];
        if (with_vals)
            vals_out[i] = vx[i];
    }
    free(x); free(y); free(vx); free(vy);
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * a4: stream compaction, the 1-bit special case ([CUDA3] "Stream
 * Compaction": predicate, exclusive scan of the predicate, scatter).  Keeps
 * every x > 0 in input order at out[0..m), writes +0.0 to out[m..n), and
 * returns m.  The comparison is the C float comparison, which follows IEEE:
 * NaN > 0 is false, -0.0 > 0 is false, a positive subnormal > 0 is true.
 * in and out are float arrays passed as their bit patterns.
 * ------------------------------------------------------------------------- */
int64_t oracle_compact_positive(const uint32_t *in_bits, uint32_t *out_bits, int64_t n)
{
    int64_t m = 0;
    for (int64_t i = 0; i < n; ++i) {
        float x;
        memcpy(&x, &in_bits[i], sizeof(x));
        if (x > 0.0f) {
            /* out position = exclusive prefix count of kept elements */
            out_bits[m] = in_bits[i];
            m += 1;
        }
    }
    for (int64_t i = m; i < n; ++i)
        out_bits[i] = 0x00000000u;     /* +0.0f */
    return m;
}

/* ---------------------------------------------------------------------------
 * a5 (definition): each of num_segments consecutive segments of
 * segment_len unsigned keys sorted ascending, independently, in place
 * ([GPUSORT] bitonic sort of <=1024 elements; [PMPP10] 10.2).  A keys-only
 * ascending sort has a unique result, so the oracle is that definition,
 * reached here with the same plain LSD counting sort as above.
 * ------------------------------------------------------------------------- */
int oracle_segmented_sort(uint32_t *keys, int64_t num_segments, int segment_len)
{
    if (num_segments < 0 || segment_len < 0)
        return ORACLE_EINVAL;
    for (int64_t s = 0; s < num_segments; ++s) {
        uint32_t *seg = keys + s * (int64_t)segment_len;
        int rc = oracle_radix_sort_keys(seg, seg, segment_len, 0);
        if (rc != ORACLE_OK)
            return rc;
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * a5 (network): the bitonic sorting network on one array whose length is a
 * power of two, as the pages define it ([GPUSORT] "binoticSort"; [PMPP10]
 * 10.2): for block size k = 2, 4, ..., len and distance j = k/2, ..., 1,
 * every element i whose partner i^j lies above it is compare-exchanged with
 * that partner, ascending when bit k of i is clear and descending when it is
 * set.  Used only to pin that the network (with 0xFFFFFFFF padding) sorts,
 * by the 0-1 principle; the parity oracle for segments is the definition
 * above.
 * ------------------------------------------------------------------------- */
int oracle_bitonic_network(uint32_t *a, int len)
{
    if (len <= 0 || (len & (len - 1)) != 0)
        return ORACLE_EINVAL;
    for (int k = 2; k <= len; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = 0; i < len; ++i) {
                int partner = i ^ j;
                if (partner <= i)
                    continue;
                int ascending = (i & k) == 0;
                uint32_t lo = a[i], hi = a[partner];
                if ((ascending && lo > hi) || (!ascending && lo < hi)) {
                    a[i] = hi;
                    a[partner] = lo;
                }
            }
        }
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * Cross-check at another digit width: the three-pass 2-bit radix sort of
 * [WGPU41], restated on the CPU.  Keys are padded with 0xFFFFFFFF to a
 * multiple of 512 (one chunk per workgroup of 256 invocations x 2 keys).
 * For each of the 16 two-bit digits:
 *   pass 1: inside each chunk, the exclusive running count of each digit
 *           value before every key (the local prefix sum), and the chunk's
 *           count of each value (the list of chunk sums);
 *   pass 2: an inclusive prefix sum of the chunk counts over the chunks,
 *           per digit value (pass 3 reads entry c-1 as the count over all chunks
 *           before c and the last entry as the overall total);
 *   pass 3: position = (keys with a smaller digit value, over all chunks)
 *           + (keys with this value in earlier chunks) + local prefix;
 *           the key and its id are written there.
 * ids travel with the keys (the page's inputId/outputId).  Only the first n
 * outputs are returned; padding keys sort after every real key because they
 * sit after all real keys in the input and every pass is stable.
 * ------------------------------------------------------------------------- */
int oracle_radix2_three_pass(const uint32_t *keys_in, const uint32_t *ids_in,
                             uint32_t *keys_out, uint32_t *ids_out, int64_t n)
{
    const int64_t chunk = 512;
    if (n < 0)
        return ORACLE_EINVAL;
    if (n == 0)
        return ORACLE_OK;
    int64_t chunks = (n + chunk - 1) / chunk;
    int64_t padded = chunks * chunk;

    uint32_t *key = malloc(sizeof(uint32_t) * (size_t)padded);
    uint32_t *id = malloc(sizeof(uint32_t) * (size_t)padded);
    uint32_t *key2 = malloc(sizeof(uint32_t) * (size_t)padded);
    uint32_t *id2 = malloc(sizeof(uint32_t) * (size_t)padded);
    uint32_t *local = malloc(sizeof(uint32_t) * (size_t)padded);   /* local prefix of the key's own digit */
    uint64_t *sums = malloc(sizeof(uint64_t) * (size_t)chunks * 4);
    if (!key || !id || !key2 || !id2 || !local || !sums) {
        free(key); free(id); free(key2); free(id2); free(local); free(sums);
        return ORACLE_ENOMEM;
    }
    for (int64_t i = 0; i < padded; ++i) {
        key[i] = i < n ? keys_in[i] : 0xFFFFFFFFu;
        id[i] = i < n ? ids_in[i] : (uint32_t)i;
    }

    for (int radix_id = 0; radix_id < 16; ++radix_id) {
        int shift = radix_id * 2;
        /* pass 1 */
        for (int64_t c = 0; c < chunks; ++c) {
            uint64_t run[4] = {0, 0, 0, 0};
            for (int64_t t = 0; t < chunk; ++t) {
                int64_t i = c * chunk + t;
                uint32_t v = (key[i] >> shift) & 3u;
                local[i] = (uint32_t)run[v];
                run[v] += 1;
            }
            for (int v = 0; v < 4; ++v)
                sums[c * 4 + v] = run[v];
        }
        /* pass 2: inclusive scan over chunks */
        for (int64_t c = 1; c < chunks; ++c)
            for (int v = 0; v < 4; ++v)
                sums[c * 4 + v] += sums[(c - 1) * 4 + v];
        /* pass 3 */
        uint64_t below_value[4];
        uint64_t acc = 0;
        for (int v = 0; v < 4; ++v) {
            below_value[v] = acc;
            acc += sums[(chunks - 1) * 4 + v];
        }
        for (int64_t c = 0; c < chunks; ++c) {
            for (int64_t t = 0; t < chunk; ++t) {
                int64_t i = c * chunk + t;
                uint32_t v = (key[i] >> shift) & 3u;
                uint64_t before_chunk = c > 0 ? sums[(c - 1) * 4 + v] : 0;
                uint64_t pos = below_value[v] + before_chunk + local[i];
                key2[pos] = key[i];
                id2[pos] = id[i];
            }
        }
        uint32_t *t;
        t = key; key = key2; key2 = t;
        t = id; id = id2; id2 = t;
    }
    for (int64_t i = 0; i < n; ++i) {
        keys_out[i] = key[i];
        ids_out[i] = id[i];
    }
    free(key); free(id); free(key2); free(id2); free(local); free(sums);
    return ORACLE_OK;
}

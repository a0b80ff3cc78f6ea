/*
 * gsort.h -- C ABI of libgsort.so: GB300 (sm_103a) stable LSD radix sort,
 * stream compaction and segmented bitonic sort.
 *
 * Sources of the operations (reference pages, by title and section):
 *   [PMPP10]  "Parallel Patterns: Sorting on the GPU" (textbook chapter 10):
 *             10.2 Bitonic Sort, 10.3 Radix Sort, 10.6 Key-Value sorting,
 *             10.7 stable vs unstable sorting, section 8 exercises.
 *   [CUDA3]   "CUDA 算子笔记 3" (CUDA operator notes 3): Stream Compaction
 *             (three kernels; decoupled look-back), Radix Sort (CPU LSD
 *             sort; processing several bits at once: histogram of every
 *             pass, scan of the bins, one-pass scatter with look-back).
 *   [WGPU41]  "WebGPU Unleashed 4.1 Radix Sort": key/id pair buffers,
 *             stable per-digit reordering.
 *   [GPUSORT] "gpu排序" (GPU sort): bitonic sort of <=1024 keys per block,
 *             padded with 0xFFFFFFFF.
 *
 * Conventions shared by every call:
 *   - Pointers named d_* are DEVICE pointers on the current CUDA device.
 *     The caller owns every buffer, including the workspace; the library
 *     never allocates or frees memory and keeps no state between calls.
 *   - Every call is asynchronous on `stream` (0 = legacy default stream).
 *     Argument errors and launch errors are returned at once.  Errors that
 *     only the device can see (a look-back wait that gave up) are recorded
 *     in the workspace and returned by gsort_check().
 *   - 32-bit data must be 4-byte aligned (else GSORT_EALIGN).  Buffers that
 *     are also 16-byte aligned take 128-bit vector paths; others take a
 *     scalar path with identical results.
 *   - n counts elements.  0 <= n <= GSORT_MAX_N (larger: GSORT_ETOOBIG);
 *     n == 0 is a no-op returning GSORT_OK.  The cap comes from the 30-bit
 *     count field of the look-back state words.
 *   - Workspaces must be 256-byte aligned (torch and cudaMalloc allocations
 *     are).  Their contents on entry do not matter.  Two calls that share a
 *     workspace must not run concurrently.
 */
#ifndef GSORT_H
#define GSORT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same definition as the CUDA runtime's, so either header may come first. */
typedef struct CUstream_st *cudaStream_t;

typedef enum gsort_status {
    GSORT_OK = 0,
    GSORT_EINVAL = -1,      /* bad argument: NULL, bad range, overlapping buffers */
    GSORT_EALIGN = -2,      /* a pointer is not 4-byte (data) or 256-byte (workspace) aligned */
    GSORT_EWORKSPACE = -3,  /* workspace missing or smaller than the *_workspace_bytes() answer */
    GSORT_ETOOBIG = -4,     /* n above the entry point's maximum (GSORT_MAX_N, or the smaller limit it states) */
    GSORT_ECUDA = -5,       /* a CUDA runtime call or kernel launch failed */
    GSORT_ETIMEOUT = -6     /* a device-side look-back wait gave up (see gsort_check) */
} gsort_status;

typedef enum gsort_key_kind {
    GSORT_KEY_U32 = 0,      /* unsigned 32-bit integers */
    GSORT_KEY_F32 = 1,      /* IEEE-754 binary32, ordered as totalOrder for non-NaN */
    GSORT_KEY_I32 = 2,      /* two's-complement 32-bit integers */
    GSORT_KEY_U64 = 3,      /* unsigned 64-bit integers */
    GSORT_KEY_F64 = 4,      /* IEEE-754 binary64, ordered as totalOrder for non-NaN */
    GSORT_KEY_I64 = 5       /* two's-complement 64-bit integers */
} gsort_key_kind;

/* Flags of gsort_radix_sort(). */
#define GSORT_DESCENDING 1  /* largest key first; equal keys keep their input order */

#define GSORT_MAX_N ((int64_t)((1 << 30) - 1))

/* Human-readable name of a status code (static string). */
const char *gsort_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int gsort_version(void);

/* ------------------------------------------------------------------------
 * Radix sort  ([PMPP10] 10.3, 10.6, 10.7; [CUDA3] Radix Sort, several bits
 * at once; [WGPU41])
 *
 * Stable LSD radix sort with 8-bit digits, least significant digit first.
 * One upfront pass reads the keys once and builds the 256-bin histogram of
 * every digit; each digit pass then scatters every element to
 *   (keys with a smaller digit) + (keys with this digit in earlier tiles)
 *   + (its stable rank among this digit's keys in its own tile),
 * where the middle term comes from a decoupled look-back over per-(tile,
 * digit) counts.  Equal keys keep their input order; values move with keys.
 *
 * Keys only, sorted by every bit of the key: equal keys are identical, so a
 * pass needs the input order only between keys that differ in the bits
 * below its digit.  There the first pass places keys in any order within
 * their bin (atomic bin cursors instead of the look-back), and a warp whose
 * keys agree below the digit ranks them by shared atomics instead of the
 * multisplit.  The output is the same (a sorted key sequence is unique);
 * the intermediate order may differ from run to run.
 *
 * Float keys (GSORT_KEY_F32): the bit pattern is mapped to an unsigned
 * integer that orders every non-NaN value as IEEE totalOrder (-inf < ... <
 * -0 < +0 < ... < +inf); the output holds the original bit patterns.
 * ([PMPP10] section 8, exercise 7 poses the question; this is the reading
 * taken.)  NaNs are not promised an order; with this map +NaN sorts after
 * +inf and -NaN before -inf.
 * ---------------------------------------------------------------------- */

/* Workspace bytes for sorting n elements (with_values != 0: pairs).
 * Holds a status word, counters, the digit histograms, two look-back
 * state regions and one ping-pong buffer per sorted array. */
size_t gsort_radix_workspace_bytes(int64_t n, int with_values);

/* Sort n 32-bit keys (kind GSORT_KEY_U32, F32 or I32) ascending by all 32
 * bits.  d_keys_in is not modified unless it equals d_keys_out (in place is
 * allowed).  Partially overlapping buffers: GSORT_EINVAL. */
int gsort_radix_keys(const void *d_keys_in, void *d_keys_out, int64_t n,
                     int kind, void *d_ws, size_t ws_bytes, cudaStream_t stream);

/* Stable sort of (key, value) pairs by key bits [begin_bit, end_bit)
 * (0 <= begin_bit <= end_bit <= 32) for the 32-bit kinds U32, F32 and I32
 * (other kinds: GSORT_EINVAL; gsort_radix_sort takes every kind).  Bits
 * outside the range do not take part in the order but are carried.
 * begin_bit == end_bit copies.  For F32 and I32 the range applies to the
 * mapped key (use 0..32).
 * d_vals_in and d_vals_out are both NULL (keys only) or both non-NULL.
 * In-place (in == out) is allowed for keys and for values. */
int gsort_radix_pairs(const void *d_keys_in, void *d_keys_out,
                      const uint32_t *d_vals_in, uint32_t *d_vals_out, int64_t n,
                      int kind, int begin_bit, int end_bit,
                      void *d_ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * General radix sort: every key kind, ascending or descending.
 * ([PMPP10] section 8, exercises 2 (64-bit keys: 8 passes of radix 256),
 * 6 (descending order) and 7 (float keys); signed keys flip the sign bit,
 * the same idea for two's complement.)
 *
 * Stable sort of n keys of `kind` (4- or 8-byte words, see gsort_key_kind),
 * with optional 32-bit values, by the bits [begin_bit, end_bit) of the
 * mapped key: the key's bit pattern taken through the order map of its kind
 * (identity for unsigned, sign bit flipped for signed, the totalOrder map for
 * floats), complemented when flags has GSORT_DESCENDING.  0 <= begin_bit <=
 * end_bit <= 8 * key bytes; 0..32 or 0..64 sorts by the whole key.  Equal
 * (masked) keys keep their input order in both directions.  Output keys
 * hold the original bit patterns.
 *
 * Keys must be aligned to their size (else GSORT_EALIGN), values to 4 bytes.
 * In place, aliasing and NULL rules as for gsort_radix_pairs.  flags other
 * than 0 and GSORT_DESCENDING: GSORT_EINVAL.  The workspace comes from
 * gsort_radix_sort_workspace_bytes() with the same kind; for 32-bit kinds it
 * equals gsort_radix_workspace_bytes().
 * ---------------------------------------------------------------------- */
size_t gsort_radix_sort_workspace_bytes(int64_t n, int kind, int with_values);

int gsort_radix_sort(const void *d_keys_in, void *d_keys_out,
                     const uint32_t *d_vals_in, uint32_t *d_vals_out, int64_t n,
                     int kind, int flags, int begin_bit, int end_bit,
                     void *d_ws, size_t ws_bytes, cudaStream_t stream);

/* The upfront histogram step on its own: d_hist_out receives
 * passes * 256 uint32 counts, passes = ceil((end_bit - begin_bit) / 8);
 * entry [p * 256 + d] counts the keys whose p-th 8-bit digit (from
 * begin_bit, last digit narrowed to end_bit) of the mapped key (ascending
 * order map of `kind`, any kind; end_bit <= 8 * key bytes) is d.  Needs no
 * workspace. */
int gsort_digit_histograms(const void *d_keys, int64_t n, int kind,
                           int begin_bit, int end_bit, uint32_t *d_hist_out,
                           cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Stream compaction  ([CUDA3] Stream Compaction: predicate, exclusive scan,
 * scatter; the single-pass decoupled look-back version)
 *
 * Writes every d_in[i] > 0 (IEEE: NaN, +0 and -0 are dropped, positive
 * subnormals kept) to d_out[0..m) in input order and +0.0 to d_out[m..n).
 * If d_num_kept is not NULL, *d_num_kept = m (device int64) on completion.
 * d_in and d_out must not overlap.
 * ---------------------------------------------------------------------- */
size_t gsort_compact_workspace_bytes(int64_t n);

int gsort_compact_positive(const float *d_in, float *d_out, int64_t n,
                           int64_t *d_num_kept, void *d_ws, size_t ws_bytes,
                           cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Allocation-free compaction.  The reference pages have no counterpart: this
 * call exists for callers that cannot provide a workspace, because they run
 * where device allocation is forbidden or too costly (the execute step of a
 * plugin whose host framework owns all device memory, a real-time loop that
 * cannot afford cudaMalloc's device-wide synchronisation and latency, a
 * handler that runs while the caller's allocator is busy).
 *
 * Same result as gsort_compact_positive, for 0 <= n <=
 * GSORT_COMPACT_NOALLOC_MAX_N (larger: GSORT_ETOOBIG).  The caller still
 * passes the input, the output and the optional kept count.  The scratch is
 * one static device array inside the library (about 4 MiB), which every GPU
 * that loads the library keeps until the process exits; this call allocates
 * nothing.  The first call on a device looks up that array's device address
 * (make that first call before any stream capture); later calls reuse it.
 * All calls share the array: calls whose work overlaps on the GPU (for
 * example on two streams at once) race and corrupt each other's results, so
 * serialise them.  A device-side look-back timeout, which does not occur in
 * normal operation, leaves the output undefined and is not reported here.
 * ---------------------------------------------------------------------- */
#define GSORT_COMPACT_NOALLOC_MAX_N ((int64_t)1 << 28)

int gsort_compact_positive_noalloc(const float *d_in, float *d_out, int64_t n,
                                   int64_t *d_num_kept, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Segmented bitonic sort  ([GPUSORT] sort of <=1024 elements in one block;
 * [PMPP10] 10.2)
 *
 * Sorts each of num_segments consecutive segments of segment_len uint32
 * keys ascending, in place, with the bitonic network held in registers
 * (one warp per segment).  1 <= segment_len <= 1024; lengths that are not a
 * power of two are padded internally with 0xFFFFFFFF.  num_segments >= 0.
 * Not stable (keys only, so the result is still unique).
 * ---------------------------------------------------------------------- */
int gsort_segmented_bitonic(uint32_t *d_keys, int64_t num_segments,
                            int segment_len, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Stable 2-way split (partition)  ([CUDA3] "Radix Sort": predicate,
 * exclusive scan, scatter of one side before the other; "Stream
 * Compaction" keeps only one side)
 *
 * Writes every element whose predicate holds, in input order, to
 * d_out[0..m) and every other element, in input order, to d_out[m..n);
 * values (optional, 32-bit) move with their elements; *d_num_true = m
 * (device int64, may be NULL).  d_in/d_vals_in must not overlap the outputs.
 * Predicates on the 32-bit word x of element i:
 *   GSORT_PRED_FLAGS       d_flags[i] != 0 (uint8 array of n entries)
 *   GSORT_PRED_BIT_SET     bit `param` of x is 1 (param < 32)
 *   GSORT_PRED_BIT_CLEAR   bit `param` of x is 0
 *   GSORT_PRED_LESS        x < param in the sort order of `kind` (U32, I32,
 *                          F32: IEEE totalOrder, so -0.0 < +0.0 and NaNs
 *                          fall outside +-inf, as in the radix sort)
 *   GSORT_PRED_POSITIVE    IEEE x > 0 for float bits (the compaction
 *                          predicate; NaN, +0 and -0 are false)
 * Traffic: one counting read, then one read and one write per element.
 * ---------------------------------------------------------------------- */
#define GSORT_PRED_FLAGS 0
#define GSORT_PRED_BIT_SET 1
#define GSORT_PRED_BIT_CLEAR 2
#define GSORT_PRED_LESS 3
#define GSORT_PRED_POSITIVE 4

size_t gsort_partition_workspace_bytes(int64_t n);

int gsort_partition(const uint32_t *d_in, uint32_t *d_out, const uint32_t *d_vals_in,
                    uint32_t *d_vals_out, int64_t n, int pred, int kind, uint32_t param,
                    const uint8_t *d_flags, int64_t *d_num_true, void *d_ws, size_t ws_bytes,
                    cudaStream_t stream);

/* ------------------------------------------------------------------------
 * 1-bit split radix sort  ([CUDA3] "Radix Sort": one predicate / scan /
 * scatter pass per bit, zeros before ones)
 *
 * Stable ascending sort of unsigned 32-bit keys (and 32-bit values) by the
 * bits [begin_bit, end_bit), one split pass per bit (up to 32): the pages'
 * bitwise LSD sort.  The zero count of every bit comes from one upfront
 * histogram read.  Same result as gsort_radix_pairs with GSORT_KEY_U32, at
 * about 8x its traffic; it exists as the pages' method and as a check of
 * the split primitive.  In place and aliasing rules as for
 * gsort_radix_pairs.
 * ---------------------------------------------------------------------- */
size_t gsort_split_sort_workspace_bytes(int64_t n, int with_values);

int gsort_split_sort(const uint32_t *d_keys_in, uint32_t *d_keys_out,
                     const uint32_t *d_vals_in, uint32_t *d_vals_out, int64_t n,
                     int begin_bit, int end_bit, void *d_ws, size_t ws_bytes,
                     cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Variable-length segmented sort  ([PMPP10] 10.5, strategy 2: radix sort
 * for the coarse order with bitonic networks for the small pieces;
 * [GPUSORT]: pieces of <= 1024 keys go to a bitonic sort)
 *
 * d_offsets holds num_segments + 1 uint32 entries with d_offsets[0] == 0,
 * d_offsets[s] <= d_offsets[s + 1] and d_offsets[num_segments] == n; segment
 * s is keys [d_offsets[s], d_offsets[s + 1]).  Each segment is sorted
 * stably by the whole key of `kind` (32-bit kinds: GSORT_KEY_U32, F32, I32;
 * others: GSORT_EINVAL), ascending, or descending with GSORT_DESCENDING;
 * equal keys keep their input order and values (optional, 32-bit) move
 * with their keys.  Segments of 2..1024 keys are sorted by one warp each
 * (register bitonic network; with values it sorts (key, position) pairs,
 * which makes it stable); longer segments by a radix sort whose tiles never
 * cross a segment boundary.  Empty segments are allowed.
 *
 * Offsets are read on the device: offsets that break the rules above make
 * the call record GSORT_EINVAL in the workspace (returned by gsort_check)
 * and leave the output unspecified; no memory outside the given arrays is
 * touched.  n == 0 is a no-op (the offsets are not read); num_segments == 0
 * requires n == 0.  In place (in == out, for keys and for values) is
 * allowed; other overlaps: GSORT_EINVAL.  The workspace comes from
 * gsort_segmented_sort_workspace_bytes(): 4.25 bytes per key for keys
 * only (8.25 with values) when every segment is long, growing with the
 * number of segments up to about 12.3 (16.3) bytes per key.
 * ---------------------------------------------------------------------- */
size_t gsort_segmented_sort_workspace_bytes(int64_t n, int64_t num_segments, int with_values);

int gsort_segmented_sort(const void *d_keys_in, void *d_keys_out,
                         const uint32_t *d_vals_in, uint32_t *d_vals_out, int64_t n,
                         const uint32_t *d_offsets, int64_t num_segments,
                         int kind, int flags, void *d_ws, size_t ws_bytes,
                         cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Device-side status: synchronises `stream`, then returns GSORT_OK or the
 * error a kernel recorded in this workspace during the last call that used
 * it (GSORT_ETIMEOUT), or GSORT_ECUDA if the stream reports an error.
 * ---------------------------------------------------------------------- */
int gsort_check(const void *d_ws, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Extended calls: the same operations with options for tracing, tuning and
 * testing.  A NULL options pointer means the defaults.
 * ---------------------------------------------------------------------- */
typedef struct gsort_options {
    /* Polls of one look-back wait before the kernel records GSORT_ETIMEOUT
     * and returns (0 = default, about a second of back-off). */
    uint32_t spin_limit;
    /* Testing only: the tile with this id never publishes its counts, so
     * waits behind it run out.  -1 = none. */
    int64_t stall_tile;
    /* Optional array of cudaEvent_t handles recorded on `stream` around the
     * launches: radix: [0] start, [1] after init, [2] after histogram,
     * [3 + p] after digit pass p; compaction: [0] start, [1] after init,
     * [2] and [3] after the scan/scatter kernel (which also writes the
     * zero tail).  Extra
     * entries are left alone; missing ones are skipped. */
    void **events;
    int num_events;
    /* Launch configuration of the digit passes of 32-bit keys (0 = default;
     * see gsort_radix_variant_name()); 64-bit keys have one configuration
     * and accept only 0. */
    int variant;
} gsort_options;

int gsort_radix_pairs_ex(const void *d_keys_in, void *d_keys_out,
                         const uint32_t *d_vals_in, uint32_t *d_vals_out, int64_t n,
                         int kind, int begin_bit, int end_bit,
                         void *d_ws, size_t ws_bytes, cudaStream_t stream,
                         const gsort_options *options);

int gsort_radix_sort_ex(const void *d_keys_in, void *d_keys_out,
                        const uint32_t *d_vals_in, uint32_t *d_vals_out, int64_t n,
                        int kind, int flags, int begin_bit, int end_bit,
                        void *d_ws, size_t ws_bytes, cudaStream_t stream,
                        const gsort_options *options);

/* Events for the segmented sort: [0] start, [1] after the classification,
 * [3] after the large segments' histograms, [4 + p] after digit pass p of
 * the large segments, [2] at the end, once the small segments are sorted too
 * (their networks run on streams of the library's own beside the large
 * segments' kernels; `stream` waits for them before [2]). */
int gsort_segmented_sort_ex(const void *d_keys_in, void *d_keys_out,
                            const uint32_t *d_vals_in, uint32_t *d_vals_out, int64_t n,
                            const uint32_t *d_offsets, int64_t num_segments,
                            int kind, int flags, void *d_ws, size_t ws_bytes,
                            cudaStream_t stream, const gsort_options *options);

int gsort_compact_positive_ex(const float *d_in, float *d_out, int64_t n,
                              int64_t *d_num_kept, void *d_ws, size_t ws_bytes,
                              cudaStream_t stream, const gsort_options *options);

/* Number of digit-pass launch configurations, and the name of one
 * ("warps x items per thread, ranking method"); NULL if out of range. */
int gsort_radix_num_variants(void);
const char *gsort_radix_variant_name(int variant);

/* Kernel launches one call makes with the default variant (for launch
 * accounting): radix: 2 for 32-bit keys and n <= 2^18 (one cooperative
 * kernel runs every pass), else 2 + passes (+1 copy-back when sorting in
 * place with an odd pass count; +1 histogram clear for 64-bit keys, see
 * gsort_radix_sort_launch_count); compaction: 2; segmented: 1 (0 when
 * there is nothing to do). */
int gsort_radix_launch_count(int64_t n, int begin_bit, int end_bit, int in_place);
int gsort_radix_sort_launch_count(int64_t n, int kind, int begin_bit, int end_bit, int in_place);

#ifdef __cplusplus
}
#endif

#endif /* GSORT_H */

/*
 * sc_scan.h -- C ABI of the GB300 (sm_103a) device-wide scan and stream
 * compaction library (libsc_gb300.so).
 *
 * What the calls compute.
 *   Inclusive scan  y[i] = x[0] (+) x[1] (+) ... (+) x[i].
 *   Exclusive scan  y[0] = I,  y[i] = x[0] (+) ... (+) x[i-1]  (I: identity of (+)).
 *   Both as defined in "Lecture 7: Parallel pattern -- prefix sum / scan:
 *   double buffering and hierarchical algorithms" (UIUC ECE408 course notes),
 *   section 1 "Scan: inclusive and exclusive", and in "Chapter 9 Parallel
 *   Patterns: Prefix Sum - Scan Algorithms" (PMPP notes), section 9.1, whose
 *   identity table gives 0 for addition and -infinity (here INT32_MIN) for max.
 *   A scan keeps the order of its operands, so (+) needs associativity but not
 *   commutativity (Lecture 7 notes, section 1).
 *   Stream compaction keeps, in input order, the elements that satisfy a
 *   predicate (Lecture 7 notes, section 2 "Applications of Scan"; PMPP notes,
 *   section 9.6 "Applications of Scan", filtering).
 *
 * Operators (dtype, op):
 *   (SC_I32, SC_SUM), (SC_U32, SC_SUM)  sum modulo 2^32 (two's complement
 *                                        wraparound; identical bits for both);
 *   (SC_F32, SC_SUM)                    float32 sum; within a tile in fp32, the
 *                                        inclusive prefix carried between tiles
 *                                        as a float-float pair (about 45 bits),
 *                                        tile totals folded in fp32 onto it;
 *                                        result within 1e-5 * sum_{k<=i} |x[k]|
 *                                        of the exact prefix (not bitwise
 *                                        reproducible: the look-back may fold
 *                                        tile totals in a different grouping
 *                                        from run to run);
 *   (SC_I32, SC_MAX)                    max, identity INT32_MIN;
 *   (SC_AFFINE_U32, SC_COMPOSE)         element i is the map h -> a_i*h + b_i
 *                                        (mod 2^32), stored as the uint32 pair
 *                                        (a_i, b_i) (8 bytes, a first);
 *                                        (a1,b1) (+) (a2,b2) = (a2*a1, a2*b1 + b2)
 *                                        (the earlier map is applied first;
 *                                        identity (1, 0)); y[i] applied to h0
 *                                        gives the recurrence h_i = a_i*h_{i-1} + b_i.
 *   The other operators the Lecture 7 notes (section 1) list for a scan, with
 *   the identities of the PMPP notes' table (section 9.1):
 *   (SC_I32 | SC_U32 | SC_I64 | SC_U64, SC_PROD)   product modulo 2^32 / 2^64,
 *                                        identity 1;
 *   (same types, SC_AND | SC_OR | SC_XOR)  bitwise, identities all ones / 0 / 0
 *                                        (xor is not on the list; it is added);
 *   (SC_I64 | SC_U64, SC_SUM)           sum modulo 2^64;
 *   (SC_I32 | SC_U32 | SC_I64 | SC_U64, SC_MAX | SC_MIN)  in the type's own
 *                                        order, identity the type's smallest /
 *                                        largest value;
 *   (SC_F32 | SC_F64, SC_MAX | SC_MIN)  identity -inf / +inf; a NaN element
 *                                        makes every later output NaN; of two
 *                                        equal values the earlier is kept, so
 *                                        -0.0 and +0.0 come out as they went in;
 *                                        exact (bit for bit, except that a NaN
 *                                        output is a NaN, not necessarily the
 *                                        input NaN's payload);
 *   (SC_F64, SC_SUM)                    float64 sum, within
 *                                        (16 * ceil(n/2048) + 64) * 2^-53 *
 *                                        sum_{k<=i} |x[k]| of the exact prefix
 *                                        (at most 16 roundings per look-back
 *                                        hop, one hop per tile of >= 2048
 *                                        elements, < 64 inside a tile);
 *   (SC_MAXCOUNT_I32, SC_MAX)           element (v, c): (v1,c1) (+) (v2,c2) is
 *                                        the pair with the larger value, the
 *                                        counts added (mod 2^32) when the values
 *                                        are equal; identity (INT32_MIN, 0) --
 *                                        the notes' "(maximum, number of
 *                                        occurrences)" compound operator.
 *
 * Conventions for every call below.
 *   - Pointers named d_* / in / out are DEVICE pointers owned by the caller
 *     (e.g. torch tensors).  Elements are contiguous.  4-byte types need
 *     4-byte alignment, 8-byte types and pairs 8-byte alignment; 16-byte
 *     aligned in/out take the vectorised path.
 *   - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t;
 *     NULL is the legacy default stream).  They never synchronise the host and
 *     never allocate in steady state: the first call on a (device, stream)
 *     pair allocates that pair's workspace (or uses one given with
 *     sc_set_workspace) and grows it only when a larger n arrives.
 *   - Calls on one stream must not overlap in time with calls on the same
 *     stream from another host thread; different streams have independent
 *     workspaces.
 *   - Calls cannot be captured into a CUDA graph: each call's look-back epoch
 *     and tile-counter base are host state that a replay would repeat.  A
 *     call whose stream is capturing returns SC_ERR_UNSUPPORTED before any
 *     launch.
 *   - n == 0 is a successful no-op (compaction writes *d_count = 0).
 *   - Argument errors are detected on the host before any launch and return
 *     SC_ERR_INVALID / SC_ERR_UNSUPPORTED.  A failure inside a kernel (a
 *     look-back wait that exceeds its time bound) is reported by
 *     sc_get_device_error; the kernel never traps and never hangs.
 */
#ifndef SC_SCAN_H
#define SC_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so this header needs no CUDA header. */
typedef struct CUstream_st *sc_stream_t;

typedef enum {
    SC_I32 = 0, SC_U32 = 1, SC_F32 = 2,
    SC_AFFINE_U32 = 3,   /* uint32 pairs (a, b), 8 bytes: the map h -> a*h + b */
    SC_I64 = 4, SC_U64 = 5, SC_F64 = 6,
    SC_MAXCOUNT_I32 = 7  /* pairs (int32 value, uint32 count), 8 bytes */
} sc_dtype;
typedef enum {
    SC_SUM = 0, SC_MAX = 1,
    SC_COMPOSE = 2,      /* SC_AFFINE_U32 only */
    SC_MIN = 3, SC_PROD = 4, SC_AND = 5, SC_OR = 6, SC_XOR = 7
} sc_op;
/* Compaction predicate "x <pred> threshold", evaluated as if in double
 * precision (every int32, uint32 and float32 value is exact in double). */
typedef enum { SC_GT = 0, SC_GE = 1, SC_LT = 2, SC_LE = 3, SC_EQ = 4, SC_NE = 5 } sc_pred;
typedef enum {
    SC_OK = 0,
    SC_ERR_INVALID = 1,          /* bad pointer, size, enum or alignment */
    SC_ERR_UNSUPPORTED = 2,      /* valid enums, but this (dtype, op) is not provided */
    SC_ERR_WORKSPACE = 3,        /* caller-bound workspace too small, or allocation failed */
    SC_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
    SC_ERR_LOOKBACK_TIMEOUT = 5, /* a kernel gave up waiting on a predecessor tile */
    SC_ERR_INTERNAL = 6          /* a kernel's bounds check caught an out-of-range position (nothing written there) */
} sc_status;

/* Library version string. */
const char *sc_version(void);

/* Human-readable name of a status code (static storage). */
const char *sc_status_string(sc_status s);

/* Bytes of device workspace a scan or compaction of n elements needs (for
 * sc_scan_batched: n = rows * cols).  Includes the tile counter, the device
 * error word and one look-back status slot (8 or 16 bytes) per tile. */
size_t sc_workspace_bytes(int64_t n);

/* Bind caller-owned device memory `d_ws` (bytes >= sc_workspace_bytes(n) of
 * the largest call to come, 256-byte aligned) as the workspace of `stream` on
 * the current device.  The library zeroes it with an async memset on `stream`
 * and never frees it.  d_ws == NULL unbinds it (the library then allocates
 * its own on the next call).  Calls whose n needs more than `bytes` return
 * SC_ERR_WORKSPACE. */
sc_status sc_set_workspace(void *d_ws, size_t bytes, sc_stream_t stream);

/* Single-pass inclusive / exclusive scan of n elements (one kernel launch).
 * in == out (in place) is allowed: every tile reads all of its input before it
 * writes any output, and writes only its own range.  Any other overlap of in
 * and out is an error (SC_ERR_INVALID). */
sc_status sc_scan_inclusive(sc_dtype dtype, sc_op op, const void *in, void *out, int64_t n, sc_stream_t stream);
sc_status sc_scan_exclusive(sc_dtype dtype, sc_op op, const void *in, void *out, int64_t n, sc_stream_t stream);

/* Independent scans of the rows of a row-major rows x cols matrix (leading
 * dimension cols, contiguous): row r of out is the scan of row r of in, each
 * starting again from the identity.  One kernel launch.  For the int32/uint32
 * sum, int32 max and float32 sum on 16-byte aligned arrays of at least 8192
 * elements with cols <= 8192 a persistent rows kernel runs with no look-back:
 * when cols divides 8192 every 8192-element tile holds whole rows; otherwise
 * (out != in only) each CTA takes a contiguous range of tiles and carries the
 * open row from tile to tile.  Everything else is a scan segmented at the
 * multiples of cols (the heads computed from the element index, no flag
 * array): on the persistent segmented kernel for operators with 4-byte
 * elements and 16-byte aligned arrays of at least 8192 elements, else on the
 * one-tile-per-CTA kernel; a chunk or tile that holds a row start publishes
 * its complete prefix at once, so look-backs stop there.  Same dtypes, ops and
 * aliasing rules as sc_scan_inclusive. */
sc_status sc_scan_batched(sc_dtype dtype, sc_op op, int exclusive, const void *in, void *out,
                          int64_t rows, int64_t cols, sc_stream_t stream);

/* Segmented scan with head flags: d_heads[i] != 0 (one byte per element,
 * device memory, n bytes) starts a new segment at i; element 0 always starts
 * one.  The running value restarts from the identity at every head, so y[i]
 * is the scan of x[s..i] (inclusive) or x[s..i-1] (exclusive: the identity at
 * s itself), s the last head at or before i.  The Lecture 7 notes (section 2)
 * name the segmented scan as the placement step of each radix-sort digit
 * pass, and (section 1) max/min scans for "predicate prefix" questions such as
 * "is this the first element of its segment that satisfies the condition";
 * the head-flag form is the plain reading of a segment boundary.  Every
 * (dtype, op) pair of the plain scans; in == out is allowed; d_heads must not
 * overlap out.  One launch: operators with 4-byte elements, on 16-byte
 * aligned in, out and d_heads of at least 8192 elements, run on the persistent
 * kernel (flags copied in bulk beside each tile; a chunk of tiles that holds a
 * head publishes its complete prefix at once), everything else on the
 * one-tile-per-CTA kernel (likewise per tile). */
sc_status sc_scan_segmented(sc_dtype dtype, sc_op op, int exclusive, const void *in, const uint8_t *d_heads,
                            void *out, int64_t n, sc_stream_t stream);

/* Histogram of int32 bin indices: d_counts[b] (int64, nbins entries) = the
 * number of i with d_bins[i] == b, 0 <= b < nbins; entries outside [0, nbins)
 * are skipped.  1 <= nbins < 2^31; d_counts must not overlap d_bins.  One
 * memset and one kernel launch (up to 1024 bins each warp counts in shared
 * memory, up to 32768 each CTA; beyond 1024 a run of equal neighbouring bins
 * shares one atomic).  Keeps no host state between calls, so unlike the other
 * calls it may be captured into a CUDA graph. */
sc_status sc_histogram(const int32_t *d_bins, int64_t n, int64_t nbins, int64_t *d_counts, sc_stream_t stream);

/* Bin offsets: d_offsets[b] (int64, nbins + 1 entries) = the number of i with
 * 0 <= d_bins[i] < b, i.e. the exclusive scan of the histogram, and
 * d_offsets[nbins] = the number of entries inside [0, nbins).  With d_bins =
 * the row indices of a COO sparse matrix and nbins = its row count these are
 * the CSR row offsets; with d_bins = a radix digit of each key, the start of
 * each bucket ("Chapter 9 Parallel Patterns: Prefix Sum - Scan Algorithms",
 * PMPP notes, section 4.2).  The histogram above, then the int64 exclusive
 * scan in place. */
sc_status sc_bin_offsets(const int32_t *d_bins, int64_t n, int64_t nbins, int64_t *d_offsets, sc_stream_t stream);

/* Radix sort ("Lecture 7" notes, section 2: one pass per digit, a split whose
 * placement is a scan; PMPP notes, section 4.2: the scan of the digit
 * histogram gives each bucket's start).
 *
 * sc_radix_pass_u32: one stable counting-sort pass: d_out receives the keys of
 * d_in ordered by the digit (key >> shift) & (2^bits - 1), keys with equal
 * digits in their input order.  1 <= bits <= 8, 0 <= shift <= 31,
 * n < 2^32; d_in and d_out must not overlap.  Three launches over
 * 4096-key tiles: each tile's digit counts (workspace: 1 KiB per tile, digit
 * major), their exclusive scan in place (which gives every tile the start of
 * its run of each digit), the placement.
 *
 * sc_radix_sort_u32: d_out = the keys of d_in in ascending order, by four 8-bit
 * passes (least significant digit first) ping-ponging through d_tmp (n keys);
 * d_in may equal d_out; d_tmp must overlap neither. */
sc_status sc_radix_pass_u32(const uint32_t *d_in, uint32_t *d_out, int64_t n, int shift, int bits,
                            sc_stream_t stream);
sc_status sc_radix_sort_u32(const uint32_t *d_in, uint32_t *d_out, uint32_t *d_tmp, int64_t n, sc_stream_t stream);

/* Fused, order-preserving stream compaction (one kernel launch): out[0..count)
 * receives, in input order, every in[i] with (in[i] <pred> threshold); the
 * number kept is written to *d_count (device int64).  out[count..n) is left
 * untouched.  dtype: SC_I32, SC_U32 or SC_F32.  in and out must not overlap. */
sc_status sc_compact_if(sc_dtype dtype, const void *in, void *out, int64_t *d_count, int64_t n,
                        sc_pred pred, double threshold, sc_stream_t stream);

/* The pages' multi-kernel hierarchical design (scan each tile and record its
 * total; scan the totals, recursively; add each tile's offset back), restated
 * for sm_103a.  Same results as the single-pass scan (float32: within the same
 * bound), about twice the memory traffic.  A comparison variant: it needs
 * extra workspace for the per-level totals (sc_hier_workspace_bytes), and it
 * covers the int32/uint32 sum, float32 sum, int32 max and affine composition
 * only (SC_ERR_UNSUPPORTED otherwise; sc_hier_workspace_bytes returns 0 for
 * other dtypes). */
sc_status sc_scan_hierarchical(sc_dtype dtype, sc_op op, int exclusive, const void *in, void *out,
                               int64_t n, sc_stream_t stream);
size_t sc_hier_workspace_bytes(sc_dtype dtype, int64_t n);

/* Scan of HOST buffers: copies h_in to the device in chunks, scans each chunk
 * with the single-pass kernel (the running total of the earlier chunks is
 * carried into the next chunk on the device), and copies the results to h_out,
 * overlapping the copies in both directions with the kernels.  h_in == h_out
 * is allowed.  Pinned (page-locked) host memory is needed for the overlap;
 * pageable memory works but is slower.  Returns after h_out holds the result
 * (it waits for earlier work on `stream` first).  Device staging memory is
 * allocated by the library on first use and kept. */
sc_status sc_scan_host(sc_dtype dtype, sc_op op, int exclusive, const void *h_in, void *h_out, int64_t n,
                       sc_stream_t stream);

/* ---- scan without any allocation ----
 *
 * sc_scan_noalloc computes exactly what sc_scan_inclusive (exclusive == 0) or
 * sc_scan_exclusive (exclusive != 0) compute, for the int32/uint32 sum, float32
 * sum, int32 max and affine composition (other operators: SC_ERR_UNSUPPORTED),
 * with the same aliasing rules, but it never allocates device memory.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot call
 * cudaMalloc: code running where the device allocator is unavailable or must
 * not be touched (inside another framework's memory pool, in an allocator's
 * own bookkeeping, or in latency-critical paths that cannot risk the implicit
 * synchronisation cudaMalloc/cudaFree may cause).  The caller passes the
 * input and output buffers as usual.
 *
 * The look-back workspace it needs lives in a fixed array inside the
 * library's device image: about 1 MiB (256 bytes + 16 bytes per 2048
 * elements of SC_NOALLOC_MAX_N), held on every GPU that loads the library
 * until the process exits.
 *   - n > SC_NOALLOC_MAX_N is rejected with SC_ERR_WORKSPACE before any launch.
 *   - The first call on a device looks up the array's device address on that
 *     device; make that first call before any stream capture begins.
 *   - All calls on a device share the one array: calls whose work can overlap
 *     on the GPU (other streams, other host threads) race and corrupt each
 *     other.  Order them on one stream, or serialise them.
 *   - The cached address belongs to the device's context of that first
 *     call: do not use this entry point across a cudaDeviceReset.
 *   - Each call clears the tile counter it uses with an 8-byte
 *     cudaMemsetAsync on `stream`, then launches one scan kernel.  Its
 *     launches are not counted by sc_launch_count.
 *   - Look-back waits stay bounded (the bound of sc_debug_set_lookback, and
 *     its test hooks, apply here too).  A wait that gives up (only if a CTA is
 *     starved for seconds) leaves that call's output incomplete and sets the
 *     array's error word, which sc_scan_noalloc_error reads and clears; calls
 *     leave the word alone. */
#define SC_NOALLOC_MAX_N (1LL << 27)
sc_status sc_scan_noalloc(sc_dtype dtype, sc_op op, int exclusive, const void *in, void *out, int64_t n,
                          sc_stream_t stream);
/* Wait for `stream`, then read and clear the error word of the fixed array on
 * the current device: SC_OK, or SC_ERR_LOOKBACK_TIMEOUT if an sc_scan_noalloc
 * call since the last query gave up a wait.  Allocates nothing (the word is
 * copied into a host variable). */
sc_status sc_scan_noalloc_error(sc_stream_t stream);

/* Wait for `stream`, then read and clear the device error word of its
 * workspace.  SC_OK when no kernel reported a failure since the last call. */
sc_status sc_get_device_error(sc_stream_t stream);

/* Wait for `stream`, then free the device memory the library keeps for it on
 * the current device: its look-back workspace (unless bound by the caller
 * with sc_set_workspace, which the library never frees) and the staging
 * buffers, streams and events sc_scan_host set up for it.  A later call on
 * the stream sets them up again.  Must not run while another call on the same
 * stream is in progress in another host thread.  SC_OK also when the stream
 * holds nothing. */
sc_status sc_release_stream(sc_stream_t stream);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t sc_launch_count(void);

/* ---- tuning and test hooks (process-wide; affect later launches) ---- */

/* Select the kernel of the uint32/int32 sum.  0 (default): the persistent
 * TMA-pipelined kernel wherever it applies (16-byte aligned arrays of more
 * than 2^22 elements -- 2^20 for the other operators' 8-byte elements; scans
 * segmented by head flags and batched rows on its segmented form or the rows
 * kernel), else the
 * one-tile-per-CTA kernel (for n <= 2^22 its shape of 8192-element tiles of
 * 512 threads, variant 4); v >= 1: one of the precompiled shapes (see
 * sc_scan_variant_info), kept for on-GPU comparison (always on the kernel the
 * shape belongs to); for one-tile segmented scans and batched rows variants
 * 1, 6, 9, 10 and 11 select their shape, any other the default.
 * Returns SC_ERR_INVALID for an unknown variant. */
sc_status sc_set_scan_variant(int variant);
/* Distance between consecutive look-back status words (every single-pass
 * kernel): 0 (default) the widest of 128, 64, 32 and 16 bytes that the
 * workspace holds for the call's tiles or chunks; 16 / 32 / 64 / 128 that many
 * bytes where the workspace holds it (else packed); -1 packed (8 bytes for
 * 4-byte carries, 16 for 8-byte ones).  SC_ERR_INVALID otherwise. */
sc_status sc_set_status_stride(int bytes);
/* Select the fused-compaction kernel: 0 (default) the persistent TMA kernel
 * with 8 compute warps, each kept element stored on its own (4-byte stores);
 * 1 the same with 16 compute warps; 2 the one-tile-per-CTA kernel (inputs that
 * are not 16-byte aligned, or smaller than one 32 KiB tile, always use the
 * latter); 3 the persistent kernel with 8 compute warps that packs each warp's
 * kept elements in shared memory and writes them as aligned 16-byte stores;
 * 4 and 5 as 0 with 4 fresh-tile and 2 re-load stages, or 2 and 4, instead
 * of 3 and 3; 6 and 7 as 0 with a pass-2 lag of 6 or 4 tiles instead of 8.
 * SC_ERR_INVALID otherwise. */
sc_status sc_set_compact_variant(int variant);
/* Select how the radix pass ranks a warp step's keys by digit: 0 (default)
 * __match_any_sync on the digit's top 3 bits and one ballot per lower bit;
 * v = 1..5: v - 1 bits by __match_any_sync, the other 8 - (v - 1) by ballots.
 * Every variant gives the same (stable) result.  SC_ERR_INVALID otherwise. */
sc_status sc_set_radix_variant(int variant);
/* Threads per CTA, items per thread and loader kind (0 direct loads,
 * 1 coalesced loads + shared-memory transpose, 2 persistent TMA pipeline;
 * for 2, threads are the CTA's compute threads) of a uint32-sum variant;
 * SC_ERR_INVALID if it does not exist. */
sc_status sc_scan_variant_info(int variant, int *threads, int *items, int *loader);

/* Kernel family of the calling host thread's last scan or compaction launch
 * (test hook: lets a test confirm which kernel a case reached). */
typedef enum {
    SC_PATH_NONE = 0,
    SC_PATH_SCAN_ONE_TILE = 1,        /* one tile per CTA (plain, segmented or batched) */
    SC_PATH_SCAN_PERSISTENT = 2,      /* persistent TMA-pipelined scan */
    SC_PATH_SEGSCAN_PERSISTENT = 3,   /* persistent scan segmented by head flags */
    SC_PATH_COMPACT_PERSISTENT = 4,   /* persistent fused compaction */
    SC_PATH_COMPACT_ONE_TILE = 5,     /* one-tile-per-CTA fused compaction */
    SC_PATH_ROWS_PERSISTENT = 6       /* persistent batched rows, every tile whole rows (no look-back) */
} sc_path;
int sc_debug_last_path(void);

/* Look-back test hooks.  stall_tile >= 0: that tile never publishes its
 * status, so its successors must time out (error SC_ERR_LOOKBACK_TIMEOUT).
 * delay_tile >= 0: that tile sleeps delay_ns before publishing (exercises
 * long look-back chains).  timeout_ns: bound on any single look-back wait
 * (0 restores the default of 2 s).  -1 turns a hook off. */
sc_status sc_debug_set_lookback(int64_t stall_tile, int64_t delay_tile, uint32_t delay_ns, uint64_t timeout_ns);

/* Phase timers of the instrumented uint32-sum variants (sc_scan_variant_info
 * lists them; they are for measurement, not production).  Waits for `stream`,
 * copies the 8 counters accumulated by that stream's launches into out8 and
 * clears them: [0] tiles, [1] ns until tile ids were known, [2] ns loading and
 * scanning tiles, [3] ns in the look-back, [4] look-back windows read,
 * [5] polls that found a predecessor not yet published, [6] ns from the
 * prefix to the end of the stores, [7] ns of whole tiles (all summed over
 * tiles). */
sc_status sc_debug_lookback_stats(sc_stream_t stream, uint64_t *out8);

#ifdef __cplusplus
}
#endif

#endif /* SC_SCAN_H */

/*
 * ordmerge.h -- C ABI of the GB300 (sm_103a) stable co-rank merge library
 * (libordmerge.so).
 *
 * Operation.  C = merge(A, B): the stable merge of two arrays that are each
 * sorted nondecreasing.  When an element of A equals an element of B, the A
 * element comes first.  The work is split by the co-rank function: for an
 * output rank k, co_rank(k) is the i (with j = k - i) such that A[0..i) and
 * B[0..j) are exactly the first k outputs, i.e. the unique i with
 *     (i == 0 || j == n || A[i-1] <= B[j])  and  (j == 0 || i == m || B[j-1] < A[i]).
 * Sources: "Co-rank Function 實作與 Basic Parallel Merge Kernel"
 * (§Co-rank Function 定義與不變式, §Binary-Search Implementation, §Important on
 * the asymmetric test); "Tiled 與 Circular Buffer Merge Kernel (Memory
 * Coalescing)" (§Block-Level Co-Rank, §Circular Buffer Merge Kernel);
 * "merge_path.cu" (coRank, mergeCpu); "排序 (Sorting) 練習題" (merge-sort
 * stages, stable sort).
 *
 * Conventions for every call below.
 *  - Array arguments are DEVICE pointers (memory the current CUDA device can
 *    address: cudaMalloc, cudaMallocAsync, managed, or a torch CUDA tensor).
 *    The caller owns them.  Element pointers must be 4-byte aligned; for
 *    key/value calls, each value array must have the same address modulo 16
 *    as its key array.  Output arrays must not overlap input arrays.
 *  - Lengths are element counts (int64).  m = 0 or n = 0 is valid (the merge
 *    is then a copy); m + n = 0 is a no-op.
 *  - Inputs must be sorted nondecreasing (signed order for int32, unsigned for
 *    uint32).  This is a precondition and is not checked; on unsorted input
 *    the output is unspecified, but every kernel still terminates.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Merge and sort calls are asynchronous with respect to the
 *    host: they validate, enqueue and return.  Errors raised while the
 *    kernels run surface at the caller's next synchronisation, and in
 *    om_device_error().
 *  - Merges allocate nothing.  The sorts' scratch (their second key and
 *    value buffers) is taken from the library's own stream-ordered memory
 *    pool (created by the first sort on each device) on `stream`
 *    (cudaMallocFromPoolAsync) and freed on the same stream (cudaFreeAsync),
 *    so it is stream-ordered; failure returns OM_ENOMEM.  The pool keeps
 *    freed scratch mapped for later calls, so a device holds up to the
 *    largest scratch any call needed until om_release_scratch().
 *  - No call exits the process or prints.  A failing call returns a status.
 */
#ifndef ORDMERGE_H
#define ORDMERGE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    OM_OK = 0,
    OM_EINVAL = 1,  /* NULL pointer with a nonzero length, negative length,
                       misaligned pointer, overlapping output */
    OM_ERANGE = 2,  /* k outside [0, m + n], or m + n overflows */
    OM_ENOMEM = 3,  /* stream-ordered scratch allocation failed */
    OM_ECUDA = 4,   /* a CUDA runtime call or kernel launch failed */
    OM_EDEVICE = 5  /* a kernel reported an error (om_device_error) */
} om_status;

/*
 * co_rank(k) of A[0..m) and B[0..n): returns i in [max(0, k-n), min(k, m)];
 * the caller derives j = k - i ("Co-rank Function 實作與 Basic Parallel Merge
 * Kernel", §Co-rank Function 定義與不變式: the function returns i only).
 * Runs one search on the device and waits for it: synchronous.  It is
 * ordered after prior work on the legacy default stream only.  Returns the
 * negated om_status (< 0) on error.
 */
int64_t om_corank_i32(int64_t k, const int32_t *A, int64_t m,
                      const int32_t *B, int64_t n);

/*
 * Batched co-rank on the device: i_out[t] = co_rank(ks[t]) for t < count.
 * ks and i_out are device arrays of int64 (each ks[t] in [0, m + n]; an
 * out-of-range k is clamped into that interval).  Asynchronous on `stream`.
 */
om_status om_corank_i32_batch(const int64_t *ks, int64_t count,
                              const int32_t *A, int64_t m,
                              const int32_t *B, int64_t n,
                              int64_t *i_out, void *stream);

/*
 * Grid-level merge-path partition: split[t] = co_rank(min(t * tile, m + n))
 * for t < count, one co-rank search per output tile boundary, run by one
 * warp each (32 probes per round) in a single launch on `stream`
 * ("Tiled 與 Circular Buffer Merge Kernel (Memory Coalescing)",
 * §Block-Level Co-Rank: one co-rank per block's output tile; "Co-rank
 * Function 實作與 Basic Parallel Merge Kernel", §Co-rank Function 定義與不變式).
 * The caller derives j_t = min(t * tile, m + n) - split[t].  split is a
 * device array of count int64 owned by the caller, 8-byte aligned, not
 * overlapping A or B.  tile >= 1 and count >= 0, else OM_EINVAL.  This is
 * the kernel om_merge_i32_noalloc runs before its tile merge; om_merge_i32
 * finds the same splitters inside its tile-merge kernel.  Allocates nothing.
 */
om_status om_partition_i32(const int32_t *A, int64_t m, const int32_t *B,
                           int64_t n, int64_t tile, int64_t count,
                           int64_t *split, void *stream);

/*
 * C[0 .. m+n) = stable merge of int32 A[0..m) and B[0..n); ties take A
 * first.  One launch on `stream`.  A merge that fits in one wave of small
 * CTAs (about 4.2 M outputs on a 152-SM GB300; the one-pass kernel: one
 * output tile per CTA, both windows loaded into shared memory at once and
 * merged by every thread) takes that kernel; a larger one takes the
 * circular-buffer tile-merge kernel, whose CTAs stream their output ranges
 * through shared-memory rings.  In either, two warps of each CTA first find
 * the co-ranks of its output range's two ends (one each).  Allocates
 * nothing.  The environment variable OM_ONE_PASS_MAX (an output count; 0:
 * never) moves the size at which the one-pass kernel stops; setting
 * OM_SUBTILES_PER_RANGE or OM_WAVES selects the tile-merge kernel.  The same
 * holds for om_merge_pairs_u32 and om_merge_keys.
 */
om_status om_merge_i32(const int32_t *A, int64_t m, const int32_t *B,
                       int64_t n, int32_t *C, void *stream);

/*
 * Stable merge of (uint32 key, uint32 value) pairs, comparing keys only
 * (unsigned order); each value travels with its key; ties take A first.
 * Outputs keysC / valsC hold m + n elements.
 */
om_status om_merge_pairs_u32(const uint32_t *keysA, const uint32_t *valsA,
                             int64_t m, const uint32_t *keysB,
                             const uint32_t *valsB, int64_t n,
                             uint32_t *keysC, uint32_t *valsC, void *stream);

/*
 * Stable sort of keys[0..n) (unsigned order), in place, carrying vals along
 * (vals may be NULL for a keys-only sort).  Built only from merges: tiles of
 * 4096 are sorted in shared memory (runs of 16 in registers, then many small
 * merges per thread block through runs of 1024 to 4096), then runs are
 * merged pairwise in co-rank-split passes ("排序 (Sorting) 練習題",
 * merge-sort stages).
 * Equal keys keep their input order.  Needs 4*n (8*n with vals) bytes of
 * stream-ordered scratch.
 */
om_status om_merge_sort_u32(uint32_t *keys, uint32_t *vals, int64_t n,
                            void *stream);

/* Human-readable name of a status (static string). */
const char *om_status_string(int status);

/*
 * Synchronises `stream`, then reads and clears the library's device error
 * word on the current device.  Returns OM_OK, OM_EDEVICE when a kernel
 * recorded an error (for example a shared-memory barrier wait that hit its
 * time limit), or OM_ECUDA.  *detail (if not NULL) receives the raw word.
 */
om_status om_device_error(void *stream, uint32_t *detail);

/* ---- tracing and counters (used by the benchmark) ---------------------- */

/*
 * With tracing on, every kernel launch is bracketed by two CUDA events on its
 * stream.  om_trace_read synchronises those events and returns, for kernel
 * kind `kind` (0 = partition, 1 = tile merge, 2 = block sort, 3 = co-rank
 * batch, 4 = the comparison merges below, 5 = one-pass merge), the number of
 * launches and their summed duration in milliseconds since the last
 * om_trace_reset.
 */
om_status om_trace_enable(int on);
om_status om_trace_reset(void);
om_status om_trace_read(int kind, int64_t *launches, double *total_ms);

/*
 * Returns the scratch the library's pool holds on the current device to the
 * system (waits for the device first).  Later calls map it again as needed.
 */
om_status om_release_scratch(void);

/* Number of kernels this library has launched since load. */
uint64_t om_launch_count(void);

/*
 * Launch planning, host only (no device call): the number of sub-tiles per
 * CTA output range the library uses for one tile-merge launch over `segs`
 * independent merges of at most `seg_len` outputs each (a merge: segs = 1;
 * a late pass of the sort: one segment per pair of runs), with sub-tiles of
 * `subtile` outputs, `bytes_per_output` bytes read plus written per output
 * and `resident_ctas` CTAs running at a time.  Ranges never cross a
 * segment.  The choice minimises  waves x (fixed cost per range + longest
 * range)  over one to eight waves, so that no launch ends on a partial wave
 * of a few CTAs.  The environment variables OM_WAVES (fixed wave count) and
 * OM_SUBTILES_PER_RANGE (fixed result) override it, here and in every call.
 * Returns a value >= 1, or 0 when an argument is not positive.
 */
int64_t om_subtiles_per_range(int64_t segs, int64_t seg_len, int64_t subtile, int64_t bytes_per_output,
                              int64_t resident_ctas);

/* ---- merge without allocating ------------------------------------------ */

/*
 * The pages have no counterpart to this call: it is a library convenience.
 *
 * Same result as om_merge_i32, in two launches that allocate nothing: the
 * partition kernel writes one co-rank splitter per output range to a fixed
 * 64 KiB array that the library keeps in device memory (a file-scope
 * __device__ object, held on every GPU that loads the library until the
 * process exits), and the tile-merge kernel reads them.  (om_merge_i32 now
 * lets each tile-merge CTA find its own splitters, so it allocates nothing
 * either; this call keeps the two-kernel form.)  For callers that cannot
 * allocate device memory on the call path: processes whose device memory is
 * reserved in full by another allocator, and code with latency bounds that
 * must not enter an allocator.
 *
 *  - m + n may be at most 2^30 = 1,073,741,824, a fixed bound of this call
 *    (the array holds 8191 output-range splitters, and ranges are lengthened
 *    as needed to fit); larger merges return OM_ERANGE and launch nothing.
 *  - The first call on each device does a one-time set-up there: it looks up
 *    the device addresses of the array and of the library's error word, sets
 *    the merge kernels' shared-memory limits and queries their occupancy.
 *    None of that allocates device memory (no memory pool is created; only
 *    the sorts make one); make that first call before any stream capture.
 *  - All calls on a device share the array.  Each call's kernels write every
 *    slot they read before reading it, so nothing needs clearing, but calls
 *    whose kernels overlap on the GPU (e.g. on different streams) race on
 *    the array and can produce wrong output: order them on one stream or
 *    with events.
 *  - With tracing off (the default) no call of this function allocates
 *    anything, on the device or the host; argument rules and errors are those
 *    of om_merge_i32.
 */
om_status om_merge_i32_noalloc(const int32_t *A, int64_t m, const int32_t *B,
                               int64_t n, int32_t *C, void *stream);

/* ---- the pages' unstaged merges, for comparison ------------------------- */

/*
 * The two merges that "merge_path.cu" measures, kept to measure what the
 * shared-memory ring design buys on this GPU.  Same result as om_merge_i32
 * (int32, ties take A first); same argument rules and errors.  Not fast paths.
 *
 * om_merge_i32_one_thread: the two-pointer merge run by one device thread
 * (one block of one thread).
 */
om_status om_merge_i32_one_thread(const int32_t *A, int64_t m,
                                  const int32_t *B, int64_t n, int32_t *C,
                                  void *stream);

/*
 * om_merge_i32_slices: one thread per slice of per_thread outputs (blocks of
 * 256 threads); each thread finds the co-ranks of both ends of its slice in
 * global memory, then merges the input intervals between them straight from
 * global memory, with no shared memory ("Co-rank Function 實作與 Basic Parallel Merge Kernel",
 * §Basic Parallel Merge Kernel; "merge_path.cu").  per_thread >= 1, else
 * OM_EINVAL.
 */
om_status om_merge_i32_slices(const int32_t *A, int64_t m, const int32_t *B,
                              int64_t n, int32_t *C, int64_t per_thread,
                              void *stream);

/* ---- other key types and descending order ------------------------------ */

/* Key types of om_merge_keys (element size 4 or 8 bytes). */
typedef enum {
    OM_KEY_I32 = 0, /* int32, signed order */
    OM_KEY_U32 = 1, /* uint32, unsigned order */
    OM_KEY_F32 = 2, /* IEEE binary32, numeric order */
    OM_KEY_I64 = 3, /* int64, signed order */
    OM_KEY_U64 = 4, /* uint64, unsigned order */
    OM_KEY_F64 = 5  /* IEEE binary64, numeric order */
} om_key_type;

typedef enum {
    OM_ASCENDING = 0,  /* inputs and output nondecreasing */
    OM_DESCENDING = 1  /* inputs and output nonincreasing */
} om_order;

/*
 * C[0 .. m+n) = stable merge of the keys A[0..m) and B[0..n) of type
 * `key_type`, both sorted in `order`; ties take A first in either order.
 * The same tile-merge kernel as om_merge_i32, for another element size and
 * comparison.  ("merge_path.cu" runs the method on float
 * keys; the co-rank test of "Co-rank Function 實作與 Basic Parallel Merge
 * Kernel", §Important, with <= and < read in the merge order.)
 *  - Floating-point keys compare by value: -0.0 and +0.0 are equal (so the
 *    A one comes first) and keep their bits.  NaN has no place in a sorted
 *    array; input holding NaN counts as unsorted (output unspecified, every
 *    kernel still terminates).
 *  - A, B and C must be aligned to the key size (4 or 8 bytes) and C must
 *    not overlap A or B.
 *  - An unknown key_type or order is OM_EINVAL.  Other rules and errors are
 *    those of om_merge_i32.
 */
om_status om_merge_keys(int key_type, int order, const void *A, int64_t m,
                        const void *B, int64_t n, void *C, void *stream);

/*
 * Stable sort of keys[0..n) of type `key_type` into `order`, in place,
 * carrying the uint32 vals along (vals may be NULL).  The pass schedule of
 * om_merge_sort_u32 with that type's compare: 4096-key tiles sorted in
 * shared memory, then co-rank-split merge passes ("排序 (Sorting) 練習題",
 * merge-sort stages).  Equal keys (including -0.0 and +0.0) keep their
 * input order in either order.
 *  - keys aligned to the key size.  Values ride only with 4-byte keys
 *    (I32, U32, F32): vals with an 8-byte key type is OM_EINVAL.  vals, if
 *    given, has the same address modulo 16 as keys and does not overlap it.
 *  - Floating-point keys must not hold NaN (unsorted output otherwise; every
 *    kernel still terminates).
 *  - Needs n * key size (plus 4 * n with vals) bytes of stream-ordered
 *    scratch.  Other rules and errors are those of om_merge_sort_u32.
 */
om_status om_merge_sort_keys(int key_type, int order, void *keys,
                             uint32_t *vals, int64_t n, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ORDMERGE_H */

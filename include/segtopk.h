/*
 * segtopk — segmented (batched) top-k by multi-pass radix digit selection,
 * written for NVIDIA GB300 (sm_103a).
 *
 * C ABI. All pointers are plain pointers; no C++ or framework types cross
 * this boundary. Every call is asynchronous on the given CUDA stream unless
 * its comment says otherwise.
 *
 * What is computed (per segment, independently):
 *   "Implement Segmented TopK using Thread-Block-Clusters" (CUB pull request),
 *   section 1 "High-level overview": for each of num_segments variable-length
 *   segments select the k largest (or smallest) keys, optionally carrying a
 *   value payload. The selection contract (which items, in which order) is
 *   the one of the CUB documentation page "Top-K: Determinism, Tie-Breaking,
 *   and Output Ordering" (sections "Requirements reference" and "Which items
 *   are selected?"), with +0.0 and -0.0 ranked as equal keys whose own bit
 *   patterns are written to the output ("Fix BlockTopK +/-0.0 handling",
 *   sections Cause and Fix).
 */
#ifndef SEGTOPK_H_
#define SEGTOPK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported entry points (the library is built with hidden visibility, so
 * that nothing else it contains can collide with another library's). */
#if defined(__GNUC__)
#define SEGTOPK_API __attribute__((visibility("default")))
#else
#define SEGTOPK_API
#endif

/* Key element types. Keys are read as raw bit patterns of this width. */
typedef enum {
  SEGTOPK_F16 = 0,  /* IEEE binary16 */
  SEGTOPK_BF16 = 1, /* bfloat16 */
  SEGTOPK_F32 = 2,  /* IEEE binary32 */
  SEGTOPK_F64 = 3,  /* IEEE binary64 */
  SEGTOPK_U32 = 4,  /* uint32_t */
  SEGTOPK_I32 = 5   /* int32_t */
} segtopk_dtype;

/* Which end of the order is selected (CUB's Max* / Min* entry points). */
typedef enum { SEGTOPK_MAX = 0, SEGTOPK_MIN = 1 } segtopk_direction;

/* Result-set reproducibility ("Top-K: Determinism, ...", "Determinism" table). */
typedef enum {
  SEGTOPK_NOT_GUARANTEED = 0,
  SEGTOPK_RUN_TO_RUN = 1,
  SEGTOPK_GPU_TO_GPU = 2
} segtopk_determinism;

/* Boundary tie policy (same page, "Tie-break" table). A concrete tie-break
 * requires SEGTOPK_GPU_TO_GPU. UNSPECIFIED is resolved as
 * PREFER_SMALLER_INDEX under RUN_TO_RUN and GPU_TO_GPU; under
 * NOT_GUARANTEED, boundary ties beyond those needed are taken in whatever
 * order the kernel meets them (any subset of the ties is a valid result). */
typedef enum {
  SEGTOPK_TIE_UNSPECIFIED = 0,
  SEGTOPK_PREFER_SMALLER_INDEX = 1,
  SEGTOPK_PREFER_LARGER_INDEX = 2
} segtopk_tie_break;

/* Output order of the selected items (same page, "Output ordering" table).
 * UNSORTED: any order; with a deterministic mode the set is fixed but the
 *         positions may differ from run to run (set membership, not
 *         positions, is what determinism pins).
 * SORTED: by key, better first; equal keys in unspecified order (this
 *         library sorts 64-bit keys on the key alone; single-warp paths
 *         with larger indices preferred write equal keys by descending
 *         index; otherwise equal keys come out in source-index order).
 * STABLE_SORTED: by key, better first; equal keys by source index ascending,
 *         whatever the tie-break. */
typedef enum {
  SEGTOPK_UNSORTED = 0,
  SEGTOPK_SORTED = 1,
  SEGTOPK_STABLE_SORTED = 2
} segtopk_ordering;

/* Status codes returned by every entry point. */
typedef enum {
  SEGTOPK_SUCCESS = 0,
  SEGTOPK_ERROR_INVALID_VALUE = 1,       /* bad enum, null pointer, negative size, k < 0 */
  SEGTOPK_ERROR_INVALID_COMBINATION = 2, /* determinism / tie_break pair not allowed */
  SEGTOPK_ERROR_NOT_SUPPORTED = 3,       /* size or k outside this library's limits */
  SEGTOPK_ERROR_MISALIGNED = 4,          /* keys pointer not aligned to its element size */
  SEGTOPK_ERROR_CUDA = 5,                /* a CUDA runtime call failed: see segtopk_last_cuda_error */
  SEGTOPK_ERROR_DEVICE = 6               /* current device is not an sm_103 GPU */
} segtopk_status;

/* Largest k this library serves (the selected items of one segment are held
 * and sorted on chip). Calls with a larger k return SEGTOPK_ERROR_NOT_SUPPORTED. */
#define SEGTOPK_MAX_K 2048

/* Largest segment length (keys) accepted: segment-local indices are 32-bit. */
#define SEGTOPK_MAX_SEGMENT_LEN 2147483647LL

/*
 * Segmented top-k.
 *
 * Semantics: "Implement Segmented TopK using Thread-Block-Clusters", sections
 * 1.2 "Radix (digit) top-k" (method), 1.5 "Final filter and output placement"
 * and 1.6 "Determinism / tie-breaking"; contract of "Top-K: Determinism,
 * Tie-Breaking, and Output Ordering"; +/-0.0 handling of "Fix BlockTopK
 * +/-0.0 handling".
 *
 * Arguments (all device pointers unless stated):
 *   key_dtype        element type of keys and out_keys.
 *   keys             key array; segment s covers elements
 *                    [segment_offsets[s], segment_offsets[s+1]). Must be
 *                    aligned to its element size (any element of a larger
 *                    array may start it). Read only.
 *   values           optional int32 payload parallel to keys (NULL: keys only).
 *   segment_offsets  int64 array of num_segments + 1 element offsets, each
 *                    non-negative and within the key array. A segment whose
 *                    end is not greater than its begin is empty.
 *   num_segments     number of segments (>= 0).
 *   k                items to select per segment (>= 0).
 *   direction, determinism, tie_break, ordering: see the enums. Valid
 *                    (determinism, tie_break) pairs: (any, UNSPECIFIED) and
 *                    (GPU_TO_GPU, PREFER_SMALLER_INDEX | PREFER_LARGER_INDEX).
 *   out_keys         num_segments * k elements; segment s writes slots
 *                    [s*k, s*k + min(k, n_s)) with the original key bits and
 *                    leaves [s*k + n_s, s*k + k) untouched when n_s < k.
 *   out_values       num_segments * k int32; required iff values != NULL;
 *                    out_values[j] = values[segment_offsets[s] + i] for the
 *                    element i written to out_keys[j].
 *   max_segment_len  host-side upper bound on every segment's length. A
 *                    negative value means unknown: the library then copies
 *                    segment_offsets to the host and waits for the stream
 *                    (a synchronising call). A bound that is too small is a
 *                    caller error: longer segments are left unwritten.
 *   stream           cudaStream_t (NULL = the legacy default stream).
 *
 * Ownership: the caller owns every buffer. The library allocates no device
 * memory; it caches device attributes and per-kernel shared-memory limits.
 * Inputs must not overlap outputs.
 *
 * Errors: argument errors are detected on the host before any launch and
 * nothing is launched. num_segments == 0 or k == 0 is a successful no-op.
 * A failed launch returns SEGTOPK_ERROR_CUDA (segtopk_last_cuda_error()
 * gives the cudaError_t). The call does not synchronise (except as noted
 * for max_segment_len < 0).
 */
SEGTOPK_API int segtopk_batched_topk(segtopk_dtype key_dtype, const void* keys, const int32_t* values,
                         const int64_t* segment_offsets, int64_t num_segments, int32_t k,
                         segtopk_direction direction, segtopk_determinism determinism,
                         segtopk_tie_break tie_break, segtopk_ordering ordering, void* out_keys,
                         int32_t* out_values, int64_t max_segment_len, void* stream);

/* Optional launch controls for segtopk_batched_topk_ex (zero = automatic). */
typedef struct {
  /* CTAs per segment: 0 chooses it from the occupancy the device reports
   * (fewest waves, ties toward the widest cluster); 1..16 forces the width
   * (widths above 8 need non-portable cluster support). */
  int32_t cluster_width;
  /* Warp-select paths (used when k <= 32): segments of at most
   * small_segment_max_len keys take one warp each, longer ones of at most
   * team_segment_max_len keys a team of eight warps each; longer segments
   * (and every segment when k > 32) take one CTA or cluster each. 0 chooses
   * the defaults below (none when cluster_width is forced); a negative value
   * turns that path off. */
  int32_t small_segment_max_len;
  int32_t team_segment_max_len;
  int32_t reserved[5]; /* must be zero */
} segtopk_options;

/* Default limits of the warp-select paths. With at least as many segments as
 * SMs: one warp per segment up to SEGTOPK_SMALL_SEGMENT_DEFAULT keys and no
 * team range (SEGTOPK_TEAM_SEGMENT_DEFAULT does not exceed it: longer
 * segments are faster on the CTA path then). With fewer segments: no
 * single-warp range and teams of eight warps up to SEGTOPK_TEAM_SEGMENT_FEW
 * keys. */
#define SEGTOPK_SMALL_SEGMENT_DEFAULT 4096
#define SEGTOPK_TEAM_SEGMENT_DEFAULT 4096
#define SEGTOPK_TEAM_SEGMENT_FEW 8192

/* segtopk_batched_topk with launch controls; options may be NULL. Returns
 * SEGTOPK_ERROR_INVALID_VALUE for a width outside 0..16 or nonzero reserved
 * fields, and SEGTOPK_ERROR_NOT_SUPPORTED when the device cannot launch the
 * requested width. Without options (and in segtopk_batched_topk), the
 * warp-select paths take the segments their default limits give when
 * k <= 32; the others take one CTA or cluster each. */
SEGTOPK_API int segtopk_batched_topk_ex(segtopk_dtype key_dtype, const void* keys, const int32_t* values,
                            const int64_t* segment_offsets, int64_t num_segments, int32_t k,
                            segtopk_direction direction, segtopk_determinism determinism,
                            segtopk_tie_break tie_break, segtopk_ordering ordering, void* out_keys,
                            int32_t* out_values, int64_t max_segment_len,
                            const segtopk_options* options, void* stream);

/*
 * segtopk_batched_topk_ex with a payload of 4- or 8-byte values: values and
 * out_values point to value_bytes-wide elements (int32_t or int64_t; any
 * 8-byte payload, such as a global index or a pointer, is copied as is).
 * value_bytes must be 4 or 8 when values is not NULL (else
 * SEGTOPK_ERROR_INVALID_VALUE). Everything else is as in
 * segtopk_batched_topk_ex; keys only when values and out_values are NULL.
 * (The pages' CUB pull request lists wider value types and larger segments
 * among its future work: "Implement Segmented TopK using
 * Thread-Block-Clusters", section 10 "Known limitations and future work".)
 */
SEGTOPK_API int segtopk_batched_topk_values(segtopk_dtype key_dtype, const void* keys, const void* values,
                                            int32_t value_bytes, const int64_t* segment_offsets,
                                            int64_t num_segments, int32_t k, segtopk_direction direction,
                                            segtopk_determinism determinism, segtopk_tie_break tie_break,
                                            segtopk_ordering ordering, void* out_keys, void* out_values,
                                            int64_t max_segment_len, const segtopk_options* options,
                                            void* stream);

/*
 * Top-k over one array (no segments): the k best of keys[0, num_keys),
 * with the same contract per mode as one segment of segtopk_batched_topk
 * (source index = array index). The CUB pull request's overview names this
 * operation (cub::DeviceTopK) beside the segmented one ("Implement Segmented
 * TopK using Thread-Block-Clusters", section 1.1).
 *
 * Method: two passes of the segmented selection. The array is split into P
 * balanced contiguous pieces (P = min(304, num_keys / max(65536, 16 k)), at
 * least 1); pass 1 writes each piece's k best, in stable sorted order, to the
 * workspace; pass 2 selects the k best of the P * k candidates. Pieces keep
 * source order and each piece's equal keys keep index order, so a
 * candidate's position orders ties as its array index does: tie-breaks and
 * stable order are exact.
 *
 * Arguments: keys, values, out_keys, out_values, workspace are device
 * pointers. values / out_values: optional payload of value_bytes (4 or 8)
 * per element, both NULL for keys only. out_keys / out_values hold k slots;
 * with num_keys < k only the first num_keys are written. workspace: at
 * least segtopk_topk_workspace_bytes(...) bytes, 256-byte aligned, owned by
 * the caller (the library allocates nothing). num_keys may exceed 2^31 as
 * long as every piece holds fewer than 2^31 keys.
 *
 * Errors as segtopk_batched_topk; a workspace that is too small returns
 * SEGTOPK_ERROR_INVALID_VALUE. Asynchronous on `stream` (up to three kernel
 * launches: the piece offsets, pass 1, pass 2).
 */
SEGTOPK_API size_t segtopk_topk_workspace_bytes(segtopk_dtype key_dtype, int32_t value_bytes, int64_t num_keys,
                                                int32_t k);
SEGTOPK_API int segtopk_topk(segtopk_dtype key_dtype, const void* keys, const void* values, int32_t value_bytes,
                             int64_t num_keys, int32_t k, segtopk_direction direction,
                             segtopk_determinism determinism, segtopk_tie_break tie_break,
                             segtopk_ordering ordering, void* out_keys, void* out_values, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * Same operation with HOST buffers: keys, values, segment_offsets, out_keys
 * and out_values are host pointers (pinned memory gives full copy
 * bandwidth). The caller also passes a device workspace of at least
 * segtopk_host_workspace_bytes(...) bytes, 256-byte aligned (the library
 * allocates nothing). The call copies the keys, the offsets and the output
 * slots to the device, runs the selection on `stream` (for pairs the kernel
 * writes each selected element's source index), copies the results back,
 * waits for the stream, and then gathers the selected values from the
 * caller's host `values` array, so that only the keys cross to the device.
 * The host outputs are ready on return.
 *
 * The host offsets are read on the host: every offset must be non-negative
 * (SEGTOPK_ERROR_INVALID_VALUE otherwise, before anything is copied or
 * launched), and max_segment_len is ignored (the true longest segment is
 * known). Slots past a short segment's length keep their host contents.
 */
SEGTOPK_API int segtopk_batched_topk_host(segtopk_dtype key_dtype, const void* keys, const int32_t* values,
                              const int64_t* segment_offsets, int64_t num_segments, int32_t k,
                              segtopk_direction direction, segtopk_determinism determinism,
                              segtopk_tie_break tie_break, segtopk_ordering ordering,
                              void* out_keys, int32_t* out_values, int64_t max_segment_len,
                              void* device_workspace, size_t workspace_bytes, void* stream);

/*
 * Size of the fixed device staging area of segtopk_batched_topk_host_noalloc:
 * 32 MiB. A request fits when segtopk_host_workspace_bytes(...) for its
 * sizes is at most this (for example about 8 million fp32 keys, with or
 * without int32 values: values stay on the host).
 */
#define SEGTOPK_NOALLOC_STAGING_BYTES (32u * 1024u * 1024u)

/*
 * segtopk_batched_topk_host for callers that cannot allocate device memory:
 * a plugin or library routine running inside a host program that owns the
 * GPU's memory (a framework whose caching allocator has reserved it, so that
 * a cudaMalloc of the caller's own would fail or fragment that pool), or
 * code held to a fixed device-memory budget with no per-call allocations.
 * The source pages have no counterpart of this entry point.
 *
 * Arguments, semantics and results are those of segtopk_batched_topk_host,
 * without the workspace: the device staging comes from a fixed array of
 * SEGTOPK_NOALLOC_STAGING_BYTES inside the library. Every GPU on which the
 * library's device code is loaded holds that array until the process exits.
 * The call runs on the current device, which must be the device of `stream`.
 *
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address once; make that first call before any stream
 * capture begins on the device. The address is kept for the life of the
 * process: a device reset (cudaDeviceReset) between calls is not supported.
 *
 * Limits and errors: a request needing more than SEGTOPK_NOALLOC_STAGING_BYTES
 * of staging returns SEGTOPK_ERROR_NOT_SUPPORTED before anything is copied.
 * Otherwise the status codes are those of segtopk_batched_topk_host. The call
 * makes no device allocation and frees nothing.
 *
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's data; each call writes every byte it reads from it, so nothing needs
 * clearing. Calls whose GPU work overlaps (calls from several host threads,
 * or on several streams of one device) race on the array: serialise them.
 * Like segtopk_batched_topk_host, the call waits for `stream` before it
 * returns.
 */
SEGTOPK_API int segtopk_batched_topk_host_noalloc(segtopk_dtype key_dtype, const void* keys, const int32_t* values,
                                      const int64_t* segment_offsets, int64_t num_segments, int32_t k,
                                      segtopk_direction direction, segtopk_determinism determinism,
                                      segtopk_tie_break tie_break, segtopk_ordering ordering,
                                      void* out_keys, int32_t* out_values, int64_t max_segment_len,
                                      void* stream);

/* Device workspace bytes segtopk_batched_topk_host needs for these sizes
 * (num_keys = number of key elements the offsets address, i.e. the largest
 * segment end): keys, offsets, output keys and, for pairs, the selected
 * source indices. Host-only arithmetic; 0 for negative or oversized
 * arguments. */
SEGTOPK_API size_t segtopk_host_workspace_bytes(segtopk_dtype key_dtype, int has_values, int64_t num_keys,
                                    int64_t num_segments, int32_t k);

/* Human-readable text of a status code (static storage). */
SEGTOPK_API const char* segtopk_status_string(int status);

/* cudaError_t of the last SEGTOPK_ERROR_CUDA on the calling thread (0 if none). */
SEGTOPK_API int segtopk_last_cuda_error(void);

/*
 * Reads and clears the device-side error word of the current device. The
 * kernels bound every wait on an asynchronous copy; a wait that gives up
 * sets this word (bit 0: copy wait timed out; bit 1: a segment longer than
 * the launch was planned for). Synchronises the device. Returns a status;
 * the word is stored in *error_word.
 */
SEGTOPK_API int segtopk_read_device_error(uint32_t* error_word);

/* Number of kernel launches the last successful call on this thread made. */
SEGTOPK_API int segtopk_last_launch_count(void);

/*
 * Diagnostics of the instrumented build (the library compiled with
 * SEGTOPK_STATS and SEGTOPK_TEST_HOOKS, a separate shared object); the
 * ordinary build returns SEGTOPK_ERROR_NOT_SUPPORTED from both and changes
 * nothing. The source pages have no counterpart of either.
 *
 * segtopk_read_stats: synchronises the device, then sums and clears the
 * per-CTA counters of the segment kernel over every launch since the last
 * read: out[0] CTAs, [1] cycles, [2] cycles to the first bound, [3] cycles
 * of the stream (first bound included), [4] cycles after it (final
 * selection, merge, output), [5] ring chunks, [6] list trims, [7] slices
 * read twice, [8] list entries at the end of the stream, [9] slices with a
 * sampled first bound, [10] digit-selection passes, [11] cycles warp 0
 * waited for copies, [12] keys, [13] chunk shares of warp 0 that held
 * candidates, [14] chunk offers that overflowed the list, [15] - [17]
 * cycles of the small sampled bound's per-warp minimums, merge and write,
 * [18] / [19] cycles of a lone CTA's final selection and of its output,
 * [20] - [22] cycles of every block selection's digit passes, counting
 * finishes and compactions; n entries are written (zeros past 23).
 *
 * segtopk_set_test_hooks: the bound (SM clock cycles) after which a wait on
 * a bulk copy gives up, and a number of bytes (a multiple of 16, at most
 * 4096) added to the expected byte count of every slice's first copy, so
 * that its wait runs out: tests of the bounded wait use it. The kernel then
 * sets bit 0 of the device error word, writes no output for the affected
 * segments and returns.
 */
SEGTOPK_API int segtopk_read_stats(uint64_t* out, int n);
SEGTOPK_API int segtopk_set_test_hooks(long long wait_limit_cycles, uint32_t first_copy_extra_bytes);

/*
 * segtopk_test_device_prep (instrumented build; host only, no CUDA call):
 * replays the per-device launch-preparation decisions the library makes
 * before every launch, on fresh records, for n launches on device ordinals
 * devices[i]. A launch of the segment kernel has cluster_widths[i] >= 1 and
 * smem_bytes[i] of dynamic shared memory; cluster_widths[i] <= 0 denotes a
 * warp-kernel launch. actions[i] receives the attribute calls that launch
 * would make, every earlier one taken to have succeeded: bit 0 raises the
 * shared-memory opt-in, bit 1 allows clusters wider than 8, bit 2 sets the
 * warp kernel's carveout; ~0 for a device ordinal outside 0..63. Function
 * attributes belong to each device's copy of a kernel, so each device gets
 * its own calls. Errors: SEGTOPK_ERROR_INVALID_VALUE for n < 0 or a null
 * array with n > 0.
 */
SEGTOPK_API int segtopk_test_device_prep(int n, const int* devices, const uint32_t* smem_bytes,
                                         const int* cluster_widths, uint32_t* actions);

#ifdef __cplusplus
}
#endif

#endif /* SEGTOPK_H_ */

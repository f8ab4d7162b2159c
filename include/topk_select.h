/*
 * Batched row-wise top-k selection on GB300 (sm_103a): the C ABI.
 *
 * The operation.  For every row r of a row-major fp32 score matrix, return the
 * k largest of the row's first L_r scores together with their in-row int32
 * indices, ordered by value descending; equal values go to the smaller index.
 * This is the selection a sparse-attention indexer runs for each query token
 * to decide which cached positions attention reads: "find the biggest 512
 * numbers in a list of a million" (The Secret GPU Kernel Behind DeepSeek V4.1
 * Flash, video transcript 2:28-2:53; the config line "index top k 512" at
 * 2:00-2:13).  Results are exact: every value comes back bit-for-bit and no
 * index repeats (DeepSeek V4.1 Flash, kernelbench model page, entry
 * "Single-launch CUDA bitonic selection").
 *
 * Value order: -inf < negatives < -0.0 < +0.0 < positives < +inf.  NaN is
 * not a value: a NaN inside a valid prefix is reported through the workspace
 * status word (TOPK_STATUS_NAN) and is left out of the selection.
 *
 * Method: one threshold per row that only rises, a shared-memory candidate
 * tray, 1024-element blocks streamed once (in units of eight consecutive
 * blocks visited in a seeded shuffled order), a bitonic sort that runs on the
 * tray only, and for short batches a split of
 * each row over several CTAs whose local winners a ticket-elected leader
 * merges (video transcript 3:18-5:45).  A long piece of a row may start from a
 * threshold that a sample of its first units only makes likely; the row's
 * result is checked against it at the end and, if fewer than k scores of the
 * row lie above it, the row is selected again (TOPK_STATUS_RESCAN).  A batch
 * of at least as many rows as the device has SMs, with rows of at most 65,536
 * scores, runs the same threshold-and-tray method with one CTA per row and
 * no split (the causal prefill's shape); results never depend on which path
 * ran.
 *
 * Memory: every pointer argument is caller-owned.  The library allocates no
 * memory, frees none, keeps no device state between calls and never
 * synchronises a stream except in topk_ws_status / topk_ws_stats, which say
 * so.  All device work is enqueued on `stream` (a cudaStream_t; NULL means the
 * legacy default stream) and runs on the device current at the call.
 *
 * Errors.  Return codes are decided on the host before anything is enqueued
 * (a launch failure is the one exception, TOPK_ERR_LAUNCH).  Problems only the
 * device can see (a NaN score, a length outside [0, n]) set bits in the
 * workspace status word; the kernels never trap and always finish.
 */
#ifndef TOPK_SELECT_H
#define TOPK_SELECT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define TOPK_OK 0
#define TOPK_ERR_SHAPE 1  /* rows < 0, n < 1, n >= 2^31, row_stride < n,
                             k < 1 or k > 2048, split out of range */
#define TOPK_ERR_NULL 2   /* scores / out_vals / out_idx NULL with rows > 0 */
#define TOPK_ERR_WS 3     /* ws NULL or not 256-byte aligned when needed */
#define TOPK_ERR_LAUNCH 4 /* the CUDA launch reported an error */
#define TOPK_ERR_ARG 5    /* another argument is invalid (see the function) */
#define TOPK_ERR_NOSPACE 6 /* topk_select_noalloc: the shape needs more workspace
                              than its built-in array holds */

/* Status bits the device sets in the workspace status word (sticky until
 * read by topk_ws_status). */
#define TOPK_STATUS_NAN 1u        /* a NaN inside some row's valid prefix */
#define TOPK_STATUS_BAD_LENGTH 2u /* lengths[r] outside [0, n]; clamped */
#define TOPK_STATUS_TIMEOUT 4u    /* a bounded wait (for a bulk copy, or for a
                                     hand-over between the CTA's warps) gave up;
                                     the affected rows' outputs are unspecified */
#define TOPK_STATUS_RESCAN 8u     /* information only: some row's speculative
                                     starting threshold left fewer than k of its
                                     scores above it, and the row was selected
                                     again from global memory (results exact) */
#define TOPK_STATUS_BOUNDS 16u    /* set by the debug build only (compiled with
                                     -DTOPK_DEBUG_BOUNDS=1): a shared- or
                                     global-memory index failed its check and
                                     the write was skipped */

/* Flags for topk_select_ex. */
#define TOPK_FLAG_IDENTITY_ORDER 1u /* visit units in address order instead of
                                       the shuffled order (diagnostic: the
                                       result is the same, the speed is not) */
#define TOPK_FLAG_TEST_STALL 256u   /* test of the bounded waits only: in every
                                       CTA the copy producer stops for good in
                                       front of its fourth ring stage, and every
                                       wait of the call gives up after 16,384
                                       polls (about a millisecond).  The call
                                       finishes, sets TOPK_STATUS_TIMEOUT and
                                       leaves the outputs unspecified; with
                                       split = 1 the workspace stays reusable
                                       (each row is one piece, no ticket) */

/* Largest supported k. */
#define TOPK_MAX_K 2048

/* Positions per block of the layer-20 block pool (topk_select_pool). */
#define TOPK_POOL_BLOCK 8

/*
 * topk_ws_bytes -- workspace size, in bytes, that topk_select needs for this
 * shape (with the automatic split plan).  Returns 0 for an invalid shape.
 *
 * The workspace holds a status word, per-row survivor and sort counters, the
 * per-row tickets of the split-row leader election and, when rows are split,
 * the CTAs' partial top-k lists (8 bytes x k rounded up to a power of two, per
 * CTA).  It is a pure function of (rows, n, k): it covers the plan of any
 * device with up to 256 SMs, so a workspace sized once serves every GPU.
 */
size_t topk_ws_bytes(int32_t rows, int64_t n, int32_t k);

/*
 * topk_select -- row-wise top-k.
 *
 *   scores           device fp32, element (r, i) at scores[r * row_stride + i],
 *                    read for i < L_r only.  Rows whose start is not 16-byte
 *                    aligned are read with plain loads instead of bulk copies.
 *   rows             number of rows (>= 0; 0 enqueues nothing).
 *   n                logical row width, 1 <= n < 2^31.
 *   row_stride       elements between row starts, >= n.
 *   lengths_or_null  device int32[rows]: L_r, the valid prefix of row r, in
 *                    [0, n]; NULL means L_r = n for every row.  A length
 *                    outside [0, n] is clamped and sets TOPK_STATUS_BAD_LENGTH.
 *   k                1 <= k <= 2048.
 *   out_vals         device fp32[rows * k]; row r's results at r * k + j.
 *   out_idx          device int32[rows * k], same layout.  Slots
 *                    j >= min(k, L_r) hold (-inf, -1).  Nothing outside
 *                    [0, rows * k) is written.
 *   ws               device workspace of at least topk_ws_bytes(rows, n, k)
 *                    bytes, 256-byte aligned, zero-filled once by the caller
 *                    after allocation.  Every call leaves the tickets at zero,
 *                    so the same workspace serves any number of later calls
 *                    in stream order; two calls that may overlap on the GPU
 *                    must not share one.
 *   stream           cudaStream_t to enqueue on (NULL: legacy default stream).
 *
 * All offsets are computed in 64-bit.  Returns TOPK_OK or an error code above;
 * on an error nothing is enqueued (except after TOPK_ERR_LAUNCH).
 */
int topk_select(const float* scores, int32_t rows, int64_t n,
                int64_t row_stride, const int32_t* lengths_or_null, int32_t k,
                float* out_vals, int32_t* out_idx, void* ws, void* stream);

/*
 * topk_split_plan -- the number of CTAs the automatic plan gives each row
 * (1 = unsplit) on the current device: the plan runs one CTA per SM (at most
 * 256), so it depends on (rows, n) and the device's SM count; with no device
 * to query it plans for 152 SMs (GB300).  0 for an invalid shape.
 */
int32_t topk_split_plan(int32_t rows, int64_t n);

/*
 * topk_ws_bytes_ex -- workspace size for an explicit split factor `split`
 * (0 = the automatic plan, else 1 <= split <= 64).  0 for an invalid shape.
 */
size_t topk_ws_bytes_ex(int32_t rows, int64_t n, int32_t k, int32_t split);

/*
 * topk_select_ex -- topk_select with the knobs the tests and the benchmark
 * use.  `split`: CTAs per row (0 = automatic, else 1..64; the workspace must
 * then be sized by topk_ws_bytes_ex with the same split).  `seed`: the 64-bit
 * Philox4x32-10 key of the block visiting order (topk_select uses a fixed
 * default).  `flags`: TOPK_FLAG_*.  The result never depends on split, seed
 * or flags; only the speed and the survivor counters do.
 */
int topk_select_ex(const float* scores, int32_t rows, int64_t n,
                   int64_t row_stride, const int32_t* lengths_or_null,
                   int32_t k, float* out_vals, int32_t* out_idx, void* ws,
                   void* stream, int32_t split, uint64_t seed, uint32_t flags);

/*
 * topk_ws_status -- synchronises `stream`, then reads and clears the status
 * word of `ws` (TOPK_STATUS_* bits) into *status_out.  Returns TOPK_OK,
 * TOPK_ERR_WS for a NULL/misaligned ws, TOPK_ERR_ARG for a NULL status_out,
 * or TOPK_ERR_LAUNCH if a CUDA call fails.
 */
int topk_ws_status(void* ws, uint32_t* status_out, void* stream);

/*
 * topk_ws_stats -- synchronises `stream`, then copies to host memory and
 * clears the per-row counters of `ws` laid out for (rows, n, k, split):
 *   survivors_out[r]  words of row r that entered a bitonic tray sort -- the
 *                     elements that ever reached a sorting step;
 *   sorts_out[r]      bitonic tray sorts run for row r;
 *   admitted_out[r]   elements of row r that passed the threshold test and
 *                     went to the tray (a superset of the sorted ones: before
 *                     each sort, words that can no longer reach the best k are
 *                     dropped).
 * Any output may be NULL.  Counters accumulate over calls until read.
 * Return codes as topk_ws_status.
 */
int topk_ws_stats(void* ws, int32_t rows, int64_t n, int32_t k, int32_t split,
                  uint32_t* survivors_out, uint32_t* sorts_out, uint32_t* admitted_out,
                  void* stream);

/*
 * topk_visit_order -- diagnostic: writes to device int32 order_out[m] the
 * order in which a CTA visits the m <= 256 units of one permutation chunk.
 * A unit is 8 consecutive 1024-element blocks (8192 elements, 32 KB; a row's
 * last unit may be shorter); unit u of a row starts at element 8192 * u.
 * Given the chunk's row, its first unit index in the row and the seed, the
 * order is the chunk's units sorted by (Philox4x32-10(counter =
 * (first_unit + j, row, 0, 0), key = seed) word 0 with its low 8 bits
 * cleared, j).  (The kernel keeps a row's short last unit out of the first
 * units of a piece, which its warm start reads: if it is among the first w of
 * a longer piece -- w = 3 for k <= 512, else up to 4 -- it trades places with
 * the entry after them, and in a piece of at most w units it trades places
 * with the last entry.  This call reports the order before that swap.)
 * Enqueued on `stream`.
 * Returns TOPK_ERR_ARG for m outside [1, 256], a negative first_unit or a
 * NULL order_out.
 */
int topk_visit_order(int32_t m, int32_t row, int64_t first_unit,
                     uint64_t seed, int32_t* order_out, void* stream);

/*
 * topk_timeline_read -- diagnostic of the instrumented build only (the library
 * compiled with -DTOPK_TIMELINE=1; every other build returns TOPK_ERR_ARG and
 * touches nothing).  Synchronises `stream`, copies the selection kernel's
 * timeline table to host_out (TOPK_TIMELINE_CTAS x TOPK_TIMELINE_SLOTS
 * uint64 values, CTA-major) and clears it.  Per CTA: global-timer stamps (ns)
 * of its start, set-up, first and last copy, each role's exit and four events
 * of each of its first eight pieces, its SM id and piece count, and SM cycles
 * spent per activity by one thread of each role.  Slot meanings are listed
 * with the table in topk_select.cu; the table holds the calls since the last
 * read (a CTA's stamps: the latest call).
 */
#define TOPK_TIMELINE_CTAS 512
#define TOPK_TIMELINE_SLOTS 128
int topk_timeline_read(unsigned long long* host_out, void* stream);

/*
 * topk_select_noalloc -- topk_select for callers that cannot allocate device
 * memory.  (An addition of this library: the pages describe no such call.)
 *
 * Some callers cannot call cudaMalloc where they select: real-time paths that
 * forbid allocation once they run (an allocation can block on the driver and
 * synchronise the device), and plug-ins whose host framework owns all device
 * memory and hands them only their input and output buffers.  This entry
 * point needs no workspace argument: it uses a 16 MiB array compiled into the
 * library (a file-scope __device__ array), which every GPU that loads the
 * library holds until the process exits.  It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *
 *   Arguments as topk_select, without `ws`.  `status_or_null`: optional device
 *   uint32 that receives this call's status word (TOPK_STATUS_* bits).
 *
 *   Limit: shapes whose topk_ws_bytes(rows, n, k) exceeds 16 MiB return
 *   TOPK_ERR_NOSPACE and enqueue nothing.
 *
 *   Set-up: the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and keeps it; make that
 *   first call before any stream capture.  Every call shares the one array:
 *   each call clears, on `stream`, the parts that must start at zero (status,
 *   tickets, counters, per-row words), and two calls that may overlap on the
 *   GPU -- on different streams, or from different host threads -- race on it
 *   and must be serialised by the caller.
 *
 * Returns TOPK_OK, TOPK_ERR_SHAPE, TOPK_ERR_NULL, TOPK_ERR_NOSPACE or
 * TOPK_ERR_LAUNCH.
 */
int topk_select_noalloc(const float* scores, int32_t rows, int64_t n,
                        int64_t row_stride, const int32_t* lengths_or_null,
                        int32_t k, float* out_vals, int32_t* out_idx,
                        uint32_t* status_or_null, void* stream);

/*
 * topk_select_pool -- topk_select plus the layer-20 block pool, in the same
 * pass over the scores.  The sweep that scores every position also groups
 * them into blocks of eight, gives each block the best score inside it,
 * keeps the best blocks with the newest ones pinned in, and upper indexers
 * score only inside that pool (The Secret GPU Kernel Behind DeepSeek V4.1
 * Flash, video transcript 7:22-7:46: about 2,000 blocks, 16,000 positions).
 *
 *   Per row r, with L_r its valid length: blocks b = 0 .. ceil(L_r / 8) - 1
 *   cover positions [8b, min(8b + 8, L_r)); a block's score is the largest of
 *   its scores (order as for topk_select: +0.0 above -0.0; NaN left out).
 *   The pool keeps the min(pinned_blocks, #blocks) newest blocks (the highest
 *   block indices) and fills the rest of its pool_blocks places with the
 *   best-scoring other blocks (score descending, ties to the smaller block
 *   index) while any is left.  out_pool[r * pool_blocks + j]: the kept block
 *   indices in ascending order, then -1.  Block b stands for positions
 *   8b .. 8b + 7 (those below L_r).
 *
 *   out_vals / out_idx: exactly as topk_select.  pool_blocks >= 1,
 *   0 <= pinned_blocks <= pool_blocks, pool_blocks - pinned_blocks <=
 *   TOPK_MAX_K.  out_pool: device int32[rows * pool_blocks], caller-owned.
 *   ws: device workspace of topk_pool_ws_bytes(...) bytes, 256-byte aligned,
 *   zero before the first call (the library leaves it so); its first word is
 *   the status word (topk_ws_status).  A row holding a NaN sets
 *   TOPK_STATUS_NAN; that row's pool is then unspecified.
 *
 * Returns TOPK_OK, TOPK_ERR_SHAPE, TOPK_ERR_ARG (pool arguments),
 * TOPK_ERR_NULL, TOPK_ERR_WS or TOPK_ERR_LAUNCH.  Enqueues two kernels on
 * `stream` (the selection, which also writes every block's maximum to the
 * workspace, then one CTA per row that picks the pool); allocates nothing.
 */
size_t topk_pool_ws_bytes(int32_t rows, int64_t n, int32_t k, int32_t pool_blocks,
                          int32_t pinned_blocks);
int topk_select_pool(const float* scores, int32_t rows, int64_t n, int64_t row_stride,
                     const int32_t* lengths_or_null, int32_t k, float* out_vals,
                     int32_t* out_idx, int32_t pool_blocks, int32_t pinned_blocks,
                     int32_t* out_pool, void* ws, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TOPK_SELECT_H */

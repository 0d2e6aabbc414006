/*
 * Sparse-attention indexer top-k with its fused output transform, for one
 * NVIDIA GB300 GPU (sm_103a). C ABI.
 *
 * What it computes. Each row b owns the window of fp32 scores
 *   scores[b * score_stride + row_starts[b] + p],  p = 0 .. seq_lens[b]-1
 * and keeps the k <= 2048 largest of them (sglang PR #35175 page,
 * "Implementation breakdown" item 2; "#26788 [JIT Kernel] DeepSeek-V4 DSA
 * indexer: faster top-k + page-table transform (runtime k <= 2048)" page,
 * "Executive summary"). Each kept position p is written transformed:
 *   PAGED : page_table[b * page_table_stride + p / page_size] * page_size
 *           + p % page_size   (PR #35175 page, "Key source snippets",
 *                              TopKProblem::transform_output / page_to_indices)
 *   RAGGED: p + out_offsets[b] (PR #35175 page, "Key source snippets",
 *                               TopKProblem::emit with its bias field)
 * When seq_lens[b] <= k every position is written and no score is read; the
 * remaining slots of the row hold -1, never transformed (PR #35175 page,
 * topk_ragged_kernel's trivial path and "Review highlights").
 *
 * Order. Scores compare by an order-preserving map of their fp32 bit pattern
 * to uint32 (a total order: -0.0 < +0.0; NaNs sort beyond +/-inf). In default
 * mode any maximal set is returned: the multiset of selected score bit
 * patterns is unique, and two results may differ only by swapping positions of
 * equal scores. With TOPK_DETERMINISTIC the lowest positions win among equal
 * scores, so the set is unique. The order of the k slots within a row is
 * unspecified.
 *
 * Memory. Every pointer argument is a DEVICE pointer unless stated otherwise.
 * The library never allocates; the caller owns all buffers. Work is enqueued
 * on `stream` (a cudaStream_t; NULL = the legacy default stream) and the calls
 * return without waiting for it. Scores are read only and never written.
 * The kernels are launched with programmatic dependent launch: they may be
 * scheduled while earlier work on the stream drains, but read and write no
 * memory until that work has completed, so stream order holds as usual.
 *
 * Errors. Argument errors are found on the host before anything is enqueued
 * and returned as a topk_status; the call then has no effect. A failed launch
 * returns TOPK_ERR_CUDA and leaves the CUDA error for cudaGetLastError().
 * Per-row data errors found on the device (seq_len < 0, row_start < 0, and
 * for packed PAGED rows page_table_row_start < 0) make that row empty (all
 * -1) and are counted in the workspace; read the count
 * with topk_read_device_errors().
 */
#ifndef SPARSE_ATTENTION_TOP_ROW_GB300_TOPK_H
#define SPARSE_ATTENTION_TOP_ROW_GB300_TOPK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TOPK_API __attribute__((visibility("default")))

/* The largest k (the pages' runtime bound, "runtime k <= 2048"). */
#define TOPK_MAX_K 2048
/* The largest supported page size (a power of two). */
#define TOPK_MAX_PAGE_SIZE (1 << 19)

typedef struct CUstream_st* topk_stream_t; /* same type as cudaStream_t */

typedef enum {
    TOPK_OK = 0,
    TOPK_ERR_ARG = 1,       /* a required pointer is null, batch < 0, a stride is negative or
                               score_stride is not a multiple of 4 */
    TOPK_ERR_ALIGN = 2,     /* scores is not 16-byte aligned */
    TOPK_ERR_K = 3,         /* k outside [1, TOPK_MAX_K] */
    TOPK_ERR_PAGE_SIZE = 4, /* page_size is not a power of two in [1, TOPK_MAX_PAGE_SIZE] */
    TOPK_ERR_WORKSPACE = 5, /* workspace is null or smaller than topk_workspace_bytes(batch) */
    TOPK_ERR_CUDA = 6       /* a CUDA call failed; cudaGetLastError() names the cause */
} topk_status;

/* flags bits */
#define TOPK_DETERMINISTIC 1u /* equal scores: lowest positions win */

/* bits of the device flags word read by topk_read_device_errors */
#define TOPK_DEVICE_FLAG_PLAN_MISMATCH 1u /* a transform found no plan for its (batch, k) and
                                             processed every row without one */
#define TOPK_DEVICE_FLAG_INTERNAL 2u      /* an internal consistency check failed (a library
                                             bug): an output slot index was out of range and
                                             the write was dropped */
#define TOPK_DEVICE_FLAG_TIMEOUT 4u       /* a wait for a bulk copy into shared memory gave up
                                             after about a second (the copy never completed);
                                             the kernel went on, so the rows it served are
                                             unreliable */

/*
 * Bytes of device workspace that topk_plan and the transforms need for
 * `batch` rows (a small header plus two int32 lists of `batch` entries).
 * Host only, pure. Returns 0 for batch < 0.
 */
TOPK_API size_t topk_workspace_bytes(int32_t batch);

/*
 * Plan: route every row by its length, once per set of seq_lens.
 * Counterpart of plan_topk_v2 / TopKKernel::plan ("#26788 [JIT Kernel]"
 * page, "Implementation breakdown": a plan kernel emits the metadata that the
 * transform dispatches on; "Key source snippets", topk.py).
 *
 *   seq_lens   int32 [batch], device. Negative entries are data errors
 *              (counted; those rows come out empty).
 *   batch      rows, >= 0.
 *   k          1 .. TOPK_MAX_K; must equal the k later given to the transform.
 *   workspace  device buffer of at least topk_workspace_bytes(batch) bytes,
 *              caller-owned; this call overwrites it. Any alignment of 16 B
 *              or more.
 *
 * One small kernel on `stream`. The plan sorts rows into length bands
 * (longest first) and, in batches of at most 64 rows, hands rows longer than
 * 32768 to a thread-block-cluster path that splits each such row over 4 SMs. A
 * transform run after it on the same stream (or otherwise ordered after it)
 * consumes the plan; one plan serves any number of transforms with the same
 * seq_lens, batch and k (e.g. every layer of a decode step). A transform whose
 * (batch, k) does not match the plan sets TOPK_DEVICE_FLAG_PLAN_MISMATCH and
 * still computes the right result, without the cluster path.
 */
TOPK_API int topk_plan(const int32_t* seq_lens, int32_t batch, int32_t k, void* workspace,
                       size_t workspace_bytes, topk_stream_t stream);

/*
 * PAGED top-k + page-table transform (decode).
 * Counterpart of topk_transform_paged / topk_transform_512_v2 ("#26788 [JIT
 * Kernel]" page, "Key source snippets", topk.py; renamed on the PR #35175
 * page, "Implementation breakdown" item 3).
 *
 *   scores            fp32, device, 16-byte aligned. Row b starts at
 *                     scores + b*score_stride; its window at + row_starts[b].
 *                     For every row the 16-byte-aligned span covering the
 *                     window, [floor4(start), ceil4(start + seq_len)), must lie
 *                     inside the allocation.
 *   score_stride      elements between rows; >= 0 and a multiple of 4
 *                     (0: all rows share one buffer).
 *   row_starts        int32 [batch] or NULL (NULL: every window starts at 0).
 *                     The logical position p counts from the window start.
 *   seq_lens          int32 [batch], the same values the plan saw; each at
 *                     most 2^31 - 8 (the window's 16-byte span is counted
 *                     in int32).
 *   page_table        int32, row b at page_table + b*page_table_stride; it must
 *                     hold ceil(seq_len / page_size) valid entries, and
 *                     page * page_size + page_size - 1 must fit int32.
 *   page_table_stride elements between page-table rows, >= 0.
 *   page_size         a power of two, 1 .. TOPK_MAX_PAGE_SIZE.
 *   batch, k          as given to topk_plan.
 *   workspace         the buffer topk_plan filled (the transform adds to its
 *                     device error count); at least topk_workspace_bytes(batch).
 *   out               int32 [batch, k], row-major; every slot is written.
 *   out_raw           int32 [batch, k] or NULL: the untransformed positions p
 *                     in the same slots as `out` (-1 in the padding).
 *   flags             0 or TOPK_DETERMINISTIC (any other bit: TOPK_ERR_ARG).
 */
TOPK_API int topk_transform_paged(const float* scores, int64_t score_stride,
                                  const int32_t* row_starts, const int32_t* seq_lens,
                                  const int32_t* page_table, int64_t page_table_stride,
                                  int32_t page_size, int32_t batch, int32_t k, void* workspace,
                                  size_t workspace_bytes, int32_t* out, int32_t* out_raw,
                                  uint32_t flags, topk_stream_t stream);

/*
 * PAGED top-k + page-table transform for packed rows (multi-query extend):
 * the score window keeps its batch-global start row_starts[b] while the
 * page-table lookup uses the row's request table and a request-local token
 * offset (the PR #33006 report, "fix(dsa): use FlashInfer fused top-k for
 * packed PAGED rows": "功能与动机" and "实现拆解" item 2, where
 * page_table_row_starts = row_starts - cu_seqlens_k[row_to_batch]).
 * A selected position p of row b writes
 *   page_table[r * page_table_stride + t / page_size] * page_size + t % page_size
 * with r = row_to_batch[b] and t = page_table_row_starts[b] + p.
 * Arguments as for topk_transform_paged, plus
 *   page_table_row_starts  int32 [batch] or NULL (0 for every row); a
 *                          negative entry is a data error (the row comes out
 *                          all -1 and the device error count goes up);
 *                          page_table_row_starts[b] + seq_lens[b] must fit
 *                          int32.
 *   row_to_batch           int32 [batch] or NULL (row b uses table row b);
 *                          caller's contract: each entry names a table row.
 * The page table must hold the entries t / page_size for every t of every
 * window. With both arrays NULL this is topk_transform_paged.
 */
TOPK_API int topk_transform_paged_packed(const float* scores, int64_t score_stride,
                                         const int32_t* row_starts, const int32_t* seq_lens,
                                         const int32_t* page_table, int64_t page_table_stride,
                                         int32_t page_size, const int32_t* page_table_row_starts,
                                         const int32_t* row_to_batch, int32_t batch, int32_t k,
                                         void* workspace, size_t workspace_bytes, int32_t* out,
                                         int32_t* out_raw, uint32_t flags, topk_stream_t stream);

/*
 * RAGGED top-k + offset transform (prefill / extend).
 * Counterpart of topk_transform_ragged_v2 / topk_ragged_kernel (PR #35175
 * page, "Implementation breakdown" items 2-3 and "Key source snippets").
 * Arguments as for topk_transform_paged, with
 *   out_offsets  int32 [batch]: added to every selected position of row b.
 *                out_offsets[b] + seq_len - 1 must fit int32. With
 *                out_offsets == row_starts the outputs are absolute
 *                positions in the flattened KV.
 * Unlike the pages' kernel, the scores buffer is never written: window heads
 * that are not 16-byte aligned are excluded by position, not masked in place.
 */
TOPK_API int topk_transform_ragged(const float* scores, int64_t score_stride,
                                   const int32_t* row_starts, const int32_t* seq_lens,
                                   const int32_t* out_offsets, int32_t batch, int32_t k,
                                   void* workspace, size_t workspace_bytes, int32_t* out,
                                   int32_t* out_raw, uint32_t flags, topk_stream_t stream);

/*
 * RAGGED top-k + offset transform fused with the SWA combine: each output row
 * is the row's top-k entries followed by its sliding-window tokens.
 * Counterpart of combine_topk_swa_indices / _combine_topk_swa_indices_kernel
 * (PR #30255 page, "sparse_prefill_utils.py"), which merges the top-k indices
 * with the sliding-window indices, topk_len = min((pos + 1) // COMPRESS_RATIO,
 * top_k), padded to PADDED_TOP_K; the page elides the body and the layout, and
 * this is the plainest reading of the signature. Fusing it saves the
 * combine's read of a [batch, k] index array.
 *
 *   scores ... flags   as for topk_transform_ragged; row b's window holds its
 *                      seq_lens[b] compressed entries (a causal query at
 *                      position pos over compressed KV has (pos + 1) //
 *                      COMPRESS_RATIO of them, which makes min(k, seq_len) the
 *                      page's topk_len).
 *   positions          int32 [batch], device: the query position pos of each
 *                      row (negative: no window tokens).
 *   window_size        tokens in the sliding window, 0 .. TOPK_MAX_SWA_WINDOW.
 *   swa_offsets        int32 [batch] or NULL: added to each window token (the
 *                      caller's map into its window KV space; NULL: 0).
 *   out_width          elements per output row (PADDED_TOP_K), at least
 *                      k + window_size.
 *   out                int32 [batch, out_width], row-major, every slot
 *                      written: slots [0, min(k, seq_len)) the selected
 *                      entries (position + out_offsets[b]; slot order
 *                      unspecified), then the window tokens pos - w + 1 .. pos
 *                      (w = min(window_size, pos + 1)) plus swa_offsets[b] in
 *                      ascending order, then -1.
 *   out_raw            int32 [batch, k] or NULL: as for topk_transform_ragged
 *                      (k columns, not out_width).
 * Status codes as for topk_transform_ragged; TOPK_ERR_ARG also for a null
 * positions array, a window outside its range or out_width < k + window_size.
 */
#define TOPK_MAX_SWA_WINDOW (1 << 20)
TOPK_API int topk_transform_ragged_swa(const float* scores, int64_t score_stride, const int32_t* row_starts,
                                       const int32_t* seq_lens, const int32_t* out_offsets, int32_t batch,
                                       int32_t k, void* workspace, size_t workspace_bytes,
                                       const int32_t* positions, int32_t window_size,
                                       const int32_t* swa_offsets, int32_t out_width, int32_t* out,
                                       int32_t* out_raw, uint32_t flags, topk_stream_t stream);

/*
 * Indexer logits: the producer upstream of the top-k, an FP8 multi-query
 * logits contraction on the tensor cores. The PR #35175 page (PR body) says
 * the contiguous-KV indexer writes its logit columns at absolute positions of
 * the batch-flattened KV, and the PR #36684 page ("Key source snippets",
 * server_args.py) ties the path to tcgen05/TMEM; neither prints the formula.
 * This computes the plainest reading, the lightning indexer's score:
 *
 *   logits[t * logits_stride + s] =
 *       kv_scale[s] * sum_{h < 64} weights[t * 64 + h] * max(0, q[t][h] . kv[s])
 *
 * for every s with max(ks[t], 0) <= s < min(ke[t], n_kv), with the dot
 * products over 128 FP8 E4M3 ("e4m3fn") coordinates accumulated in fp32.
 * Nothing outside each row's window is written, so row t is then the RAGGED
 * transform's window at row_start = ks[t], seq_len = ke[t] - ks[t] (with
 * score_stride = logits_stride).
 *
 *   q            device, [n_q, 64, 128] E4M3 codes (one byte each), row-major,
 *                16-byte aligned.
 *   kv           device, [n_kv, 128] E4M3 codes, row-major, 16-byte aligned.
 *   kv_scale     device fp32 [n_kv].
 *   weights      device fp32 [n_q, 64], row-major, 16-byte aligned.
 *   ks, ke       device int32 [n_q]: each query's key window (clamped to
 *                [0, n_kv); ke <= ks: an empty row, nothing written).
 *   n_q          queries, 0 .. TOPK_INDEXER_MAX_QUERIES.
 *   n_kv         keys, 0 .. TOPK_INDEXER_MAX_KEYS (int32 tile coordinates).
 *   logits       device fp32, row t at logits + t * logits_stride; the
 *                caller's buffer holds every written column.
 *   device_flags device uint32, required: TOPK_DEVICE_FLAG_TIMEOUT is OR-ed
 *                in if a wait on the kernel's own copies or MMAs gave up
 *                (the result is then unreliable); the caller zeroes it.
 * Status: TOPK_ERR_ARG for a negative count or stride, n_q or n_kv above
 * its maximum, or a null pointer; TOPK_ERR_ALIGN for q, kv or weights off 16 bytes;
 * TOPK_ERR_CUDA for a failed launch or tensor-map encoding. n_q == 0 or
 * n_kv == 0 is TOPK_OK and enqueues nothing. One launch, with programmatic
 * dependent launch like every kernel of the library.
 */
#define TOPK_INDEXER_HEADS 64
#define TOPK_INDEXER_DIM 128
#define TOPK_INDEXER_MAX_QUERIES (1 << 24)
#define TOPK_INDEXER_MAX_KEYS ((1 << 30) - 256)
TOPK_API int topk_indexer_logits(const uint8_t* q, const uint8_t* kv, const float* kv_scale,
                                 const float* weights, const int32_t* ks, const int32_t* ke, int32_t n_q,
                                 int32_t n_kv, float* logits, int64_t logits_stride,
                                 uint32_t* device_flags, topk_stream_t stream);

/*
 * Reads the workspace's device error count (rows with seq_len < 0 seen by the
 * plan, plus rows with row_start < 0, or for packed PAGED rows
 * page_table_row_start < 0, seen by each transform since the plan) and the
 * device flags word into HOST memory. Synchronises `stream`.
 *   host_error_rows  host int32*, required.
 *   host_flags       host uint32*, or NULL.
 */
TOPK_API int topk_read_device_errors(const void* workspace, int32_t* host_error_rows,
                                     uint32_t* host_flags, topk_stream_t stream);

/*
 * Allocation-free plan + RAGGED transform. The pages have no counterpart; this
 * entry point exists for callers that cannot allocate device memory, for
 * example a plugin host that hands a library only its input and output
 * buffers, or a serving process that reserves all GPU memory up front (for its
 * KV cache) and forbids allocations afterwards. It computes exactly what
 * topk_plan followed by topk_transform_ragged computes, with the plan's
 * workspace taken from an array built into the library instead of from the
 * caller.
 *
 *   Arguments as for topk_transform_ragged, without the workspace.
 *   batch must be at most TOPK_NOALLOC_MAX_BATCH; a larger batch returns
 *   TOPK_ERR_WORKSPACE and enqueues nothing.
 *
 * The built-in workspace is about 128 KB, held by every GPU that loads the
 * library until the process exits. The first call on a device looks up its
 * address (no allocation); make that first call before any stream capture.
 * Every call on a device shares the one array and rewrites it: calls whose
 * GPU work may overlap (different streams, or different host threads without
 * ordering) race and must be serialised by the caller. Device data-error
 * counts of this entry point are not reported.
 */
#define TOPK_NOALLOC_MAX_BATCH 16384
TOPK_API int topk_transform_ragged_noalloc(const float* scores, int64_t score_stride,
                                           const int32_t* row_starts, const int32_t* seq_lens,
                                           const int32_t* out_offsets, int32_t batch, int32_t k,
                                           int32_t* out, int32_t* out_raw, uint32_t flags,
                                           topk_stream_t stream);

/*
 * How many kernels one transform of `batch` rows launches on the current
 * device (after the plan's one): 1 or 2 (0 for batch <= 0; -1 if the device
 * cannot be queried). A batch whose every row can own a thread-block cluster
 * runs in one kernel; batches of up to 64 rows beyond that add the cluster
 * kernel for their long rows to the per-row kernel. Host only; the first call
 * on a device sets up the kernels' attributes, like the first transform.
 */
TOPK_API int topk_transform_launches(int32_t batch);

/* A static, human-readable name for a topk_status value. Host only. */
TOPK_API const char* topk_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_ATTENTION_TOP_ROW_GB300_TOPK_H */

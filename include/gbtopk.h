/*
 * gbtopk — batched variable-length exact top-K for the sparse-attention
 * (DSA) indexer decode step, on NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Every pointer argument is a plain pointer; "device" means it must
 * point into CUDA device memory (or managed memory) of the current device,
 * "host" means ordinary host memory.  All buffers are owned by the caller;
 * the library allocates nothing, keeps no state between calls and never
 * reads device data on the host, so every call can be captured in a CUDA
 * graph and replayed with new seq_lens / lengths contents.
 *
 * Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 * default stream).  Host-side argument checks happen before anything is
 * enqueued; a negative status means nothing was enqueued.
 */
#ifndef GBTOPK_H
#define GBTOPK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types of the score matrix. */
#define GBTOPK_F32 0  /* IEEE binary32 */
#define GBTOPK_BF16 1 /* bfloat16 */
#define GBTOPK_F16 2  /* IEEE binary16 */

/* Status codes. */
#define GBTOPK_OK 0
#define GBTOPK_HINT_DISCARDED 1 /* warning: pre_idx unusable, ran hint-free (result still exact) */
#define GBTOPK_EINVAL (-1)       /* shape, dtype, grouping or null-pointer error */
#define GBTOPK_EALIGN (-2)       /* an output (or the score base) is misaligned */
#define GBTOPK_EOVERLAP (-3)     /* two output buffers overlap */
#define GBTOPK_EUNSUPPORTED (-4) /* outside the supported envelope (e.g. top_k too large) */
#define GBTOPK_ECUDA (-5)        /* the CUDA runtime refused the launch */
#define GBTOPK_EWORKSPACE (-6)   /* workspace missing, misaligned or too small */
#define GBTOPK_ETIMEOUT (-7)     /* device flag: a bounded wait gave up (see gbtopk_device_status) */

/* Largest supported top_k. */
#define GBTOPK_MAX_TOP_K 16384

/* Flags of the `deterministic` argument (FlashInfer compact page-table PR
 * body, "SMALL/LARGE tie selection" and the deterministic output order).
 * 0 asks for none: ties at the k-th value are resolved arbitrarily and the
 * selected columns come in no particular order. */
#define GBTOPK_SORTED 1     /* each row ordered by (value descending, column ascending);
                               alone it implies GBTOPK_TIE_SMALL */
#define GBTOPK_TIE_SMALL 2  /* among values equal to the k-th, keep the smallest columns */
#define GBTOPK_TIE_LARGE 4  /* among values equal to the k-th, keep the largest columns */

/*
 * gbtopk_varlen — top-K over decode-step indexer logits.
 *
 * Defined by the FlashInfer `flashinfer.top_k_varlen` page (parameters
 * logits, seq_lens, top_k, pre_idx, compress_ratio, next_n, return_values,
 * out_indices, out_values; "returns") and the TensorRT-LLM PR #17821
 * "self-sampling (GVR V2) top-K decode kernels" (exactness, MTP window,
 * short-row and value-padding conventions).
 *
 *  logits       device, [num_rows, width] of `dtype`, inner stride 1, row
 *               stride `row_stride` elements (>= width; arena views with a
 *               padded stride are accepted).  Must be aligned to the element
 *               size.  Columns at or beyond a row's valid count are never read.
 *  seq_lens     device int32 [num_rows / next_n]: KV-token lengths.  Row r
 *               (request i = r / next_n, t = r % next_n) ranks its first
 *               n_r = max(0, (seq_lens[i] - next_n + t + 1) / compress_ratio)
 *               columns, clamped to `width`.
 *  next_n       >= 1, and num_rows % next_n == 0.
 *  compress_ratio >= 1.
 *  top_k        1 .. GBTOPK_MAX_TOP_K.
 *  pre_idx      device int32 [num_rows / next_n, top_k] or NULL: the previous
 *               step's top-K columns of each request, raw (no +1 offset),
 *               pre_idx[i][0] the argmax.  It only steers the threshold guess
 *               and never changes the result.  Entries outside [0, n_r)
 *               (including -1) and duplicates are ignored.  A pointer that
 *               is not 16-byte aligned is discarded with status
 *               GBTOPK_HINT_DISCARDED.
 *  out_indices  device int32 [num_rows, top_k], 16-byte aligned.  Row r gets
 *               min(top_k, n_r) column indices followed by -1.
 *  out_values   device, dtype of logits, [num_rows, top_k], 16-byte aligned,
 *               or NULL.  Selected values are bit copies; padding slots hold
 *               the lowest finite value of the dtype.
 *  deterministic  0 or a set of GBTOPK_SORTED / GBTOPK_TIE_SMALL /
 *               GBTOPK_TIE_LARGE (the two tie modes exclude each other;
 *               other bits are GBTOPK_EINVAL).  0: ties at the k-th value
 *               are resolved arbitrarily and the selected columns come in no
 *               particular order.  1 (GBTOPK_SORTED): ties take the smallest
 *               columns and each row is ordered by (value descending, column
 *               ascending).  A tie mode fixes the selected set; without
 *               GBTOPK_SORTED its order is unspecified.  Short rows
 *               (n_r <= top_k) come in column order unless sorted.
 *  workspace    device scratch of at least gbtopk_workspace_bytes(...) bytes,
 *               256-byte aligned.  Its first 4 bytes are a status word that
 *               should start at zero (see gbtopk_device_status); everything
 *               else is scratch that each call writes before reading (the
 *               row's guess, chunk ticket and candidate counters are written
 *               by the call's first kernel), so the contents need no
 *               initialisation and one workspace serves any sequence of
 *               calls on one stream.  Calls that may overlap in
 *               time (different streams, concurrent graph replays) need
 *               separate workspaces.
 *  stream       cudaStream_t.
 *
 * Returns GBTOPK_OK / GBTOPK_HINT_DISCARDED, or a negative status (nothing
 * enqueued).  num_rows == 0 is a no-op.
 */
int gbtopk_varlen(const void *logits, int dtype, int64_t num_rows, int64_t width,
                  int64_t row_stride, const int32_t *seq_lens, int32_t next_n,
                  int32_t compress_ratio, int32_t top_k, const int32_t *pre_idx,
                  int32_t *out_indices, void *out_values, int deterministic,
                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * gbtopk_page_table_transform — top-K fused with the compact page-table
 * transform.
 *
 * Defined by the FlashInfer compact page-table PR body quoted on the SGLang
 * PR #33237 page ("--dsa-topk-backend flashinfer with fused top-k"): for a
 * selected local score index idx,
 *     page = page_table[r, pt_row_start_r + idx / page_size]
 *     out  = page * page_size + idx % page_size,     out_raw = idx,
 * with -1 padding kept in both outputs, which stay positionally aligned.
 *
 *  scores       device, [num_rows, width] of `dtype`, inner stride 1, row
 *               stride `row_stride` elements.
 *  lengths      device int32 [num_rows]: valid scores per row.
 *  row_starts   device int32 [num_rows] or NULL: offset of the row's first
 *               valid score, in score elements.  The valid window is
 *               [row_start, row_start + length) clamped to the width; a
 *               row_start outside [0, width] gives an empty row.  Indices
 *               are local to row_start.
 *  page_table   device int32 [num_rows, pt_cols], inner stride 1, row stride
 *               pt_row_stride entries (non-contiguous tables are accepted).
 *  pt_row_starts  device int32 [num_rows] or NULL: first page-table entry of
 *               each row, in page-table entries.  NULL means row_starts when
 *               page_size == 1 and 0 when row_starts is NULL; NULL together
 *               with row_starts and page_size > 1 is GBTOPK_EINVAL.
 *  page_size    1 .. 2^30.  A page-table column outside [0, pt_cols) yields
 *               -1 in `out` (out_raw still holds idx).  page * page_size +
 *               idx % page_size is computed modulo 2^32: keeping it inside
 *               int32 is the caller's responsibility.
 *  top_k        1 .. GBTOPK_MAX_TOP_K.
 *  out          device int32 [num_rows, top_k], 16-byte aligned.
 *  out_raw      device int32 [num_rows, top_k], 16-byte aligned, or NULL; must
 *               not overlap `out` (GBTOPK_EOVERLAP).
 *  deterministic, workspace, stream: as for gbtopk_varlen.
 */
int gbtopk_page_table_transform(const void *scores, int dtype, int64_t num_rows,
                                int64_t width, int64_t row_stride,
                                const int32_t *lengths, const int32_t *row_starts,
                                const int32_t *page_table, int64_t pt_cols,
                                int64_t pt_row_stride, const int32_t *pt_row_starts,
                                int32_t page_size, int32_t top_k, int32_t *out,
                                int32_t *out_raw, int deterministic, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * gbtopk_ragged_transform — top-K fused with the ragged KV index offset.
 *
 * Defined by the SGLang TopK ops wiki, fast_topk_transform_ragged_fused (its
 * top-k indices shifted by a per-row offset for a ragged KV layout, the
 * offsets topk_indices_offset of shape (B)): the selection is the one of
 * gbtopk_page_table_transform's rows, and each selected row-local index idx
 * is written as idx + topk_indices_offset[r] (modulo 2^32); -1 padding stays
 * -1.
 *
 *  scores, lengths, row_starts, top_k, deterministic, workspace, stream:
 *               as for gbtopk_page_table_transform (valid window
 *               [row_start, row_start + length) clamped to the width).
 *  topk_indices_offset  device int32 [num_rows].
 *  out          device int32 [num_rows, top_k], 16-byte aligned.
 */
int gbtopk_ragged_transform(const void *scores, int dtype, int64_t num_rows, int64_t width,
                            int64_t row_stride, const int32_t *lengths, const int32_t *row_starts,
                            const int32_t *topk_indices_offset, int32_t top_k, int32_t *out,
                            int deterministic, void *workspace, size_t workspace_bytes, void *stream);

/*
 * gbtopk_page_table_transform_cu_seqlens — top-K fused with a page_size-1
 * page table indexed by request.
 *
 * Defined by the SGLang TopK ops wiki, fast_topk_transform_fused (page table
 * with page_size 1 and cu_seqlens_q of shape (Batch + 1)): score row r
 * belongs to request b with cu_seqlens_q[b] <= r < cu_seqlens_q[b + 1], and
 * each selected row-local index idx is written as page_table[b, idx]; an idx
 * at or beyond pt_cols gives -1, and a row that no request covers is empty
 * (all -1).
 *
 *  scores, lengths, row_starts, top_k, deterministic, workspace, stream:
 *               as for gbtopk_page_table_transform.
 *  page_table   device int32 [num_reqs, pt_cols], inner stride 1, row stride
 *               pt_row_stride entries.
 *  cu_seqlens_q device int32 [num_reqs + 1], nondecreasing.
 *  out          device int32 [num_rows, top_k], 16-byte aligned.
 */
int gbtopk_page_table_transform_cu_seqlens(const void *scores, int dtype, int64_t num_rows,
                                           int64_t width, int64_t row_stride, const int32_t *lengths,
                                           const int32_t *row_starts, const int32_t *page_table,
                                           int64_t pt_cols, int64_t pt_row_stride,
                                           const int32_t *cu_seqlens_q, int64_t num_reqs,
                                           int32_t top_k, int32_t *out, int deterministic,
                                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * gbtopk_workspace_bytes — scratch needed by a call with this geometry.
 * A pure function of its arguments (capture-stable).  The workspace holds a
 * device status word plus, when rows are long enough to be split across
 * thread blocks, per-row candidate buffers, counters and histograms (the
 * multi-CTA split described on the FlashInfer `top_k_varlen` page, parameter
 * `workspace`).  Returns 0 for invalid arguments.
 */
size_t gbtopk_workspace_bytes(int64_t num_rows, int64_t width, int32_t top_k, int dtype);

/*
 * gbtopk_device_status — reads (and clears) the device status word of a
 * workspace.  Synchronises `stream`.  *flags receives a bit set:
 *   bit 0  a bounded wait on an asynchronous copy gave up; the affected rows
 *          (on the three-kernel path: every row of that call) were
 *          recomputed from global memory, so the outputs are exact;
 *   bit 1  a copy did not land even within a second bounded wait: the
 *          outputs of that call are not reliable (the shared memory the copy
 *          targets was not reused; rows whose selection needed it were left
 *          unwritten or written unsorted).
 * The waits are bounded by a poll count; the environment variable
 * GBTOPK_WAIT_POLLS (a positive integer, read once per process) lowers the
 * first wait's count, which exercises the recovery of bit 0 in tests.
 * Returns GBTOPK_OK, GBTOPK_EINVAL or GBTOPK_ECUDA.  The pages define no
 * such call.
 */
int gbtopk_device_status(void *workspace, uint32_t *flags, void *stream);

/*
 * gbtopk_plan_query — the launch plan for a geometry, for inspection and
 * tests.  `out` must hold 13 entries: out[0..12] = {columns per chunk of a
 * split row, chunks of the widest split row (1 when no row is split),
 * longest row finished by the one-block row kernel, row-kernel shared
 * memory bytes, split (0/1), candidate entries reserved per split row,
 * stream-kernel shared memory bytes (0 unless split rows take the three-
 * kernel path), finalize-kernel shared memory bytes (likewise), workspace
 * bytes, workspace bytes per row, row-kernel shared memory bytes with
 * GBTOPK_SORTED, fused (1 when split rows take the two-kernel path: the
 * row kernel's guess, then one chunk-kernel block per chunk, the row's last
 * block selecting it), chunk-kernel shared memory bytes (fused plans)}.
 * Returns GBTOPK_OK or GBTOPK_EINVAL / GBTOPK_EUNSUPPORTED (nothing is
 * written then).
 */
int gbtopk_plan_query(int64_t num_rows, int64_t width, int32_t top_k, int dtype,
                      int64_t *out);

/*
 * gbtopk_varlen_static_ws — gbtopk_varlen without a caller-provided
 * workspace.  The pages define no such call; it exists for callers that
 * cannot allocate device memory where they need top-K: code running while
 * a CUDA graph is being captured (cudaMalloc cannot be captured), engines
 * whose device memory belongs to an external allocator or planner that
 * forbids side allocations, and plugin hosts that only pass in tensors they
 * own.  It allocates nothing: the scratch is one 16 MiB buffer compiled into
 * the library (a file-scope __device__ array), reserved on every GPU that
 * loads the library and held until the process exits.
 *
 * Arguments, outputs and status codes are those of gbtopk_varlen, minus the
 * workspace.  A geometry whose workspace (gbtopk_workspace_bytes) exceeds
 * 16 MiB is refused with GBTOPK_EWORKSPACE before anything is enqueued; for
 * example a 64 x 163840 fp32 batch with top_k 2048 needs about 6.3 MiB.
 *
 * The first call on a device looks up the buffer's device address (once per
 * device); make that first call before capturing a CUDA graph.  The address
 * belongs to the device's context: after cudaDeviceReset the process must
 * not call this entry point again.  All calls on a device share the one
 * buffer and its contents carry over between calls (nothing needs clearing:
 * each call writes the scratch it reads), so calls that may overlap in time
 * on the GPU — other streams, concurrent graph replays, other host threads —
 * race on it and must be serialised by the caller.  The buffer's device
 * status word (see gbtopk_device_status) cannot be read on this path: the
 * bounded-wait flags of these calls are not reported.
 */
int gbtopk_varlen_static_ws(const void *logits, int dtype, int64_t num_rows, int64_t width,
                            int64_t row_stride, const int32_t *seq_lens, int32_t next_n,
                            int32_t compress_ratio, int32_t top_k, const int32_t *pre_idx,
                            int32_t *out_indices, void *out_values, int deterministic,
                            void *stream);

/* Human-readable name of a status code (static string).  The pages define no
 * such call; the codes follow the error cases of the FlashInfer
 * `top_k_varlen` page ("Raises") and the status convention above. */
const char *gbtopk_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* GBTOPK_H */

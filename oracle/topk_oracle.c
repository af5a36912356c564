/*
 * Plain CPU oracle for batched variable-length exact top-K.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library: it is the plain definition written out, slow on purpose.
 *
 * What it computes (sources are the four pages on the DSA indexer top-K):
 *
 *  - Row length (FlashInfer `top_k_varlen` docs, parameter `seq_lens`;
 *    TensorRT-LLM PR #17821, "MTP coverage"): row r belongs to request
 *    i = r / next_n with offset t = r % next_n and ranks its first
 *    max(0, (seq_lens[i] - next_n + t + 1) // compress_ratio) columns,
 *    clamped to the buffer width.  A non-positive numerator is an empty row.
 *
 *  - Selection (TensorRT-LLM PR #17821, summary and "Test coverage": exact
 *    top-K, ties interchangeable, signed zeros equal): the valid columns are
 *    ordered by (value descending, column ascending) and the first
 *    min(k, n) are kept.  Values are compared as fp64 (every fp32, bf16 and
 *    fp16 value widens exactly), so -0.0 and +0.0 compare equal and fall
 *    back to the column order.  NaN is outside the contract.
 *
 *  - Padding (TensorRT-LLM PR #17821, short-path and value-output commits):
 *    unused index slots are -1; unused value slots hold the lowest finite
 *    value of the dtype (fp32 -FLT_MAX; bf16 0xFF7F and fp16 0xFBFF by the
 *    same convention).  Selected values are bit copies of the input.
 *
 *  - Compact page-table transform (SGLang PR #33237, quoted FlashInfer PR
 *    body): for a selected local index idx,
 *        page   = page_table[row, pt_row_start + idx / page_size]
 *        out    = page * page_size + idx % page_size,   out_raw = idx,
 *    -1 stays -1 in both.  row_starts are in score elements,
 *    page_table_row_starts in page-table entries.
 *
 * Readings where the pages are silent (each one is listed in the design
 * notes):
 *  - output order is (value desc, index asc) for every row, including rows
 *    with n <= k;
 *  - a page-table row's valid columns are [row_start, row_start + len)
 *    clamped to the width; a row_start outside [0, width] gives an empty row;
 *  - a page-table column outside [0, pt_cols) yields -1 in `out`;
 *  - page * page_size + idx % page_size must fit in int32 (error otherwise).
 *
 * Two more epilogues of the same selection (SGLang TopK ops wiki,
 * fast_topk_transform_ragged_fused and fast_topk_transform_fused):
 *  - ragged KV offset: out = idx + topk_indices_offset[row], -1 stays -1;
 *  - page table with page_size 1 over requests: row r belongs to request b
 *    with cu_seqlens_q[b] <= r < cu_seqlens_q[b + 1], and
 *    out = page_table[b, idx], -1 stays -1.
 * Readings: idx is the row-local index in both (relative to row_start); a
 * row no request covers is empty (all -1); an idx at or beyond pt_cols
 * yields -1; idx + offset must fit in int32 (error otherwise).
 *
 * Tie selection (FlashInfer compact page-table PR body: "SMALL/LARGE tie
 * selection", independent of the canonical output-order sort): SMALL keeps,
 * among values equal to the k-th, the smallest columns (the selection
 * above); LARGE keeps the largest.  The kept set is reported in the
 * canonical (value desc, index asc) order in both modes.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define OR_F32 0
#define OR_BF16 1
#define OR_F16 2

#define OR_OK 0
#define OR_EINVAL (-1)
#define OR_ENOMEM (-2)
#define OR_ERANGE (-3)

static int elem_size(int dtype)
{
    return dtype == OR_F32 ? 4 : 2;
}

/* Exact widening of one stored element to double. */
static double widen(const void *base, int dtype, int64_t i)
{
    if (dtype == OR_F32) {
        float f;
        memcpy(&f, (const char *)base + 4 * i, 4);
        return (double)f;
    }
    uint16_t h;
    memcpy(&h, (const char *)base + 2 * i, 2);
    if (dtype == OR_BF16) {
        /* bfloat16 is the upper half of an IEEE binary32 */
        uint32_t u = (uint32_t)h << 16;
        float f;
        memcpy(&f, &u, 4);
        return (double)f;
    }
    /* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits */
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 31;
    int fr = h & 1023;
    double mag;
    if (ex == 0)
        mag = ldexp((double)fr, -24); /* zero and subnormals */
    else if (ex == 31)
        mag = fr ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + fr), ex - 25);
    return sign ? -mag : mag;
}

/* Valid column count of row t of a request (FlashInfer `top_k_varlen` docs,
 * parameter `seq_lens`).  Integer arithmetic in 64 bits; the numerator is
 * tested before dividing so the floor division never sees a negative. */
int64_t oracle_row_length(int64_t seq_len, int64_t next_n, int64_t t,
                          int64_t compress_ratio, int64_t width)
{
    int64_t num = seq_len - next_n + t + 1;
    if (num <= 0)
        return 0;
    int64_t n = num / compress_ratio;
    return n < width ? n : width;
}

typedef struct {
    double v;
    int64_t j;
} item_t;

static int by_value_desc_index_asc(const void *a, const void *b)
{
    const item_t *x = (const item_t *)a;
    const item_t *y = (const item_t *)b;
    if (x->v > y->v)
        return -1;
    if (x->v < y->v)
        return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j ? 1 : 0);
}

static void write_pad_value(void *out_val, int dtype, int64_t slot)
{
    if (dtype == OR_F32) {
        uint32_t u = 0xFF7FFFFFu; /* -FLT_MAX */
        memcpy((char *)out_val + 4 * slot, &u, 4);
    } else {
        uint16_t u = dtype == OR_BF16 ? 0xFF7Fu : 0xFBFFu;
        memcpy((char *)out_val + 2 * slot, &u, 2);
    }
}

/* Top-k of one row whose column 0 sits at `row` and which has n valid
 * columns.  Writes k indices (local to `row`) and optionally k values. */
int oracle_select_row(const void *row, int dtype, int64_t n, int32_t k,
                      int32_t *out_idx, void *out_val)
{
    if (k < 1 || n < 0 || (dtype != OR_F32 && dtype != OR_BF16 && dtype != OR_F16))
        return OR_EINVAL;
    int es = elem_size(dtype);
    item_t *items = NULL;
    if (n > 0) {
        items = (item_t *)malloc((size_t)n * sizeof(item_t));
        if (!items)
            return OR_ENOMEM;
        for (int64_t j = 0; j < n; ++j) {
            items[j].v = widen(row, dtype, j);
            items[j].j = j;
        }
        qsort(items, (size_t)n, sizeof(item_t), by_value_desc_index_asc);
    }
    int64_t m = n < k ? n : k;
    for (int64_t s = 0; s < k; ++s) {
        if (s < m) {
            out_idx[s] = (int32_t)items[s].j;
            if (out_val)
                memcpy((char *)out_val + es * s, (const char *)row + es * items[s].j, es);
        } else {
            out_idx[s] = -1;
            if (out_val)
                write_pad_value(out_val, dtype, s);
        }
    }
    free(items);
    return OR_OK;
}

/* The whole batch of FlashInfer `top_k_varlen`: logits [num_rows, width]
 * with row stride `row_stride` elements; seq_lens [num_rows / next_n]. */
static int by_value_desc_index_desc(const void *a, const void *b)
{
    const item_t *x = (const item_t *)a;
    const item_t *y = (const item_t *)b;
    if (x->v > y->v)
        return -1;
    if (x->v < y->v)
        return 1;
    return (x->j > y->j) ? -1 : (x->j < y->j ? 1 : 0);
}

/* Top-k of one row with LARGE ties: the first min(k, n) columns in
 * (value desc, index desc) order are kept, then reported in the canonical
 * (value desc, index asc) order; padding as for oracle_select_row. */
int oracle_select_row_large_ties(const void *row, int dtype, int64_t n, int32_t k,
                                 int32_t *out_idx, void *out_val)
{
    if (k < 1 || n < 0 || (dtype != OR_F32 && dtype != OR_BF16 && dtype != OR_F16))
        return OR_EINVAL;
    int es = elem_size(dtype);
    item_t *items = NULL;
    const int64_t m = (n < k) ? n : k;  /* kept columns */
    if (n > 0) {
        items = (item_t *)malloc((size_t)n * sizeof(item_t));
        if (!items)
            return OR_ENOMEM;
        for (int64_t j = 0; j < n; ++j) {
            items[j].v = widen(row, dtype, j);
            items[j].j = j;
        }
        qsort(items, (size_t)n, sizeof(item_t), by_value_desc_index_desc);
        qsort(items, (size_t)m, sizeof(item_t), by_value_desc_index_asc);
    }
    for (int64_t s = 0; s < k; ++s) {
        if (s < m) {
            out_idx[s] = (int32_t)items[s].j;
            if (out_val)
                memcpy((char *)out_val + es * s, (const char *)row + es * items[s].j, es);
        } else {
            out_idx[s] = -1;
            if (out_val)
                write_pad_value(out_val, dtype, s);
        }
    }
    free(items);
    return OR_OK;
}

/* oracle_topk_varlen with a tie mode: tie_large = 0 keeps the smallest
 * columns among ties, 1 the largest. */
int oracle_topk_varlen_ties(const void *logits, int dtype, int64_t num_rows,
                            int64_t width, int64_t row_stride,
                            const int32_t *seq_lens, int32_t next_n,
                            int32_t compress_ratio, int32_t k, int tie_large,
                            int32_t *out_idx, void *out_val)
{
    if (num_rows < 0 || width < 0 || row_stride < width || next_n < 1 ||
        compress_ratio < 1 || k < 1 || num_rows % next_n != 0)
        return OR_EINVAL;
    int es = elem_size(dtype);
    for (int64_t r = 0; r < num_rows; ++r) {
        int64_t n = oracle_row_length(seq_lens[r / next_n], next_n, r % next_n,
                                      compress_ratio, width);
        const char *row = (const char *)logits + (size_t)(r * row_stride) * es;
        void *ov = out_val ? (char *)out_val + (size_t)(r * k) * es : NULL;
        int rc = tie_large ? oracle_select_row_large_ties(row, dtype, n, k, out_idx + r * k, ov)
                           : oracle_select_row(row, dtype, n, k, out_idx + r * k, ov);
        if (rc != OR_OK)
            return rc;
    }
    return OR_OK;
}

int oracle_topk_varlen(const void *logits, int dtype, int64_t num_rows,
                       int64_t width, int64_t row_stride,
                       const int32_t *seq_lens, int32_t next_n,
                       int32_t compress_ratio, int32_t k, int32_t *out_idx,
                       void *out_val)
{
    if (num_rows < 0 || width < 0 || row_stride < width || next_n < 1 ||
        compress_ratio < 1 || k < 1 || num_rows % next_n != 0)
        return OR_EINVAL;
    int es = elem_size(dtype);
    for (int64_t r = 0; r < num_rows; ++r) {
        int64_t n = oracle_row_length(seq_lens[r / next_n], next_n, r % next_n,
                                      compress_ratio, width);
        const char *row = (const char *)logits + (size_t)(r * row_stride) * es;
        int rc = oracle_select_row(row, dtype, n, k, out_idx + r * k,
                                   out_val ? (char *)out_val + (size_t)(r * k) * es : NULL);
        if (rc != OR_OK)
            return rc;
    }
    return OR_OK;
}

/* Valid window of a page-table row: [row_start, row_start + len) clamped
 * to the width; a start outside [0, width] makes the row empty. */
int64_t oracle_ragged_length(int64_t len, int64_t row_start, int64_t width)
{
    if (row_start < 0 || row_start > width || len <= 0)
        return 0;
    int64_t room = width - row_start;
    return len < room ? len : room;
}

/* Fused top-k + compact page-table transform (SGLang PR #33237, quoted
 * FlashInfer PR body).  scores [num_rows, width] with row stride; lengths
 * per row; optional row_starts (score elements); page_table [*, pt_cols]
 * with row stride pt_row_stride; optional pt_row_starts (entries). */
int oracle_page_table_transform(const void *scores, int dtype, int64_t num_rows,
                                int64_t width, int64_t row_stride,
                                const int32_t *lengths, const int32_t *row_starts,
                                const int32_t *page_table, int64_t pt_cols,
                                int64_t pt_row_stride, const int32_t *pt_row_starts,
                                int32_t page_size, int32_t k, int32_t *out,
                                int32_t *out_raw)
{
    if (num_rows < 0 || width < 0 || row_stride < width || k < 1 ||
        page_size < 1 || pt_cols < 0 || pt_row_stride < pt_cols)
        return OR_EINVAL;
    if (page_size > 1 && row_starts && !pt_row_starts)
        return OR_EINVAL; /* starts are in different units; must be explicit */
    int es = elem_size(dtype);
    int32_t *raw = (int32_t *)malloc((size_t)k * sizeof(int32_t));
    if (!raw)
        return OR_ENOMEM;
    for (int64_t r = 0; r < num_rows; ++r) {
        int64_t rs = row_starts ? row_starts[r] : 0;
        int64_t n = oracle_ragged_length(lengths[r], rs, width);
        const char *row = (const char *)scores + (size_t)(r * row_stride + (n > 0 ? rs : 0)) * es;
        int rc = oracle_select_row(row, dtype, n, k, raw, NULL);
        if (rc != OR_OK) {
            free(raw);
            return rc;
        }
        int64_t pt_start = pt_row_starts ? pt_row_starts[r] : (page_size == 1 ? rs : 0);
        for (int32_t s = 0; s < k; ++s) {
            int32_t idx = raw[s];
            if (out_raw)
                out_raw[r * k + s] = idx;
            if (idx < 0) {
                out[r * k + s] = -1;
                continue;
            }
            int64_t col = pt_start + idx / page_size;
            if (col < 0 || col >= pt_cols) {
                out[r * k + s] = -1;
                continue;
            }
            int64_t page = page_table[r * pt_row_stride + col];
            int64_t phys = page * page_size + idx % page_size;
            if (phys < INT32_MIN || phys > INT32_MAX) {
                free(raw);
                return OR_ERANGE;
            }
            out[r * k + s] = (int32_t)phys;
        }
    }
    free(raw);
    return OR_OK;
}

/* Ragged KV offset transform (SGLang TopK ops, fast_topk_transform_ragged_fused):
 * each selected row-local index idx becomes idx + offsets[row]; -1 stays -1. */
int oracle_ragged_offset_transform(const void *scores, int dtype, int64_t num_rows,
                                   int64_t width, int64_t row_stride,
                                   const int32_t *lengths, const int32_t *row_starts,
                                   const int32_t *offsets, int32_t k, int32_t *out)
{
    if (num_rows < 0 || width < 0 || row_stride < width || k < 1 || !offsets)
        return OR_EINVAL;
    int es = elem_size(dtype);
    int32_t *raw = (int32_t *)malloc((size_t)k * sizeof(int32_t));
    if (!raw)
        return OR_ENOMEM;
    for (int64_t r = 0; r < num_rows; ++r) {
        int64_t rs = row_starts ? row_starts[r] : 0;
        int64_t n = oracle_ragged_length(lengths[r], rs, width);
        const char *row = (const char *)scores + (size_t)(r * row_stride + (n > 0 ? rs : 0)) * es;
        int rc = oracle_select_row(row, dtype, n, k, raw, NULL);
        if (rc != OR_OK) {
            free(raw);
            return rc;
        }
        for (int32_t s = 0; s < k; ++s) {
            if (raw[s] < 0) {
                out[r * k + s] = -1;
                continue;
            }
            int64_t v = (int64_t)raw[s] + (int64_t)offsets[r];
            if (v < INT32_MIN || v > INT32_MAX) {
                free(raw);
                return OR_ERANGE;
            }
            out[r * k + s] = (int32_t)v;
        }
    }
    free(raw);
    return OR_OK;
}

/* Page-table transform with page_size 1 over requests (SGLang TopK ops,
 * fast_topk_transform_fused): row r belongs to request b with
 * cu_seqlens_q[b] <= r < cu_seqlens_q[b + 1] (a row no request covers is
 * empty), and each selected row-local index idx becomes page_table[b, idx]
 * (-1 when idx >= pt_cols); -1 stays -1. */
int oracle_seqs_page_table_transform(const void *scores, int dtype, int64_t num_rows,
                                     int64_t width, int64_t row_stride,
                                     const int32_t *lengths, const int32_t *row_starts,
                                     const int32_t *page_table, int64_t pt_cols,
                                     int64_t pt_row_stride, const int32_t *cu_seqlens_q,
                                     int64_t num_reqs, int32_t k, int32_t *out)
{
    if (num_rows < 0 || width < 0 || row_stride < width || k < 1 || num_reqs < 0 ||
        pt_cols < 0 || pt_row_stride < pt_cols || !cu_seqlens_q)
        return OR_EINVAL;
    int es = elem_size(dtype);
    int32_t *raw = (int32_t *)malloc((size_t)k * sizeof(int32_t));
    if (!raw)
        return OR_ENOMEM;
    for (int64_t r = 0; r < num_rows; ++r) {
        int64_t b = -1;
        for (int64_t q = 0; q < num_reqs; ++q)  /* plain linear search */
            if (cu_seqlens_q[q] <= r && r < cu_seqlens_q[q + 1]) {
                b = q;
                break;
            }
        int64_t rs = row_starts ? row_starts[r] : 0;
        int64_t n = b < 0 ? 0 : oracle_ragged_length(lengths[r], rs, width);
        const char *row = (const char *)scores + (size_t)(r * row_stride + (n > 0 ? rs : 0)) * es;
        int rc = oracle_select_row(row, dtype, n, k, raw, NULL);
        if (rc != OR_OK) {
            free(raw);
            return rc;
        }
        for (int32_t s = 0; s < k; ++s) {
            int32_t idx = raw[s];
            out[r * k + s] = (idx < 0 || idx >= pt_cols) ? -1 : page_table[b * pt_row_stride + idx];
        }
    }
    free(raw);
    return OR_OK;
}

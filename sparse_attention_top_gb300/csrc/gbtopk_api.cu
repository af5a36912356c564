// Host side of gbtopk: argument checks, the launch plan, and the C ABI
// declared in include/gbtopk.h.  No device data is ever read on the host.
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include <cuda_runtime.h>

#include "gbtopk.h"
#include "gbtopk_internal.h"

namespace gbtopk {
namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_bytes(int dtype) { return dtype == GBTOPK_F32 ? 4 : 2; }

bool overlaps(const void *a, size_t an, const void *b, size_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

}  // namespace

// The plan depends only on (num_rows, width, top_k, dtype): never on the
// contents of seq_lens / lengths, so it is fixed at CUDA-graph capture.
//
// Rows of up to direct_max columns are finished by the row kernel alone
// (one block per row, the row staged in shared memory).  When the width
// allows longer rows, those are split into chunks.  With top_k up to
// kPairSortMax the split rows run through two kernels: the row kernel
// (threshold guess) and the chunk kernel (one block per kFusedChunkBytes
// chunk, the row's last block selecting the row).  Larger top_k takes three:
// the row kernel, the persistent stream kernel (kChunkBytes chunks) and the
// finalize kernel, which has room for the larger selection.
int make_plan(int64_t num_rows, int64_t width, int32_t top_k, int dtype, Plan *plan) {
    if (num_rows < 0 || width < 0 || top_k < 1 ||
        (dtype != GBTOPK_F32 && dtype != GBTOPK_BF16 && dtype != GBTOPK_F16))
        return GBTOPK_EINVAL;
    if (top_k > GBTOPK_MAX_TOP_K) return GBTOPK_EUNSUPPORTED;
    if (width > INT32_MAX || num_rows > INT32_MAX) return GBTOPK_EUNSUPPORTED;
    const int es = elem_bytes(dtype);
    const int64_t chunk = kChunkBytes / es;
    Plan pl{};
    int sel_cap = 32;
    while (sel_cap < top_k) sel_cap <<= 1;
    pl.sel_cap = sel_cap;
    pl.chunk = static_cast<int32_t>(chunk);
    // the guess: its kGuessBins counters followed by the sample (kSampleSize
    // keys); direct rows then reuse the region for the candidate histogram
    // (kBins counters) and the selection (sel_cap pairs), the sample being dead
    const size_t guess = static_cast<size_t>(kGuessBins) * 4 + static_cast<size_t>(kSampleSize) * 4;
    const size_t sel_bytes = static_cast<size_t>(sel_cap) * 8;
    size_t hist = sel_bytes > guess ? sel_bytes : guess;
    if (hist < static_cast<size_t>(kBins) * 4) hist = static_cast<size_t>(kBins) * 4;
    if (width * es <= kDirectBytes) {
        pl.split = 0;
        pl.direct_max = static_cast<int32_t>(width);
        pl.chunks_per_row = 1;
    } else if (sel_cap <= kPairSortMax &&
               num_rows * ((width + kFusedChunkBytes / es - 1) / (kFusedChunkBytes / es)) <= kFusedMaxSlots) {
        // every row longer than top_k: row kernel guess, then one chunk
        // kernel block per kFusedChunkBytes of the row
        pl.split = 1;
        pl.fused = 1;
        pl.direct_max = top_k;
        const int64_t fchunk = kFusedChunkBytes / es;
        pl.chunk = static_cast<int32_t>(fchunk);
        pl.chunks_per_row = static_cast<int32_t>((width + fchunk - 1) / fchunk);
        if (pl.chunks_per_row > kThreads) return GBTOPK_EUNSUPPORTED;
        pl.block_rows = num_rows;
        pl.fused_smem = kCtrlBytes + kFusedStageBytes;
        pl.final_sel_bytes = static_cast<size_t>(kPairSortMax) * 8;
        int64_t entries = 0;
        for (int64_t j = 1; j <= pl.chunks_per_row; ++j) {
            int64_t n_min = (j - 1) * fchunk + 1;
            if (n_min <= pl.direct_max) n_min = pl.direct_max + 1;
            if (n_min > width || n_min > j * fchunk) continue;
            const int64_t e = j * static_cast<int64_t>(chunk_seg_cap(n_min, top_k, pl.chunk));
            entries = e > entries ? e : entries;
        }
        pl.row_seg_entries = entries;
        pl.ws_row_bytes = align_up(ws_seg_offset(pl.chunks_per_row) + 8 * static_cast<size_t>(entries), 256);
    } else {
        // every row longer than top_k runs through the split pipeline
        pl.split = 1;
        pl.direct_max = top_k;
        pl.chunks_per_row = static_cast<int32_t>((width + chunk - 1) / chunk);
        if (pl.chunks_per_row > kThreads) return GBTOPK_EUNSUPPORTED;  // the same width limit as the fused path
        pl.block_rows = num_rows < kMaxBlockRows ? num_rows : kMaxBlockRows;
        // control block, the row table of one launch, the ring (a small
        // batch's stream block still fits beside a row-kernel block)
        pl.stream_smem = kCtrlBytes + align_up(static_cast<size_t>(pl.block_rows + 1) * 16, 128) +
                         static_cast<size_t>(kStages) * kStageBytes;
        // finalize: control, histogram / selection, boundary bin, chunk
        // offsets, then the gathered candidates (up to kGatherCandidates;
        // the region doubles as the sorted-output scratch)
        pl.final_sel_bytes = static_cast<size_t>(sel_cap) * 8 > static_cast<size_t>(kFinalHistBytes)
                                 ? static_cast<size_t>(sel_cap) * 8
                                 : static_cast<size_t>(kFinalHistBytes);
        const size_t fixed = kCtrlBytes + pl.final_sel_bytes + static_cast<size_t>(kFinalBCap) * 8 +
                             4 * static_cast<size_t>(kFinalThreads) + 4 * static_cast<size_t>(kCoarseBins);
        size_t gather = static_cast<size_t>(kGatherCandidates) * 8;
        if (fixed + gather > kMaxSmemBytes) gather = kMaxSmemBytes > fixed ? (kMaxSmemBytes - fixed) / 16 * 16 : 0;
        if (gather < det_scratch_bytes(sel_cap)) return GBTOPK_EUNSUPPORTED;
        pl.final_smem = fixed + gather;
        // candidate entries per row: the largest chunks x per-chunk capacity
        // over the row lengths the width allows (capacity shrinks as n grows,
        // so within a chunk count the shortest row is the worst case)
        int64_t entries = 0;
        for (int64_t j = 1; j <= pl.chunks_per_row; ++j) {
            int64_t n_min = (j - 1) * chunk + 1;
            if (n_min <= pl.direct_max) n_min = pl.direct_max + 1;
            if (n_min > width || n_min > j * chunk) continue;
            const int64_t e = j * static_cast<int64_t>(chunk_seg_cap(n_min, top_k, pl.chunk));
            entries = e > entries ? e : entries;
        }
        pl.row_seg_entries = entries;
        pl.ws_row_bytes = align_up(ws_seg_offset(pl.chunks_per_row) + 8 * static_cast<size_t>(entries), 256);
    }
    // the row kernel stages direct rows only in plans without a split
    // pipeline; the sorted output's scratch reuses the stage (free once the
    // row is selected)
    const size_t stage = pl.split ? 0 : align_up(static_cast<size_t>(pl.direct_max) * es, 16) + 32;
    pl.off_hist = kCtrlBytes;
    pl.off_stage = align_up(pl.off_hist + hist, 128);
    pl.det_bytes = det_scratch_bytes(sel_cap);
    pl.row_smem_sorted = pl.off_stage + (stage > pl.det_bytes ? stage : pl.det_bytes);
    // split plans select nothing in the row kernel unless the output is
    // sorted (short rows are written straight out): the guess's counters only
    // (its sample stays in registers; 4 KB with the control block), so three
    // chunk-kernel blocks fit beside four row-kernel blocks on one SM
    pl.row_smem = pl.split ? align_up(pl.off_hist + static_cast<size_t>(kGuessBins) * 4, 128) : pl.off_stage + stage;
    if (pl.row_smem_sorted > kMaxSmemBytes) return GBTOPK_EUNSUPPORTED;
    pl.ws_bytes = kWsHeaderBytes + static_cast<size_t>(num_rows) * pl.ws_row_bytes;
    *plan = pl;
    return GBTOPK_OK;
}

}  // namespace gbtopk

using gbtopk::Params;
using gbtopk::Plan;

namespace {

// `deterministic` is a set of GBTOPK_SORTED / GBTOPK_TIE_SMALL /
// GBTOPK_TIE_LARGE flags; the two tie modes exclude each other.
int check_common(const void *x, int dtype, int64_t num_rows, int64_t width, int64_t row_stride,
                 int32_t top_k, const void *out, int deterministic, const void *workspace,
                 size_t workspace_bytes, Plan *plan) {
    const int all = GBTOPK_SORTED | GBTOPK_TIE_SMALL | GBTOPK_TIE_LARGE;
    if ((deterministic & ~all) != 0 || ((deterministic & GBTOPK_TIE_SMALL) && (deterministic & GBTOPK_TIE_LARGE)))
        return GBTOPK_EINVAL;
    const int rc = gbtopk::make_plan(num_rows, width, top_k, dtype, plan);
    if (rc != GBTOPK_OK) return rc;
    if (num_rows == 0) return GBTOPK_OK;
    if (row_stride < width && num_rows > 1) return GBTOPK_EINVAL;
    if (!out) return GBTOPK_EINVAL;
    if (width > 0 && !x) return GBTOPK_EINVAL;
    if (x && !gbtopk::aligned(x, static_cast<size_t>(gbtopk::elem_bytes(dtype)))) return GBTOPK_EALIGN;
    if (!gbtopk::aligned(out, 16)) return GBTOPK_EALIGN;
    if (!workspace || !gbtopk::aligned(workspace, 256) || workspace_bytes < plan->ws_bytes)
        return GBTOPK_EWORKSPACE;
    return GBTOPK_OK;
}

// Poll limit of the first bounded wait on each bulk copy: kSpinLimit, or
// the positive value of the environment variable GBTOPK_WAIT_POLLS (read
// once per process).  A small value makes those waits give up, which runs
// the recovery path (the affected rows are recomputed from global memory,
// the status word's timeout bit is set) without any fault.
uint32_t first_wait_polls() {
    static const uint32_t polls = [] {
        const char *v = std::getenv("GBTOPK_WAIT_POLLS");
        if (!v || !*v) return gbtopk::kSpinLimit;
        char *end = nullptr;
        const unsigned long x = std::strtoul(v, &end, 10);
        return (end && *end == '\0' && x > 0 && x <= gbtopk::kSpinLimit) ? static_cast<uint32_t>(x)
                                                                         : gbtopk::kSpinLimit;
    }();
    return polls;
}

int launch(int dtype, const Params &p0, void *stream) {
    Params p = p0;
    p.wait_polls = first_wait_polls();
    const cudaError_t e = gbtopk::launch_topk(dtype, p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GBTOPK_OK : GBTOPK_ECUDA;
}

}  // namespace

extern "C" {

int gbtopk_varlen(const void *logits, int dtype, int64_t num_rows, int64_t width,
                  int64_t row_stride, const int32_t *seq_lens, int32_t next_n,
                  int32_t compress_ratio, int32_t top_k, const int32_t *pre_idx,
                  int32_t *out_indices, void *out_values, int deterministic, void *workspace,
                  size_t workspace_bytes, void *stream) {
    if (next_n < 1 || compress_ratio < 1 || num_rows < 0 || num_rows % next_n != 0)
        return GBTOPK_EINVAL;
    Plan plan;
    int rc = check_common(logits, dtype, num_rows, width, row_stride, top_k, out_indices, deterministic,
                          workspace, workspace_bytes, &plan);
    if (rc != GBTOPK_OK || num_rows == 0) return rc;
    if (!seq_lens) return GBTOPK_EINVAL;
    const size_t nout = static_cast<size_t>(num_rows) * static_cast<size_t>(top_k);
    if (out_values) {
        if (!gbtopk::aligned(out_values, 16)) return GBTOPK_EALIGN;
        if (gbtopk::overlaps(out_indices, nout * 4, out_values, nout * gbtopk::elem_bytes(dtype)))
            return GBTOPK_EOVERLAP;
    }
    int status = GBTOPK_OK;
    if (pre_idx && !gbtopk::aligned(pre_idx, 16)) {
        pre_idx = nullptr;
        status = GBTOPK_HINT_DISCARDED;
    }
    Params p{};
    p.x = logits;
    p.num_rows = num_rows;
    p.width = width;
    p.row_stride = num_rows > 1 ? row_stride : (row_stride > width ? row_stride : width);
    p.seq_lens = seq_lens;
    p.next_n = next_n;
    p.compress_ratio = compress_ratio;
    p.pre_idx = pre_idx;
    p.k = top_k;
    p.deterministic = deterministic;
    p.out_idx = out_indices;
    p.out_val = out_values;
    p.ws = static_cast<uint8_t *>(workspace);
    p.plan = plan;
    rc = launch(dtype, p, stream);
    return rc != GBTOPK_OK ? rc : status;
}

int gbtopk_ragged_transform(const void *scores, int dtype, int64_t num_rows, int64_t width,
                            int64_t row_stride, const int32_t *lengths, const int32_t *row_starts,
                            const int32_t *topk_indices_offset, int32_t top_k, int32_t *out,
                            int deterministic, void *workspace, size_t workspace_bytes, void *stream) {
    if (num_rows < 0) return GBTOPK_EINVAL;
    Plan plan;
    int rc = check_common(scores, dtype, num_rows, width, row_stride, top_k, out, deterministic,
                          workspace, workspace_bytes, &plan);
    if (rc != GBTOPK_OK || num_rows == 0) return rc;
    if (!lengths || !topk_indices_offset) return GBTOPK_EINVAL;
    Params p{};
    p.x = scores;
    p.num_rows = num_rows;
    p.width = width;
    p.row_stride = num_rows > 1 ? row_stride : (row_stride > width ? row_stride : width);
    p.next_n = 1;
    p.compress_ratio = 1;
    p.lengths = lengths;
    p.row_starts = row_starts;
    p.k = top_k;
    p.deterministic = deterministic;
    p.out_idx = out;
    p.idx_offset = topk_indices_offset;
    p.page_size = 1;
    p.ws = static_cast<uint8_t *>(workspace);
    p.plan = plan;
    return launch(dtype, p, stream);
}

int gbtopk_page_table_transform_cu_seqlens(const void *scores, int dtype, int64_t num_rows,
                                           int64_t width, int64_t row_stride, const int32_t *lengths,
                                           const int32_t *row_starts, const int32_t *page_table,
                                           int64_t pt_cols, int64_t pt_row_stride,
                                           const int32_t *cu_seqlens_q, int64_t num_reqs,
                                           int32_t top_k, int32_t *out, int deterministic,
                                           void *workspace, size_t workspace_bytes, void *stream) {
    if (num_rows < 0 || num_reqs < 0 || pt_cols < 0) return GBTOPK_EINVAL;
    if (num_reqs > 1 && pt_row_stride < pt_cols) return GBTOPK_EINVAL;
    Plan plan;
    int rc = check_common(scores, dtype, num_rows, width, row_stride, top_k, out, deterministic,
                          workspace, workspace_bytes, &plan);
    if (rc != GBTOPK_OK || num_rows == 0) return rc;
    if (!lengths || !page_table || !cu_seqlens_q) return GBTOPK_EINVAL;
    Params p{};
    p.x = scores;
    p.num_rows = num_rows;
    p.width = width;
    p.row_stride = num_rows > 1 ? row_stride : (row_stride > width ? row_stride : width);
    p.next_n = 1;
    p.compress_ratio = 1;
    p.lengths = lengths;
    p.row_starts = row_starts;
    p.k = top_k;
    p.deterministic = deterministic;
    p.out_idx = out;
    p.page_table = page_table;
    p.pt_cols = pt_cols;
    p.pt_row_stride = num_reqs > 1 ? pt_row_stride : (pt_row_stride > pt_cols ? pt_row_stride : pt_cols);
    p.page_size = 1;
    p.cu_seqlens_q = cu_seqlens_q;
    p.num_reqs = num_reqs;
    p.ws = static_cast<uint8_t *>(workspace);
    p.plan = plan;
    return launch(dtype, p, stream);
}

int gbtopk_page_table_transform(const void *scores, int dtype, int64_t num_rows, int64_t width,
                                int64_t row_stride, const int32_t *lengths,
                                const int32_t *row_starts, const int32_t *page_table,
                                int64_t pt_cols, int64_t pt_row_stride,
                                const int32_t *pt_row_starts, int32_t page_size, int32_t top_k,
                                int32_t *out, int32_t *out_raw, int deterministic, void *workspace,
                                size_t workspace_bytes, void *stream) {
    if (page_size < 1 || page_size > (1 << 30) || pt_cols < 0 || num_rows < 0) return GBTOPK_EINVAL;
    if (num_rows > 1 && pt_row_stride < pt_cols) return GBTOPK_EINVAL;
    if (page_size > 1 && row_starts && !pt_row_starts) return GBTOPK_EINVAL;
    Plan plan;
    int rc = check_common(scores, dtype, num_rows, width, row_stride, top_k, out, deterministic,
                          workspace, workspace_bytes, &plan);
    if (rc != GBTOPK_OK || num_rows == 0) return rc;
    if (!lengths || !page_table) return GBTOPK_EINVAL;
    const size_t nout = static_cast<size_t>(num_rows) * static_cast<size_t>(top_k) * 4;
    if (out_raw) {
        if (!gbtopk::aligned(out_raw, 16)) return GBTOPK_EALIGN;
        if (gbtopk::overlaps(out, nout, out_raw, nout)) return GBTOPK_EOVERLAP;
    }
    Params p{};
    p.x = scores;
    p.num_rows = num_rows;
    p.width = width;
    p.row_stride = num_rows > 1 ? row_stride : (row_stride > width ? row_stride : width);
    p.next_n = 1;
    p.compress_ratio = 1;
    p.lengths = lengths;
    p.row_starts = row_starts;
    p.k = top_k;
    p.deterministic = deterministic;
    p.out_idx = out;
    p.out_raw = out_raw;
    p.page_table = page_table;
    p.pt_cols = pt_cols;
    p.pt_row_stride = pt_row_stride;
    p.pt_row_starts = pt_row_starts;
    p.page_size = page_size;
    p.pt_start_is_row_start = (!pt_row_starts && page_size == 1 && row_starts) ? 1 : 0;
    p.ws = static_cast<uint8_t *>(workspace);
    p.plan = plan;
    return launch(dtype, p, stream);
}

size_t gbtopk_workspace_bytes(int64_t num_rows, int64_t width, int32_t top_k, int dtype) {
    Plan plan;
    if (gbtopk::make_plan(num_rows, width, top_k, dtype, &plan) != GBTOPK_OK) return 0;
    return plan.ws_bytes;
}

int gbtopk_device_status(void *workspace, uint32_t *flags, void *stream) {
    if (!workspace || !flags || !gbtopk::aligned(workspace, 256)) return GBTOPK_EINVAL;
    uint32_t host = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&host, workspace, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return GBTOPK_ECUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof(host), s) != cudaSuccess) return GBTOPK_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GBTOPK_ECUDA;
    *flags = host;
    return GBTOPK_OK;
}

int gbtopk_plan_query(int64_t num_rows, int64_t width, int32_t top_k, int dtype, int64_t *out) {
    if (!out) return GBTOPK_EINVAL;
    Plan plan;
    const int rc = gbtopk::make_plan(num_rows, width, top_k, dtype, &plan);
    if (rc != GBTOPK_OK) return rc;
    out[0] = plan.chunk;
    out[1] = plan.chunks_per_row;
    out[2] = plan.direct_max;
    out[3] = static_cast<int64_t>(plan.row_smem);
    out[4] = plan.split;
    out[5] = plan.row_seg_entries;
    out[6] = static_cast<int64_t>(plan.stream_smem);
    out[7] = static_cast<int64_t>(plan.final_smem);
    out[8] = static_cast<int64_t>(plan.ws_bytes);
    out[9] = static_cast<int64_t>(plan.ws_row_bytes);
    out[10] = static_cast<int64_t>(plan.row_smem_sorted);
    out[11] = plan.fused;
    out[12] = static_cast<int64_t>(plan.fused_smem);
    return GBTOPK_OK;
}

const char *gbtopk_status_str(int status) {
    switch (status) {
        case GBTOPK_OK: return "GBTOPK_OK";
        case GBTOPK_HINT_DISCARDED: return "GBTOPK_HINT_DISCARDED: pre_idx not 16-byte aligned; ran hint-free";
        case GBTOPK_EINVAL: return "GBTOPK_EINVAL: invalid shape, dtype, grouping or null pointer";
        case GBTOPK_EALIGN: return "GBTOPK_EALIGN: misaligned output or score buffer";
        case GBTOPK_EOVERLAP: return "GBTOPK_EOVERLAP: output buffers overlap";
        case GBTOPK_EUNSUPPORTED: return "GBTOPK_EUNSUPPORTED: outside the supported envelope";
        case GBTOPK_ECUDA: return "GBTOPK_ECUDA: CUDA launch failed";
        case GBTOPK_EWORKSPACE: return "GBTOPK_EWORKSPACE: workspace missing, misaligned or too small";
        case GBTOPK_ETIMEOUT: return "GBTOPK_ETIMEOUT: a bounded device wait gave up";
        default: return "unknown gbtopk status";
    }
}

}  // extern "C"

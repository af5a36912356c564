// Host side of gbtopk: argument checks, the launch plan, and the C ABI
// declared in include/gbtopk.h.  No device data is ever read on the host.
#include <cstdint>
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
int make_plan(int64_t num_rows, int64_t width, int32_t top_k, int dtype, Plan *plan) {
    if (num_rows < 0 || width < 0 || top_k < 1 ||
        (dtype != GBTOPK_F32 && dtype != GBTOPK_BF16 && dtype != GBTOPK_F16))
        return GBTOPK_EINVAL;
    if (top_k > GBTOPK_MAX_TOP_K) return GBTOPK_EUNSUPPORTED;
    if (width > INT32_MAX) return GBTOPK_EUNSUPPORTED;
    const int es = elem_bytes(dtype);
    const int64_t chunk_max = kChunkBytes / es;
    Plan pl{};
    pl.threads = kThreads;
    int sel_cap = 32;
    while (sel_cap < top_k) sel_cap <<= 1;
    pl.sel_cap = sel_cap;
    if (width <= chunk_max) {
        pl.chunk = static_cast<int32_t>(align_up(static_cast<size_t>(width < 1 ? 1 : width), 32));
        pl.chunks_per_row = 1;
        pl.split = 0;
        pl.gcap = 0;
    } else {
        pl.chunk = static_cast<int32_t>(chunk_max);
        pl.chunks_per_row = static_cast<int32_t>((width + chunk_max - 1) / chunk_max);
        pl.split = 1;
        // Fixed per-row layout (independent of top_k, dtype and width) so one
        // workspace serves every geometry: candidate scratch of one call can
        // never land under another call's counters.
        pl.gcap = gbtopk::kRowCandCap;
    }
    pl.grid = num_rows * pl.chunks_per_row;
    if (pl.grid > INT32_MAX) return GBTOPK_EUNSUPPORTED;
    // Shared memory: control block | histogram (kBins counters; also the
    // row sample and, once the histogram is consumed, the selection buffer)
    // | staged chunk (also candidate / boundary-bin scratch).
    size_t hist = static_cast<size_t>(sel_cap) * 8;
    if (pl.split || width > kExactMax) {
        hist = hist > static_cast<size_t>(kBins) * 4 ? hist : static_cast<size_t>(kBins) * 4;
        hist = hist > static_cast<size_t>(kSampleSize) * 4 ? hist : static_cast<size_t>(kSampleSize) * 4;
    }
    const size_t stage = align_up((static_cast<size_t>(pl.chunk) + 16 / es) * es, 16);
    pl.off_hist = kCtrlBytes;
    pl.off_stage = align_up(pl.off_hist + hist, 16);
    pl.smem = pl.off_stage + stage;
    pl.ws_row_bytes = pl.split ? kRowBytes : 0;
    pl.ws_bytes = kWsHeaderBytes + static_cast<size_t>(num_rows) * pl.ws_row_bytes;
    *plan = pl;
    return GBTOPK_OK;
}

}  // namespace gbtopk

using gbtopk::Params;
using gbtopk::Plan;

namespace {

int check_common(const void *x, int dtype, int64_t num_rows, int64_t width, int64_t row_stride,
                 int32_t top_k, const void *out, const void *workspace, size_t workspace_bytes,
                 Plan *plan) {
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

int launch(int dtype, const Params &p, void *stream) {
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
    int rc = check_common(logits, dtype, num_rows, width, row_stride, top_k, out_indices, workspace,
                          workspace_bytes, &plan);
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
    p.deterministic = deterministic ? 1 : 0;
    p.out_idx = out_indices;
    p.out_val = out_values;
    p.ws = static_cast<uint8_t *>(workspace);
    p.plan = plan;
    rc = launch(dtype, p, stream);
    return rc != GBTOPK_OK ? rc : status;
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
    int rc = check_common(scores, dtype, num_rows, width, row_stride, top_k, out, workspace,
                          workspace_bytes, &plan);
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
    p.deterministic = deterministic ? 1 : 0;
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
    out[2] = plan.threads;
    out[3] = static_cast<int64_t>(plan.smem);
    out[4] = plan.split;
    out[5] = plan.gcap;
    out[6] = plan.grid;
    out[7] = static_cast<int64_t>(plan.ws_bytes);
    out[8] = static_cast<int64_t>(plan.ws_row_bytes);
    out[9] = static_cast<int64_t>(gbtopk::kRowCounterBytes);
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

// Internal declarations shared by the host API (gbtopk_api.cu) and the
// device code (gbtopk_kernels.cu).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace gbtopk {

constexpr int kThreads = 256;          // threads per block
constexpr int kSampleGroups = 256;     // one group of 8 consecutive columns per thread
constexpr int kSampleSize = kSampleGroups * 8;
constexpr int kBinBits = 12;
constexpr int kBins = 1 << kBinBits;   // candidate histogram bins
constexpr int kRankMax = 256;          // boundary-bin size resolved by rank counting
constexpr int kExactMax = 3072;        // rows up to this length: plain exact radix select
constexpr size_t kCtrlBytes = 2048;    // per-block control block (counters, scan, digit histogram)
constexpr int kChunkBytes = 32768;     // staged bytes per block for split rows
constexpr size_t kWsHeaderBytes = 256; // device status word + padding
constexpr int kRowHeaderBytes = 32;    // ticket, count, flags, t_lo, bin shift, pad
constexpr int kRowCandCap = 16384;     // candidates per split row (8 x the largest top_k)
// Per-row workspace of a split row: header + histogram (kept zero between
// calls), then candidate scratch.
constexpr size_t kRowCounterBytes = kRowHeaderBytes + 4 * kBins;
constexpr size_t kRowBytes = (kRowCounterBytes + 8 * static_cast<size_t>(kRowCandCap) + 255) / 256 * 256;
constexpr uint32_t kSpinLimit = 1u << 22;

// Per-row flags in the split-row workspace.
constexpr uint32_t kRowOverflow = 1u;  // a block lost candidates: recompute the row
// Bits of the device status word.
constexpr uint32_t kStatusWaitTimeout = 1u;

struct Plan {
    int32_t chunk;        // columns staged per block
    int32_t chunks_per_row;
    int32_t threads;
    int32_t split;        // 1 when rows wider than `chunk` are cut across blocks
    int32_t gcap;         // candidate capacity per split row
    int32_t sel_cap;      // power of two >= top_k (selection / sort buffer)
    int64_t grid;
    size_t smem;          // dynamic shared memory per block
    size_t ws_row_bytes;  // per-row workspace bytes (split plans)
    size_t ws_bytes;      // total workspace bytes
    // shared-memory layout (byte offsets)
    size_t off_hist, off_stage;
};

// Kernel arguments.  Row-length source: varlen mode when seq_lens != null,
// ragged (page-table) mode when lengths != null.
struct Params {
    const void *x;
    int64_t num_rows, width, row_stride;
    const int32_t *seq_lens;
    int32_t next_n, compress_ratio;
    const int32_t *lengths;
    const int32_t *row_starts;
    const int32_t *pre_idx;
    int32_t k;
    int32_t deterministic;
    int32_t *out_idx;
    void *out_val;
    int32_t *out_raw;
    const int32_t *page_table;   // null: no transform
    int64_t pt_cols, pt_row_stride;
    const int32_t *pt_row_starts;
    int32_t page_size;
    int32_t pt_start_is_row_start;
    uint8_t *ws;
    Plan plan;
};

// Builds the launch plan; returns a gbtopk status.
int make_plan(int64_t num_rows, int64_t width, int32_t top_k, int dtype, Plan *plan);

// Enqueues the selection kernel (device code lives in gbtopk_kernels.cu).
cudaError_t launch_topk(int dtype, const Params &p, cudaStream_t stream);

}  // namespace gbtopk

// Internal declarations shared by the host API (gbtopk_api.cu) and the
// device code (gbtopk_kernels.cu).  Not part of the public ABI.
#pragma once

#include <cmath>
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace gbtopk {

constexpr int kThreads = 256;          // threads per block (row and stream kernels)
constexpr int kFinalThreads = 512;     // threads per block of the finalize kernel
constexpr int kSampleGroups = 256;     // one group of 8 consecutive columns per thread
constexpr int kSampleSize = kSampleGroups * 8;
constexpr int kBinBits = 12;
constexpr int kBins = 1 << kBinBits;   // candidate histogram bins
constexpr int kGuessBins = 1024;       // bins of the sample's threshold search (each round)
constexpr int kRankMax = 256;          // boundary-bin size resolved by rank counting
constexpr int kRankAllMax = 64;        // the same in the finalize (a block radix select above)
constexpr size_t kCtrlBytes = 2048;    // per-block control block (counters, scan, digit histogram)
constexpr int kChunkBytes = 65536;     // bytes per stream chunk (one bulk copy)
constexpr int kStages = 3;             // bulk-copy ring depth of the stream kernel
constexpr int kGroupWarps = 16;        // consumer warps that share one chunk
constexpr int kDirectBytes = 65536;    // rows of at most this many bytes: one block per row
constexpr int kStageBytes = kChunkBytes + 32;  // a chunk plus its 16-byte alignment slack
constexpr int kStreamThreads = 544;    // stream kernel: 1 producer warp + 16 consumer warps
constexpr int kFinalHistBytes = 16384; // finalize histogram / selection buffer
constexpr int kMaxBlockRows = 2048;    // rows per launch of the split pipeline
constexpr int kFinalBCap = 2048;       // boundary-bin members the finalize kernel can hold
constexpr int kGatherCandidates = 8192; // candidates the finalize kernel gathers into shared memory
constexpr size_t kMaxSmemBytes = 232448;  // dynamic shared memory one block may opt into (227 KB)
constexpr int kPairSortMax = 2048;     // sorted output copies up to this many pairs, else 16-bit positions
constexpr size_t kWsHeaderBytes = 256; // device status word + padding
constexpr size_t kRowInfoBytes = 16;   // t_lo, coarse bin shift, chunk ticket (written by the row kernel)
constexpr uint32_t kSpinLimit = 1u << 22;
// Coarse candidate bins of a split row's final selection: keys t_lo .. t_est
// (the guess and its estimate of the k-th key) fill the lower half of the
// bins, one key per bin when that range is short, the top bin open-ended.
constexpr int kCoarseBins = 256;

// Fused split path (top_k <= kPairSortMax): one block of kThreads per chunk
// of kFusedChunkBytes, finalized in its own shared memory by the row's last
// block.  The finalize regions inside the chunk's stage (byte offsets):
// boundary list, chunk offsets, coarse-bin slot counters, gathered
// candidates, and the selection (up to kPairSortMax pairs) at the end; the
// sorted-output scratch reuses everything before the selection once the row
// is selected.
constexpr int kFusedChunkBytes = 65536;
constexpr int kFusedStageBytes = kFusedChunkBytes + 32;
constexpr int kFusedBCap = 256;
constexpr int kFusedOffChOff = kFusedBCap * 8;
constexpr int kFusedOffFill = kFusedOffChOff + kThreads * 4;
constexpr int kFusedOffCand = kFusedOffFill + kCoarseBins * 4;
constexpr int kFusedOffSel = kFusedStageBytes - kPairSortMax * 8;
constexpr int kFusedGatherCap = (kFusedOffSel - kFusedOffCand) / 16 * 2;
// The fused path serves batches of up to kFusedMaxSlots (row, chunk) slots:
// about four waves of three chunk blocks per SM.  Larger batches stream
// through the persistent kernel's ring, which keeps every SM's copies in
// flight while its consumers filter.
constexpr int64_t kFusedMaxSlots = 2048;

// Flags of Params::deterministic (the public GBTOPK_SORTED / GBTOPK_TIE_*).
constexpr int kSortedFlag = 1;
constexpr int kTieSmallFlag = 2;
constexpr int kTieLargeFlag = 4;

// Tie mode among values equal to the k-th: 0 any, 1 smallest columns (also
// implied by the sorted flag alone), 2 largest columns.
__host__ __device__ inline int tie_mode(int flags) {
    return (flags & kTieLargeFlag) ? 2 : ((flags & (kSortedFlag | kTieSmallFlag)) ? 1 : 0);
}
__host__ __device__ inline bool sorted_output(int flags) { return (flags & kSortedFlag) != 0; }

// Bits of the device status word.
constexpr uint32_t kStatusWaitTimeout = 1u;
constexpr uint32_t kStatusCopyLost = 2u;  // a bulk copy never completed: outputs unreliable

struct Plan {
    int32_t fused;           // 1: split rows run through the chunk kernel (row guess + chunk kernel)
    int32_t chunk;           // elements per chunk of a split row
    int32_t direct_max;      // rows up to this length are finished by the row kernel
    int32_t chunks_per_row;  // chunks of the widest split row (0: no split rows possible)
    int32_t split;           // 1 when some row can exceed direct_max
    int32_t sel_cap;         // power of two >= top_k
    size_t final_sel_bytes;  // finalize histogram / selection region (>= sel_cap pairs)
    size_t det_bytes;        // sorted-output scratch (det_scratch_bytes(sel_cap))
    size_t row_smem_sorted;  // row kernel shared memory when the output is sorted
    int32_t stream_grid;     // persistent stream blocks
    int64_t row_seg_entries; // candidate entries reserved per split row
    size_t row_smem, stream_smem, final_smem;
    size_t fused_smem;       // chunk kernel (fused plans)
    size_t off_hist, off_stage;  // row kernel layout
    size_t ws_row_bytes;     // per-row workspace bytes (split plans)
    size_t ws_bytes;         // total workspace bytes
    int64_t block_rows;      // rows per launch of the split pipeline
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
    int32_t deterministic;       // kSortedFlag | kTieSmallFlag | kTieLargeFlag
    int32_t *out_idx;
    void *out_val;
    int32_t *out_raw;
    const int32_t *page_table;  // null: no transform
    int64_t pt_cols, pt_row_stride;
    const int32_t *pt_row_starts;
    int32_t page_size;
    int32_t pt_start_is_row_start;
    const int32_t *idx_offset;    // ragged KV: out = idx + idx_offset[row] (null: none)
    const int32_t *cu_seqlens_q;  // page-table row = request of the score row (null: the row itself)
    int64_t num_reqs;
    uint8_t *ws;   // status word at ws[0], the call's stream abort word at ws[4]; per-row blocks from kWsHeaderBytes
    uint32_t wait_polls;  // poll limit of each first bounded wait on a bulk copy (kSpinLimit unless testing)
    int64_t row0;  // first row of this launch (the split pipeline runs in row blocks)
    int64_t rows;  // rows of this launch
    Plan plan;
};

// Guess rank: the sample rank whose key is taken as the threshold guess,
// r = e + 6 sqrt(e) + 2 with e = m k / n the expected number of sample
// elements at or above the k-th largest of the row.  Single precision
// (IEEE-rounded on host and device alike; FP64 is slow on this GPU).
__host__ __device__ inline uint32_t guess_rank(int64_t n, int32_t k) {
    const float e = static_cast<float>(kSampleSize) * static_cast<float>(k) / static_cast<float>(n);
    float r = ceilf(e + 6.0f * sqrtf(e) + 2.0f);
    if (r > static_cast<float>(kSampleSize)) r = static_cast<float>(kSampleSize);
    return static_cast<uint32_t>(r);
}

// Byte offsets inside a split row's workspace block: the row info, one
// count per chunk, the row's coarse candidate histogram (kCoarseBins
// counters, zeroed by the row kernel, counted by the chunk kernel), then
// the chunk segments.
__host__ __device__ inline size_t ws_hist_offset(int32_t chunks_per_row) {
    return (kRowInfoBytes + 4 * static_cast<size_t>(chunks_per_row) + 15) / 16 * 16;
}
__host__ __device__ inline size_t ws_seg_offset(int32_t chunks_per_row) {
    return ws_hist_offset(chunks_per_row) + static_cast<size_t>(kCoarseBins) * 4;
}

// Candidate capacity of one chunk of a split row with n valid columns (1.5x
// the guessed fraction of the chunk plus 256, in multiples of 64); the same
// arithmetic on host (workspace sizing) and device.
__host__ __device__ inline int32_t chunk_seg_cap(int64_t n, int32_t k, int32_t chunk) {
    const uint32_t r = guess_rank(n, k);
    const int64_t cap = (3 * static_cast<int64_t>(r) * chunk) / (2 * kSampleSize) + 256;
    const int64_t c = cap < chunk ? cap : chunk;
    return static_cast<int32_t>((c + 63) / 64 * 64);
}

// Scratch of the sorted output for up to m_cap pairs: kBins counters, then
// a 64-bit order key, a 16-bit position and a 16-bit inverse-map entry per
// pair (m_cap <= kPairSortMax), or the positions alone.
__host__ __device__ inline size_t det_scratch_bytes(int32_t m_cap) {
    const size_t per = m_cap <= kPairSortMax ? 12 : 2;
    return static_cast<size_t>(kBins) * 4 + ((per * static_cast<size_t>(m_cap) + 15) / 16) * 16;
}

// Builds the launch plan; returns a gbtopk status.
int make_plan(int64_t num_rows, int64_t width, int32_t top_k, int dtype, Plan *plan);

// Enqueues the kernels of one call (device code lives in gbtopk_kernels.cu).
cudaError_t launch_topk(int dtype, const Params &p, cudaStream_t stream);

}  // namespace gbtopk
